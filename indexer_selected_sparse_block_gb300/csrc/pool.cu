// pool.cu -- block mean pooling of the raw index keys (sfa_pool_index_keys).
//
// The indexer works on one mean-pooled key per block of compress_ratio tokens, pooled from the
// raw index keys: the model pools before it normalises and rotates them (llama.cpp commit
// "model: add Qwen3.8-Flash-Next (qwen4exp)", QSA paragraphs).
//
// HBM-bound streaming kernel: each thread owns one 16-byte chunk of one pooled row, reads the
// chunk of the block's cr raw rows with 16-byte loads (a warp covers whole 128/256-byte rows),
// sums in fp32 in token order, divides by cr (IEEE), and writes the hi and lo bf16 halves.
// Optionally it also writes the row's error-bound factor for the bounded scores,
//   r_b = (|lo_b|_2 + 2^-14 |hi_b|_2) * (1 + 2^-16)
// from the stored bf16 halves (the chunks of a row are consecutive lanes: a shuffle sum); the
// factor (1 + 2^-16) covers the fp32 rounding of the two norms (128 squares: < 2^-17).
// Bytes per block: cr * d_idx * sizeof(X) read + 4 * d_idx (+ 4) written.
#include "sfa_common.cuh"

namespace sfa {
namespace {

template <typename T>
struct Vec8;  // eight input elements as fp32
template <>
struct Vec8<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&v)[8]) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};
template <>
struct Vec8<float> {
    static __device__ __forceinline__ void load(const float *p, float (&v)[8]) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};

// grid: (ceil(rows * chunks / 256), n_seq); one thread per (pooled row, 8-element chunk).
template <typename T>
__global__ void __launch_bounds__(256) pool_kernel(const T *__restrict__ X, int64_t x_seq_stride,
                                                   int d_idx, int cr, int64_t blk_begin,
                                                   int64_t n_rows, __nv_bfloat16 *__restrict__ Kbar,
                                                   int64_t kbar_seq_stride, float *__restrict__ Kr,
                                                   int64_t kr_seq_stride) {
    pdl_wait();
    pdl_trigger();
    const int chunks = d_idx >> 3;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool valid = gid < n_rows * chunks;
    const int64_t b = blk_begin + (valid ? gid / chunks : 0);
    const int c = (int)(gid % chunks);
    const int64_t seq = blockIdx.y;
    float lo2 = 0.f, hi2 = 0.f;
    if (valid) {
        const T *src = X + seq * x_seq_stride + b * cr * d_idx + c * 8;
        float sum[8];
        Vec8<T>::load(src, sum);
        for (int t = 1; t < cr; ++t) {
            float v[8];
            Vec8<T>::load(src + (int64_t)t * d_idx, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) sum[i] += v[i];
        }
        const float rcr = (float)cr;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float m0 = __fdiv_rn(sum[2 * i], rcr), m1 = __fdiv_rn(sum[2 * i + 1], rcr);
            const __nv_bfloat16 h0 = __float2bfloat16_rn(m0), h1 = __float2bfloat16_rn(m1);
            const __nv_bfloat16 l0 = __float2bfloat16_rn(m0 - __bfloat162float(h0));
            const __nv_bfloat16 l1 = __float2bfloat16_rn(m1 - __bfloat162float(h1));
            hi[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
            lo[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
            const float fh0 = __bfloat162float(h0), fh1 = __bfloat162float(h1);
            const float fl0 = __bfloat162float(l0), fl1 = __bfloat162float(l1);
            hi2 = fmaf(fh0, fh0, fmaf(fh1, fh1, hi2));
            lo2 = fmaf(fl0, fl0, fmaf(fl1, fl1, lo2));
        }
        __nv_bfloat16 *dst = Kbar + seq * kbar_seq_stride + b * (2 * d_idx) + c * 8;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(dst + d_idx) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (Kr) {   // chunks divides 32: a row's chunks are aligned consecutive lanes
        for (int o = 1; o < chunks; o <<= 1) {
            hi2 += __shfl_xor_sync(0xFFFFFFFFu, hi2, o);
            lo2 += __shfl_xor_sync(0xFFFFFFFFu, lo2, o);
        }
        if (valid && c == 0)
            Kr[seq * kr_seq_stride + b] =
                (sqrtf(lo2) + 6.103515625e-05f * sqrtf(hi2)) * (1.0f + 1.52587890625e-05f);
    }
}

}  // namespace
}  // namespace sfa

extern "C" int sfa_pool_index_keys(const void *X, int x_dtype, int64_t x_seq_stride, int n_seq,
                                   int d_idx, int compress_ratio, int64_t blk_begin,
                                   int64_t blk_end, void *Kbar, int64_t kbar_seq_stride,
                                   float *Kbar_r, int64_t kr_seq_stride, sfa_stream_t stream) {
    using namespace sfa;
    if (!X || !Kbar || n_seq < 1 || compress_ratio < 1 || compress_ratio > 64) return SFA_ERR_INVALID_ARG;
    if (x_dtype != SFA_BF16 && x_dtype != SFA_F32) return SFA_ERR_INVALID_ARG;
    if (d_idx != 32 && d_idx != 64 && d_idx != 96 && d_idx != 128) return SFA_ERR_UNSUPPORTED;
    if (blk_begin < 0 || blk_end < blk_begin) return SFA_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Kbar)) return SFA_ERR_INVALID_ARG;
    if (x_seq_stride < blk_end * compress_ratio * d_idx) return SFA_ERR_INVALID_ARG;
    if (kbar_seq_stride < blk_end * 2 * d_idx || kbar_seq_stride % 8 != 0) return SFA_ERR_INVALID_ARG;
    if (Kbar_r && d_idx == 96) return SFA_ERR_UNSUPPORTED;   // a row's chunks must tile a warp
    if (Kbar_r && kr_seq_stride < blk_end) return SFA_ERR_INVALID_ARG;
    const size_t esz = x_dtype == SFA_BF16 ? 2 : 4;
    if ((x_seq_stride * esz) % 16 != 0) return SFA_ERR_INVALID_ARG;
    const int64_t n_rows = blk_end - blk_begin;
    if (n_rows == 0) return SFA_OK;
    const int64_t threads = n_rows * (d_idx / 8);
    const int64_t nblk = (threads + 255) / 256;
    if (nblk > 0x7FFFFFFF || n_seq > 65535) return SFA_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)nblk, (unsigned)n_seq);
    auto *out = reinterpret_cast<__nv_bfloat16 *>(Kbar);
    const cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e =
        x_dtype == SFA_BF16
            ? launch_pdl(pool_kernel<__nv_bfloat16>, grid, dim3(256), 0, st,
                         reinterpret_cast<const __nv_bfloat16 *>(X), x_seq_stride, d_idx,
                         compress_ratio, blk_begin, n_rows, out, kbar_seq_stride, Kbar_r,
                         kr_seq_stride)
            : launch_pdl(pool_kernel<float>, grid, dim3(256), 0, st,
                         reinterpret_cast<const float *>(X), x_seq_stride, d_idx,
                         compress_ratio, blk_begin, n_rows, out, kbar_seq_stride, Kbar_r,
                         kr_seq_stride);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}
