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
// Optionally the pooled key is normalised and rotated before it is split (the indexer key
// cache holds raw keys because pooling precedes the norm and the rotation; the indexer ropes
// with the main attention's rotary width -- llama.cpp commit "model: add Qwen3.8-Flash-Next
// (qwen4exp)", indexer key cache paragraph): RMS or layer norm over the row (statistics by a
// shuffle sum over the row's lanes, fp32), then the first n_rot dims turned pairwise at the
// block's position b*cr + pos_offset, NeoX pairs (j, j + n_rot/2) through a shuffle with the
// partner lane, or adjacent pairs (2j, 2j + 1) within a thread.  Angles and their sines and
// cosines are computed in double: at positions near 1e6 an fp32 angle is off by ~0.06 rad.
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

struct KeyTransform {
    int norm;                    // 0 none, 1 RMS, 2 layer
    const float *gamma, *beta;   // [d_idx] gain, [d_idx] bias (layer norm)
    float eps;
    int n_rot;                   // rotated dims (0: none)
    double log2_base;            // log2 of the rotary base
    int neox;                    // 1: pairs (j, j + n_rot/2); 0: (2j, 2j + 1)
    int64_t pos_offset;          // block b sits at position b * cr + pos_offset
};

// Paged layout: the raw key of position t of sequence s sits in row cell_of[s * stride + t] of
// a flat [n_cells][d_idx] array; blocks are still cut on positions.  cell_of null: per-sequence
// layout.  A cell outside [0, n_cells) reads as a zero row and raises SFA_DEV_BAD_CELL.
struct CellMap {
    const int32_t *cell_of;
    int64_t stride, n_cells;
    int32_t *status;
};

// Sum over the `chunks` lanes that hold one row (aligned groups; chunks divides 32).
__device__ __forceinline__ float row_sum(float v, int chunks) {
    for (int o = 1; o < chunks; o <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// grid: (ceil(rows * chunks / 256), n_seq); one thread per (pooled row, 8-element chunk).
template <typename T>
__global__ void __launch_bounds__(256) pool_kernel(const T *__restrict__ X, int64_t x_seq_stride,
                                                   int d_idx, int cr, int64_t blk_begin,
                                                   int64_t n_rows, __nv_bfloat16 *__restrict__ Kbar,
                                                   int64_t kbar_seq_stride, float *__restrict__ Kr,
                                                   int64_t kr_seq_stride, const KeyTransform tf,
                                                   const CellMap cm) {
    pdl_wait();
    const int chunks = d_idx >> 3;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool valid = gid < n_rows * chunks;
    const int64_t b = blk_begin + (valid ? gid / chunks : 0);
    const int c = (int)(gid % chunks);
    const int64_t seq = blockIdx.y;
    float mv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // this chunk of the pooled row
    if (valid) {
        const T *src = X + seq * x_seq_stride + b * cr * d_idx + c * 8;
        auto load_row = [&](int t, float (&v)[8]) {   // chunk c of the raw key of token b*cr + t
            if (!cm.cell_of) {
                Vec8<T>::load(src + (int64_t)t * d_idx, v);
                return;
            }
            const int32_t cell = __ldg(cm.cell_of + seq * cm.stride + b * cr + t);
            if (cell >= 0 && (int64_t)cell < cm.n_cells) {
                Vec8<T>::load(X + (int64_t)cell * d_idx + c * 8, v);
                return;
            }
            set_status(cm.status, SFA_DEV_BAD_CELL);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
        };
        float sum[8];
        load_row(0, sum);
        for (int t = 1; t < cr; ++t) {
            float v[8];
            load_row(t, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) sum[i] += v[i];
        }
        const float rcr = (float)cr;
#pragma unroll
        for (int i = 0; i < 8; ++i) mv[i] = __fdiv_rn(sum[i], rcr);
    }
    if (tf.norm) {   // uniform: every lane takes part in the row sums
        float mu = 0.f;
        if (tf.norm == 2) {
            float s1 = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) s1 += mv[i];
            mu = __fdiv_rn(row_sum(s1, chunks), (float)d_idx);
        }
        float s2 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s2 = fmaf(mv[i] - mu, mv[i] - mu, s2);
        const float r = __fsqrt_rn(__fdiv_rn(row_sum(s2, chunks), (float)d_idx) + tf.eps);
        if (valid) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int d = c * 8 + i;
                const float y = __fdiv_rn(mv[i] - mu, r) * __ldg(tf.gamma + d);
                mv[i] = tf.norm == 2 ? y + __ldg(tf.beta + d) : y;
            }
        }
    }
    if (tf.n_rot) {
        const double pos = (double)(b * cr + tf.pos_offset);
        const int d0 = c * 8;
        if (tf.neox) {   // pairs (j, j + half): whole chunks, the partner half/8 lanes away
            const int half = tf.n_rot / 2;
            const int lane = threadIdx.x & 31;
            const int src_lane = d0 < half ? lane + half / 8 : (d0 < tf.n_rot ? lane - half / 8 : lane);
            float pv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pv[i] = __shfl_sync(0xFFFFFFFFu, mv[i], src_lane);
            if (valid && d0 < tf.n_rot) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int d = d0 + i, j = d < half ? d : d - half;
                    double sn, cs;
                    sincos(pos * exp2(-2.0 * j / tf.n_rot * tf.log2_base), &sn, &cs);
                    const float fc = (float)cs, fs = (float)sn;
                    mv[i] = d < half ? fmaf(mv[i], fc, -pv[i] * fs)    // x_j cos - x_{j+half} sin
                                     : fmaf(pv[i], fs, mv[i] * fc);   // x_j sin + x_{j+half} cos
                }
            }
        } else if (valid && d0 < tf.n_rot) {   // pairs (2j, 2j + 1) inside the chunk
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const int j = (d0 + i) / 2;
                double sn, cs;
                sincos(pos * exp2(-2.0 * j / tf.n_rot * tf.log2_base), &sn, &cs);
                const float fc = (float)cs, fs = (float)sn, a = mv[i], bb = mv[i + 1];
                mv[i] = fmaf(a, fc, -bb * fs);
                mv[i + 1] = fmaf(a, fs, bb * fc);
            }
        }
    }
    float lo2 = 0.f, hi2 = 0.f;
    if (valid) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float m0 = mv[2 * i], m1 = mv[2 * i + 1];
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

namespace sfa {
namespace {

int run_pool(const void *X, int x_dtype, int64_t x_seq_stride, int n_seq, int d_idx,
             int compress_ratio, int64_t blk_begin, int64_t blk_end, void *Kbar,
             int64_t kbar_seq_stride, float *Kbar_r, int64_t kr_seq_stride,
             const KeyTransform &tf, cudaStream_t st, const CellMap &cm = CellMap{}) {
    if (!X || !Kbar || n_seq < 1 || compress_ratio < 1 || compress_ratio > 64) return SFA_ERR_INVALID_ARG;
    if (x_dtype != SFA_BF16 && x_dtype != SFA_F32) return SFA_ERR_INVALID_ARG;
    if (d_idx != 32 && d_idx != 64 && d_idx != 96 && d_idx != 128) return SFA_ERR_UNSUPPORTED;
    if (blk_begin < 0 || blk_end < blk_begin) return SFA_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Kbar)) return SFA_ERR_INVALID_ARG;
    if (cm.cell_of) {   // x_seq_stride is unused: the map gives every row
        if (cm.n_cells < 1 || cm.stride < blk_end * compress_ratio) return SFA_ERR_INVALID_ARG;
    } else if (x_seq_stride < blk_end * compress_ratio * d_idx) {
        return SFA_ERR_INVALID_ARG;
    }
    if (kbar_seq_stride < blk_end * 2 * d_idx || kbar_seq_stride % 8 != 0) return SFA_ERR_INVALID_ARG;
    // the row statistics, the NeoX partner and the bound factors work on whole-warp lane groups
    if ((Kbar_r || tf.norm || tf.n_rot) && d_idx == 96) return SFA_ERR_UNSUPPORTED;
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
    const cudaError_t e =
        x_dtype == SFA_BF16
            ? launch_pdl(pool_kernel<__nv_bfloat16>, grid, dim3(256), 0, st,
                         reinterpret_cast<const __nv_bfloat16 *>(X), x_seq_stride, d_idx,
                         compress_ratio, blk_begin, n_rows, out, kbar_seq_stride, Kbar_r,
                         kr_seq_stride, tf, cm)
            : launch_pdl(pool_kernel<float>, grid, dim3(256), 0, st,
                         reinterpret_cast<const float *>(X), x_seq_stride, d_idx,
                         compress_ratio, blk_begin, n_rows, out, kbar_seq_stride, Kbar_r,
                         kr_seq_stride, tf, cm);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

}  // namespace
}  // namespace sfa

extern "C" int sfa_pool_index_keys(const void *X, int x_dtype, int64_t x_seq_stride, int n_seq,
                                   int d_idx, int compress_ratio, int64_t blk_begin,
                                   int64_t blk_end, void *Kbar, int64_t kbar_seq_stride,
                                   float *Kbar_r, int64_t kr_seq_stride, sfa_stream_t stream) {
    const sfa::KeyTransform none{};
    return sfa::run_pool(X, x_dtype, x_seq_stride, n_seq, d_idx, compress_ratio, blk_begin,
                         blk_end, Kbar, kbar_seq_stride, Kbar_r, kr_seq_stride, none,
                         (cudaStream_t)stream);
}

extern "C" int sfa_pool_index_keys_transformed(const void *X, int x_dtype, int64_t x_seq_stride,
                                               int n_seq, int d_idx, int compress_ratio,
                                               int64_t blk_begin, int64_t blk_end, int norm,
                                               const float *gamma, const float *beta, float eps,
                                               int n_rot, float rope_base, int rope_neox,
                                               int64_t pos_offset, void *Kbar,
                                               int64_t kbar_seq_stride, float *Kbar_r,
                                               int64_t kr_seq_stride, sfa_stream_t stream) {
    using namespace sfa;
    if (norm < 0 || norm > 2) return SFA_ERR_INVALID_ARG;
    if (norm >= 1 && !gamma) return SFA_ERR_INVALID_ARG;
    if (norm == 2 && !beta) return SFA_ERR_INVALID_ARG;
    if (norm && !(eps >= 0.f && isfinite(eps))) return SFA_ERR_INVALID_ARG;
    if (n_rot < 0 || n_rot % 2 != 0 || n_rot > d_idx) return SFA_ERR_INVALID_ARG;
    if (n_rot && rope_neox && n_rot % 16 != 0) return SFA_ERR_UNSUPPORTED;   // whole-chunk pairs
    if (n_rot && !(rope_base > 0.f && isfinite(rope_base))) return SFA_ERR_INVALID_ARG;
    KeyTransform tf{};
    tf.norm = norm;
    tf.gamma = gamma;
    tf.beta = beta;
    tf.eps = eps;
    tf.n_rot = n_rot;
    tf.log2_base = n_rot ? log2((double)rope_base) : 0.0;
    tf.neox = rope_neox ? 1 : 0;
    tf.pos_offset = pos_offset;
    return run_pool(X, x_dtype, x_seq_stride, n_seq, d_idx, compress_ratio, blk_begin, blk_end,
                    Kbar, kbar_seq_stride, Kbar_r, kr_seq_stride, tf, (cudaStream_t)stream);
}

extern "C" int sfa_pool_index_keys_paged(const void *X, int x_dtype, int64_t n_cells,
                                         const int32_t *cell_of, int64_t n_pos_cap, int n_seq,
                                         int d_idx, int compress_ratio, int64_t blk_begin,
                                         int64_t blk_end, void *Kbar, int64_t kbar_seq_stride,
                                         float *Kbar_r, int64_t kr_seq_stride,
                                         int32_t *dev_status, sfa_stream_t stream) {
    if (!cell_of) return SFA_ERR_INVALID_ARG;
    const sfa::KeyTransform none{};
    const sfa::CellMap cm{cell_of, n_pos_cap, n_cells, dev_status};
    return sfa::run_pool(X, x_dtype, 0, n_seq, d_idx, compress_ratio, blk_begin, blk_end, Kbar,
                         kbar_seq_stride, Kbar_r, kr_seq_stride, none, (cudaStream_t)stream, cm);
}
