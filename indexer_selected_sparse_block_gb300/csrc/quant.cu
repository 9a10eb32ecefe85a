// quant.cu -- q8_0 quantization of KV cache rows (sfa_quantize_kv_q8_0).
//
// The qwen4exp commits in llama.cpp let the QSA attention path read a quantized KV cache; q8_0
// is the 8-bit block format of the llama.cpp caches described there.  Each row of d elements
// is cut into blocks of 32.  Per block: delta = max |x| / 127 in binary32, each code is x / delta
// (binary32) rounded half away from zero (0 when delta = 0), and the stored scale is delta
// rounded to binary16 with ties to even.  A cache row holds the d int8 codes, the d/32
// binary16 scales, and zero bytes up to a multiple of 16.
//
// One warp per block: lane j holds element j, the block maximum comes from a shuffle tree,
// every lane writes its code and lane 0 the scale; the lanes of a row's last block also write
// its padding.  Bytes per row: d * sizeof(x) read, q8_row_bytes(d) written.
#include "sfa_common.cuh"

namespace sfa {
namespace {

__device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_float(float v) { return v; }

template <typename T>
__global__ void __launch_bounds__(256) quant_q8_kernel(const T *__restrict__ X, int64_t n_inner,
                                                       int d, int64_t x_outer_stride,
                                                       uint8_t *__restrict__ Y,
                                                       int64_t y_outer_stride, int64_t n_blocks,
                                                       int32_t *status) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t blk = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (blk >= n_blocks) return;   // whole warps: blk is the same for all 32 lanes
    const int nb = d / 32, rb = q8_row_bytes(d);
    const int64_t row = blk / nb;
    const int b = (int)(blk - row * nb);
    const int64_t o = row / n_inner, i = row - o * n_inner;
    const T *xr = X + o * x_outer_stride + i * d;
    uint8_t *yr = Y + o * y_outer_stride + i * rb;
    const float x = to_float(xr[b * 32 + lane]);
    float amax = fabsf(x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const float delta = __fdiv_rn(amax, 127.f);
    const int q = delta == 0.f ? 0 : (int)roundf(__fdiv_rn(x, delta));
    yr[b * 32 + lane] = (uint8_t)(int8_t)q;
    if (lane == 0) {
        const __half h = __float2half_rn(delta);
        *reinterpret_cast<__half *>(yr + d + 2 * b) = h;
        if (__hisinf(h)) set_status(status, SFA_DEV_FP16_RANGE);
    }
    const int used = d + d / 16;
    if (b == nb - 1 && lane < rb - used) yr[used + lane] = 0;
}

}  // namespace
}  // namespace sfa

extern "C" size_t sfa_q8_0_row_bytes(int d) {
    return d > 0 && d % 32 == 0 ? (size_t)sfa::q8_row_bytes(d) : 0;
}

extern "C" int sfa_quantize_kv_q8_0(const void *X, int x_dtype, int64_t n_outer, int64_t n_inner,
                                    int d, int64_t x_outer_stride, void *Y,
                                    int64_t y_outer_stride, int32_t *dev_status,
                                    sfa_stream_t stream) {
    using namespace sfa;
    if (!X || !Y) return SFA_ERR_INVALID_ARG;
    if (x_dtype != SFA_BF16 && x_dtype != SFA_F32) return SFA_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 512 && d != 576) return SFA_ERR_UNSUPPORTED;
    if (n_outer < 0 || n_inner < 0) return SFA_ERR_INVALID_ARG;
    const int64_t rb = q8_row_bytes(d);
    if (n_outer > 1 && (x_outer_stride < n_inner * d || y_outer_stride < n_inner * rb))
        return SFA_ERR_INVALID_ARG;
    if (!aligned16(Y) || y_outer_stride % 16 != 0) return SFA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(X) % (x_dtype == SFA_BF16 ? 2 : 4) != 0) return SFA_ERR_INVALID_ARG;
    const int64_t n_blocks = n_outer * n_inner * (d / 32);
    if (n_blocks == 0) return SFA_OK;
    const int64_t grid = (n_blocks * 32 + 255) / 256;
    if (grid > 0x7FFFFFFF) return SFA_ERR_UNSUPPORTED;
    auto *y = reinterpret_cast<uint8_t *>(Y);
    const cudaError_t e =
        x_dtype == SFA_BF16
            ? launch_pdl(quant_q8_kernel<__nv_bfloat16>, dim3((unsigned)grid), dim3(256), 0,
                         (cudaStream_t)stream, reinterpret_cast<const __nv_bfloat16 *>(X), n_inner,
                         d, x_outer_stride, y, y_outer_stride, n_blocks, dev_status)
            : launch_pdl(quant_q8_kernel<float>, dim3((unsigned)grid), dim3(256), 0,
                         (cudaStream_t)stream, reinterpret_cast<const float *>(X), n_inner, d,
                         x_outer_stride, y, y_outer_stride, n_blocks, dev_status);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}
