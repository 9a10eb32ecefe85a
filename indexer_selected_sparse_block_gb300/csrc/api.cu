// api.cu -- status strings, the device status read-back, the per-device SM count cache, and the
// row copy of sfa_copy_cache_rows.
#include <mutex>
#include <set>
#include <utility>

#include "sfa_common.cuh"

namespace sfa {

int device_sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

namespace {
std::mutex g_smem_mu;
std::set<std::pair<int, const void *>> g_smem_raised;   // (device, kernel)
}  // namespace

bool smem_limit_raised(const void *kernel) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lock(g_smem_mu);
    return g_smem_raised.count({dev, kernel}) != 0;
}

void mark_smem_limit_raised(const void *kernel) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    std::lock_guard<std::mutex> lock(g_smem_mu);
    g_smem_raised.insert({dev, kernel});
}

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

void *current_context() {
    typedef CUresult (*GetCtxFn)(CUcontext *);
    static GetCtxFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<GetCtxFn>(ptr);
    });
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return reinterpret_cast<void *>(ctx);
}

}  // namespace sfa

extern "C" const char *sfa_status_string(int status) {
    switch (status) {
        case SFA_OK: return "SFA_OK";
        case SFA_ERR_INVALID_ARG: return "SFA_ERR_INVALID_ARG: an argument the call cannot accept";
        case SFA_ERR_UNSUPPORTED: return "SFA_ERR_UNSUPPORTED: a shape the library has no kernel for";
        case SFA_ERR_CUDA: return "SFA_ERR_CUDA: the CUDA runtime reported an error";
        case SFA_ERR_WORKSPACE: return "SFA_ERR_WORKSPACE: workspace missing or too small";
        default: return "unknown sfa status";
    }
}

namespace sfa {
namespace {

// Rows of row_bytes bytes from src (pitch sp) to dst (pitch dp), either side device memory or
// page-locked host memory the device addresses: SM loads and stores, 16 bytes at a time when
// every address and size allows.  A kernel rather than a copy-engine transfer: a step's few
// hundred kilobytes of inputs arrive in a few microseconds instead of ~10 (the copy engine's
// start-up), and the next kernel follows it by programmatic dependent launch.
__global__ void __launch_bounds__(256)
    copy_rows_kernel(uint8_t *__restrict__ dst, int64_t dp, const uint8_t *__restrict__ src,
                     int64_t sp, int64_t row_bytes, int64_t n_rows, int vec16) {
    pdl_wait();
    const int64_t per_row = vec16 ? row_bytes >> 4 : row_bytes;
    const int64_t total = per_row * n_rows;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
        const int64_t r = e / per_row, c = e - r * per_row;
        if (vec16)
            *reinterpret_cast<uint4 *>(dst + r * dp + 16 * c) =
                *reinterpret_cast<const uint4 *>(src + r * sp + 16 * c);
        else
            dst[r * dp + c] = src[r * sp + c];
    }
}

// Several such copies in one launch: copy blockIdx.y of the list.
struct RowCopies {
    sfa_row_copy c[SFA_MAX_ROW_COPIES];
    int vec16[SFA_MAX_ROW_COPIES];
};
__global__ void __launch_bounds__(256) copy_rows_multi_kernel(const RowCopies rc) {
    pdl_wait();
    const sfa_row_copy &c = rc.c[blockIdx.y];
    const int vec16 = rc.vec16[blockIdx.y];
    uint8_t *dst = reinterpret_cast<uint8_t *>(c.dst);
    const uint8_t *src = reinterpret_cast<const uint8_t *>(c.src);
    const int64_t per_row = vec16 ? c.row_bytes >> 4 : c.row_bytes;
    const int64_t total = per_row * c.n_rows;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
        const int64_t r = e / per_row, k = e - r * per_row;
        if (vec16)
            *reinterpret_cast<uint4 *>(dst + r * c.dst_pitch + 16 * k) =
                *reinterpret_cast<const uint4 *>(src + r * c.src_pitch + 16 * k);
        else
            dst[r * c.dst_pitch + k] = src[r * c.src_pitch + k];
    }
}

bool copy_valid(const sfa_row_copy &c) {
    return c.n_rows >= 0 && c.row_bytes >= 1 && c.dst_pitch >= c.row_bytes &&
           c.src_pitch >= c.row_bytes && (c.n_rows == 0 || (c.dst && c.src));
}
bool copy_vec16(const sfa_row_copy &c) {
    return aligned16(c.dst) && aligned16(c.src) && c.dst_pitch % 16 == 0 &&
           c.src_pitch % 16 == 0 && c.row_bytes % 16 == 0;
}

}  // namespace
}  // namespace sfa

extern "C" int sfa_copy_cache_rows_multi(int n, const sfa_row_copy *copies, sfa_stream_t stream) {
    using namespace sfa;
    if (n < 0 || n > SFA_MAX_ROW_COPIES || (n > 0 && !copies)) return SFA_ERR_INVALID_ARG;
    RowCopies rc{};
    int64_t most = 0;
    int m = 0;
    for (int k = 0; k < n; ++k) {
        if (!copy_valid(copies[k])) return SFA_ERR_INVALID_ARG;
        if (copies[k].n_rows == 0) continue;
        rc.c[m] = copies[k];
        rc.vec16[m] = copy_vec16(copies[k]);
        const int64_t t = (rc.vec16[m] ? copies[k].row_bytes / 16 : copies[k].row_bytes) *
                          copies[k].n_rows;
        most = t > most ? t : most;
        ++m;
    }
    if (m == 0) return SFA_OK;
    int64_t blocks = (most + 255) / 256;
    const int64_t cap = 4 * (int64_t)device_sm_count();
    if (blocks > cap) blocks = cap;
    if (launch_pdl(copy_rows_multi_kernel, dim3((unsigned)blocks, (unsigned)m), dim3(256), 0,
                   (cudaStream_t)stream, rc) != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

extern "C" int sfa_copy_cache_rows(void *dst, int64_t dst_pitch, const void *src,
                                   int64_t src_pitch, int64_t row_bytes, int64_t n_rows,
                                   sfa_stream_t stream) {
    using namespace sfa;
    if (n_rows < 0 || row_bytes < 1 || dst_pitch < row_bytes || src_pitch < row_bytes)
        return SFA_ERR_INVALID_ARG;
    if (n_rows == 0) return SFA_OK;
    if (!dst || !src) return SFA_ERR_INVALID_ARG;
    const bool vec16 = aligned16(dst) && aligned16(src) && dst_pitch % 16 == 0 &&
                       src_pitch % 16 == 0 && row_bytes % 16 == 0;
    const int64_t total = (vec16 ? row_bytes / 16 : row_bytes) * n_rows;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = 4 * (int64_t)device_sm_count();
    if (blocks > cap) blocks = cap;
    if (launch_pdl(copy_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, (cudaStream_t)stream,
                   reinterpret_cast<uint8_t *>(dst), dst_pitch, reinterpret_cast<const uint8_t *>(src),
                   src_pitch, row_bytes, n_rows, (int)vec16) != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

extern "C" int sfa_read_device_status(const int32_t *dev_status, int32_t *host_out,
                                      sfa_stream_t stream) {
    if (!dev_status || !host_out) return SFA_ERR_INVALID_ARG;
    if (cudaMemcpyAsync(host_out, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost,
                        (cudaStream_t)stream) != cudaSuccess)
        return SFA_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SFA_ERR_CUDA;
    return SFA_OK;
}
