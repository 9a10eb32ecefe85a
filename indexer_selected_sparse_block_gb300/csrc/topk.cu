// topk.cu -- the budget rule: the indexer_top_k best blocks of each query (sfa_topk_blocks).
//
// The budget holds the indexer_top_k best blocks; the tail that does not fill a block is
// attended anyway, and a query that sees no more blocks than the budget keeps them all
// (llama.cpp commit "model: add Qwen3.8-Flash-Next (qwen4exp)", QSA paragraphs).
// Order: score descending, then block index ascending (the tie rule of this library).  The
// kept ids are written ascending and the row is padded with -1 (the sparse index rows of
// llama.cpp PR #27970 "CUDA + ggml: add sparse-fa for DSV4/GLM" are padded the same way).
//
// Exact and deterministic without sorting: an MSB-first radix select over the 32-bit
// order-preserving image of each score finds the k-th largest key T and how many of the
// keys equal to T are taken (the lowest-index ones); a stable compaction in index order then
// emits the kept blocks already ascending.  Long rows are cut into chunks: one CTA selects
// the local top-k of each chunk (the global top-k lies in the union of the local ones, as
// the order is total), and a second CTA per query selects from the candidates.
#include "sfa_common.cuh"

namespace sfa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCand = 16384;     // candidates per query entering the merge
constexpr int kMaxChunk = 32768;    // scores per chunk CTA
constexpr int kBaseChunk = 8192;
constexpr int kMaxChunks = 256;     // chunks per query

// Order-preserving image of a score: larger score -> larger key; -0 == +0; NaN lowest.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelShared {
    int hist[kWarps][256];
    int warp_tot[kWarps];
    uint32_t prefix, mask;
    int remaining;
};

// Exclusive block-wide prefix sum of one int per thread.
__device__ __forceinline__ int block_excl_scan(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int base = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const int t = warp_tot[w];
        if (w < warp) base += t;
        total += t;
    }
    __syncthreads();
    return base + x - v;
}

// Selects the k largest of keys[0..n) (ties: lower index first), n > k.  Calls
// emit(index, rank) for each kept item with rank = its position in index order (0..k-1).
template <typename Emit>
__device__ void cta_select(const uint32_t *keys, int n, int k, SelShared &sh, Emit emit) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        sh.prefix = 0;
        sh.mask = 0;
        sh.remaining = k;
    }
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < kWarps * 256; i += kThreads) (&sh.hist[0][0])[i] = 0;
        __syncthreads();
        const uint32_t prefix = sh.prefix, mask = sh.mask;
        for (int i = tid; i < n; i += kThreads) {
            const uint32_t key = keys[i];
            if ((key & mask) == prefix) atomicAdd(&sh.hist[warp][(key >> shift) & 255u], 1);
        }
        __syncthreads();
        // reduce the per-warp histograms into row 0
        for (int b = tid; b < 256; b += kThreads) {
            int s = 0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += sh.hist[w][b];
            sh.hist[0][b] = s;
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns digits 255-8l .. 248-8l (descending)
            int c[8], local = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                c[e] = sh.hist[0][255 - 8 * lane - e];
                local += c[e];
            }
            int incl = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = incl - local;
            const int rem = sh.remaining;
            if (excl < rem && rem <= incl) {
                int cum = excl;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (cum + c[e] >= rem) {
                        const uint32_t digit = (uint32_t)(255 - 8 * lane - e);
                        sh.prefix = prefix | (digit << shift);
                        sh.mask = mask | (255u << shift);
                        sh.remaining = rem - cum;
                        break;
                    }
                    cum += c[e];
                }
            }
        }
        __syncthreads();
    }
    const uint32_t T = sh.prefix;
    const int take_eq = sh.remaining;  // how many keys equal to T are kept (lowest index first)
    // stable compaction in index order over contiguous per-thread ranges
    const int per = (n + kThreads - 1) / kThreads;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int n_eq = 0;
    for (int i = lo; i < hi; ++i) n_eq += keys[i] == T;
    int tot;
    int eq_before = block_excl_scan(n_eq, sh.warp_tot, tot);
    int n_sel = 0;
    {
        int e = eq_before;
        for (int i = lo; i < hi; ++i) {
            const uint32_t key = keys[i];
            if (key > T) ++n_sel;
            else if (key == T) { n_sel += e < take_eq; ++e; }
        }
    }
    int rank = block_excl_scan(n_sel, sh.warp_tot, tot);
    int e = eq_before;
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = keys[i];
        bool keep = key > T;
        if (key == T) { keep = e < take_eq; ++e; }
        if (keep) emit(i, rank++);
    }
    __syncthreads();
}

__device__ __forceinline__ int visible_blocks(const int32_t *q_pos, int i, int cr, int64_t n_blk_max,
                                              int32_t *status) {
    const int pos = q_pos[i];
    if (pos < 0) {
        set_status(status, SFA_DEV_BAD_QUERY);
        return 0;
    }
    const int64_t b = (int64_t)(pos + 1) / cr;
    if (b > n_blk_max) {
        set_status(status, SFA_DEV_BAD_QUERY);
        return (int)n_blk_max;
    }
    return (int)b;
}

struct TopkParams {
    const float *scores;
    const int32_t *q_pos;
    int32_t *blk_idx, *n_sel;
    uint32_t *cand_key;
    int32_t *cand_id, *cand_n;
    int32_t *status;
    int64_t score_stride, n_blk_max;
    int cr, top_k, chunk, n_chunks;
};

// grid (n_chunks, n_q).  Rows that fit the budget, or one chunk, are finished here.
__global__ void __launch_bounds__(kThreads) topk_chunk_kernel(const TopkParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    SelShared &sh = *reinterpret_cast<SelShared *>(smem);
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + sizeof(SelShared));
    const int i = blockIdx.y, c = blockIdx.x;
    const int B = visible_blocks(p.q_pos, i, p.cr, p.n_blk_max, c == 0 ? p.status : nullptr);
    const int k = p.top_k;
    int32_t *out = p.blk_idx + (int64_t)i * k;
    if (B <= k) {  // every block fits the budget
        if (c == 0) {
            for (int j = threadIdx.x; j < k; j += kThreads) out[j] = j < B ? j : -1;
            if (threadIdx.x == 0) p.n_sel[i] = B;
        }
        return;
    }
    const int b0 = c * p.chunk;
    const int n = min(B - b0, p.chunk);
    const bool single = B <= p.chunk;
    if (n <= 0) {
        if (threadIdx.x == 0) p.cand_n[(int64_t)i * p.n_chunks + c] = 0;
        return;
    }
    const float *row = p.scores + (int64_t)i * p.score_stride + b0;
    for (int j = threadIdx.x; j < n; j += kThreads) keys[j] = order_key(row[j]);
    __syncthreads();
    if (single) {
        cta_select(keys, n, k, sh, [&](int idx, int rank) { out[rank] = b0 + idx; });
        if (threadIdx.x == 0) p.n_sel[i] = k;
        return;
    }
    uint32_t *ck = p.cand_key + ((int64_t)i * p.n_chunks + c) * k;
    int32_t *ci = p.cand_id + ((int64_t)i * p.n_chunks + c) * k;
    if (n <= k) {
        for (int j = threadIdx.x; j < n; j += kThreads) {
            ck[j] = keys[j];
            ci[j] = b0 + j;
        }
        if (threadIdx.x == 0) p.cand_n[(int64_t)i * p.n_chunks + c] = n;
        return;
    }
    cta_select(keys, n, k, sh, [&](int idx, int rank) {
        ck[rank] = keys[idx];
        ci[rank] = b0 + idx;
    });
    if (threadIdx.x == 0) p.cand_n[(int64_t)i * p.n_chunks + c] = k;
}

// grid (n_q).  Merges the per-chunk candidates of rows longer than one chunk.
__global__ void __launch_bounds__(kThreads) topk_merge_kernel(const TopkParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    SelShared &sh = *reinterpret_cast<SelShared *>(smem);
    __shared__ int s_off[kMaxChunks + 1];
    const int i = blockIdx.x;
    const int B = visible_blocks(p.q_pos, i, p.cr, p.n_blk_max, nullptr);
    const int k = p.top_k;
    if (B <= k || B <= p.chunk) return;
    const int nc = (B + p.chunk - 1) / p.chunk;
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + sizeof(SelShared));
    int32_t *ids = reinterpret_cast<int32_t *>(keys + (size_t)p.n_chunks * k);
    if (threadIdx.x == 0) {
        int off = 0;
        for (int c = 0; c < nc; ++c) {
            s_off[c] = off;
            off += p.cand_n[(int64_t)i * p.n_chunks + c];
        }
        s_off[nc] = off;
    }
    __syncthreads();
    const int m = s_off[nc];
    for (int c = 0; c < nc; ++c) {
        const int cnt = s_off[c + 1] - s_off[c];
        const uint32_t *ck = p.cand_key + ((int64_t)i * p.n_chunks + c) * k;
        const int32_t *ci = p.cand_id + ((int64_t)i * p.n_chunks + c) * k;
        for (int j = threadIdx.x; j < cnt; j += kThreads) {
            keys[s_off[c] + j] = ck[j];
            ids[s_off[c] + j] = ci[j];
        }
    }
    __syncthreads();
    int32_t *out = p.blk_idx + (int64_t)i * k;
    cta_select(keys, m, k, sh, [&](int idx, int rank) { out[rank] = ids[idx]; });
    if (threadIdx.x == 0) p.n_sel[i] = k;
}

// Chunk length for rows of up to n_blk_max scores (0 when unsupported).
int chunk_len(int64_t n_blk_max, int top_k) {
    int64_t ch = kBaseChunk;
    const int64_t max_chunks = min(kMaxCand / top_k, kMaxChunks);
    if (max_chunks < 1) return 0;
    while ((n_blk_max + ch - 1) / ch > max_chunks) ch += 1024;
    return ch > kMaxChunk ? 0 : (int)ch;
}

}  // namespace
}  // namespace sfa

extern "C" size_t sfa_topk_workspace_bytes(int n_q, int64_t n_blk_max, int top_k) {
    using namespace sfa;
    if (n_q <= 0 || top_k <= 0 || n_blk_max <= 0) return 0;
    const int ch = chunk_len(n_blk_max, top_k);
    if (ch == 0) return 0;
    const int64_t nc = (n_blk_max + ch - 1) / ch;
    if (nc <= 1) return 0;
    return (size_t)n_q * nc * ((size_t)top_k * 8 + 4) + 256;
}

extern "C" int sfa_topk_blocks(const float *scores, int64_t score_stride, const int32_t *q_pos,
                               int n_q, int compress_ratio, int top_k, int64_t n_blk_max,
                               int32_t *blk_idx, int32_t *n_sel, void *workspace,
                               size_t workspace_bytes, int32_t *dev_status,
                               sfa_stream_t stream) {
    using namespace sfa;
    if (!q_pos || !blk_idx || !n_sel || n_q < 0 || compress_ratio < 1 || n_blk_max < 0)
        return SFA_ERR_INVALID_ARG;
    if (top_k < 1 || top_k > 2048) return SFA_ERR_UNSUPPORTED;
    if (n_blk_max > 0 && (!scores || score_stride < n_blk_max)) return SFA_ERR_INVALID_ARG;
    if (n_q == 0) return SFA_OK;
    const int64_t nb = n_blk_max > 0 ? n_blk_max : 1;
    const int ch = chunk_len(nb, top_k);
    if (ch == 0) return SFA_ERR_UNSUPPORTED;
    const int nc = (int)((nb + ch - 1) / ch);
    const size_t need = sfa_topk_workspace_bytes(n_q, nb, top_k);
    if (need > 0 && (!workspace || workspace_bytes < need)) return SFA_ERR_WORKSPACE;
    if (n_q > 65535) return SFA_ERR_UNSUPPORTED;
    TopkParams p{};
    p.scores = scores;
    p.q_pos = q_pos;
    p.blk_idx = blk_idx;
    p.n_sel = n_sel;
    p.status = dev_status;
    p.score_stride = score_stride;
    p.n_blk_max = n_blk_max;
    p.cr = compress_ratio;
    p.top_k = top_k;
    p.chunk = ch;
    p.n_chunks = nc;
    if (need > 0) {
        uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
        const size_t n_cand = (size_t)n_q * nc * top_k;
        p.cand_key = reinterpret_cast<uint32_t *>(ws);
        p.cand_id = reinterpret_cast<int32_t *>(ws + n_cand * 4);
        p.cand_n = reinterpret_cast<int32_t *>(ws + n_cand * 8);
    }
    const cudaStream_t st = (cudaStream_t)stream;
    const size_t smem1 = sizeof(SelShared) + (size_t)ch * 4;
    static bool attr = false;
    if (!attr) {
        if (!allow_max_dynamic_smem(topk_chunk_kernel) || !allow_max_dynamic_smem(topk_merge_kernel))
            return SFA_ERR_CUDA;
        attr = true;
    }
    topk_chunk_kernel<<<dim3(nc, n_q), kThreads, smem1, st>>>(p);
    SFA_CHECK_LAUNCH();
    if (nc > 1) {
        const size_t smem2 = sizeof(SelShared) + (size_t)nc * top_k * 8;
        topk_merge_kernel<<<n_q, kThreads, smem2, st>>>(p);
        SFA_CHECK_LAUNCH();
    }
    return SFA_OK;
}
