// topk.cu -- the budget rule: the indexer_top_k best blocks of each query (sfa_topk_blocks).
//
// The budget holds the indexer_top_k best blocks; the tail that does not fill a block is
// attended anyway, and a query that sees no more blocks than the budget keeps them all
// (llama.cpp commit "model: add Qwen3.8-Flash-Next (qwen4exp)", QSA paragraphs).
// Order: score descending, then block index ascending (the tie rule of this library).  The
// kept ids are written ascending and the row is padded with -1 (the sparse index rows of
// llama.cpp PR #27970 "CUDA + ggml: add sparse-fa for DSV4/GLM" are padded the same way).
//
// Exact and deterministic without sorting: a radix select on the order-preserving 32-bit
// image of each score.  One CTA (512 threads, small shared memory, several CTAs per SM so
// that their latency chains overlap) per row chunk; the scores stay in L2 and are read
// three times, coalesced:
//   1. keys' top 12 bits -> 4096-bin histogram; a block-wide scan finds the bin that holds
//      the k-th largest key;
//   2. per warp segment, count the keys above that bin; the keys of the cut bin are gathered
//      (in any order: their ranking below does not depend on it);
//   3. the cut bin's keys get a second 12-bit histogram (bits 19..8); keys above its cut bin
//      are kept, and the few keys sharing the 24-bit cut prefix are ranked by counting in the
//      order (key desc, index asc).  Kept cut-bin keys are marked in a bitmask;
//   4. per warp segment, the kept indices are written in index order (ballots + a scan of
//      the warps' counts), already ascending.
// Degenerate rows (over 2048 keys in the first cut bin, or over 512 sharing a 24-bit prefix
// at the cut) fall back to an 8-bit MSB-first radix select.  Rows are cut into chunks when
// long, or when too few rows exist to fill the GPU; a second CTA per row then selects among
// the chunks' candidates (the global top-k lies in the union of the local ones, as the order
// is total).
#include "sfa_common.cuh"

namespace sfa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;                  // 12-bit digits
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kMaxCand = 2048;               // first cut bin keys resolved on the second digit
constexpr int kMaxTie = 512;                 // keys sharing the 24-bit cut prefix
constexpr int kMaxChunk = 65536;             // scores per chunk CTA
constexpr int kMinChunk = 4096;              // smallest chunk worth a CTA
constexpr int kMaxMerge = 16384;             // candidates per row entering the merge
constexpr int kMaxChunks = 256;              // chunks per row
constexpr int kHistWarps = 8;                // privatised histograms of the fallback

// Order-preserving image of a score: larger score -> larger key; -0 == +0; NaN lowest.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The elements of a selection: either a chunk of one query's score row (row != nullptr:
// key(i) from the score, id b0 + i) or a row's compacted chunk candidates (keys / ids, written
// by this CTA, so read with coherent loads).  One runtime form keeps a single copy of the
// selection code, which runs once per row on an instruction cache that is otherwise cold.
struct SelSrc {
    const float *row;
    const uint32_t *keys;
    const int32_t *ids;
    int b0;
    __device__ __forceinline__ uint32_t key(int i) const {
        return row ? order_key(__ldg(row + i)) : keys[i];
    }
    __device__ __forceinline__ int id(int i) const { return row ? b0 + i : ids[i]; }
};

struct __align__(16) Smem {
    union {
        int hist[kBins];
        int radix_hist[kHistWarps][256];
    };
    int warp_tot[kWarps];
    int warp_keep[kWarps];
    int cut_bin, cut_above, cut_count, n_cand, n_tie;
    uint32_t prefix, mask;
    int remaining;
    uint32_t cand_key[kMaxCand];
    int cand_idx[kMaxCand];
    uint32_t tie_key[kMaxTie];
    int tie_idx[kMaxTie];
};

__device__ __forceinline__ uint32_t lanemask_lt() { return (1u << (threadIdx.x & 31)) - 1u; }
__device__ __forceinline__ int segment_len(int n) {
    return (((n + kWarps - 1) / kWarps) + 31) & ~31;
}
// Exclusive scan of one count per warp (all lanes pass the warp's count): the warp's base.
__device__ __forceinline__ int warp_base_scan(int warp_count, int *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_tot[warp] = warp_count;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    __syncthreads();
    return base;
}

// All threads: the bin of hist[0..kBins) (ordered by key) that holds the k-th largest
// element, with the count above it and its own count, into sh.cut_*.
__device__ __forceinline__ void find_cut(Smem &sh, int k) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int top = kBins - 1 - kBinsPerThread * tid;   // this thread's bins: top .. top-7
    int h[kBinsPerThread], local = 0;
#pragma unroll
    for (int e = 0; e < kBinsPerThread; ++e) {
        h[e] = sh.hist[top - e];
        local += h[e];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sh.warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += sh.warp_tot[w];
    const int excl = base + incl - local;
    if (excl < k && k <= excl + local) {
        int cum = excl;
#pragma unroll
        for (int e = 0; e < kBinsPerThread; ++e) {
            if (cum + h[e] >= k) {
                sh.cut_bin = top - e;
                sh.cut_above = cum;
                sh.cut_count = h[e];
                break;
            }
            cum += h[e];
        }
    }
    __syncthreads();
}

// Writes kept element i at output position rank: its block id, and its key when the
// output is a chunk's candidate list.
__device__ __forceinline__ void emit(const SelSrc &src, int i, int rank, int32_t *out_id,
                                     uint32_t *out_key) {
    out_id[rank] = src.id(i);
    if (out_key) out_key[rank] = src.key(i);
}

// Fallback: 8-bit MSB-first radix select of the k largest keys of src[0..n) (ties: lower
// index first), k < n, written in index order.
__device__ __noinline__ void radix_select(const SelSrc src, int n, int k, int32_t *out_id,
                                          uint32_t *out_key) {
    extern __shared__ __align__(16) uint8_t smem[];
    Smem &sh = *reinterpret_cast<Smem *>(smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        sh.prefix = 0;
        sh.mask = 0;
        sh.remaining = k;
    }
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < kHistWarps * 256; i += kThreads) (&sh.radix_hist[0][0])[i] = 0;
        __syncthreads();
        const uint32_t prefix = sh.prefix, mask = sh.mask;
        for (int i = tid; i < n; i += kThreads) {
            const uint32_t key = src.key(i);
            if ((key & mask) == prefix)
                atomicAdd(&sh.radix_hist[warp & (kHistWarps - 1)][(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid < 256) {
            int s = 0;
            for (int w = 1; w < kHistWarps; ++w) s += sh.radix_hist[w][tid];
            sh.radix_hist[0][tid] += s;
        }
        __syncthreads();
        if (warp == 0) {
            int local = 0;
            for (int e = 0; e < 8; ++e) local += sh.radix_hist[0][255 - 8 * lane - e];
            int incl = local;
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = incl - local;
            const int rem = sh.remaining;
            if (excl < rem && rem <= incl) {
                int cum = excl;
                for (int e = 0; e < 8; ++e) {
                    const int c = sh.radix_hist[0][255 - 8 * lane - e];
                    if (cum + c >= rem) {
                        const uint32_t digit = (uint32_t)(255 - 8 * lane - e);
                        sh.prefix = prefix | (digit << shift);
                        sh.mask = mask | (255u << shift);
                        sh.remaining = rem - cum;
                        break;
                    }
                    cum += c;
                }
            }
        }
        __syncthreads();
    }
    const uint32_t T = sh.prefix;
    const int take_eq = sh.remaining;
    const int seg = segment_len(n);
    const int lo = min(n, warp * seg), hi = min(n, lo + seg);
    int n_eq = 0;
    for (int b = lo; b < hi; b += 32) {
        const int i = b + lane;
        n_eq += __popc(__ballot_sync(0xFFFFFFFFu, i < hi && src.key(i) == T));
    }
    int e = warp_base_scan(n_eq, sh.warp_tot);  // equal keys before this warp's segment
    int n_keep = 0;
    for (int pass = 0; pass < 2; ++pass) {
        int ee = e, rank = 0;
        if (pass == 1) rank = warp_base_scan(n_keep, sh.warp_tot);
        for (int b = lo; b < hi; b += 32) {
            const int i = b + lane;
            const uint32_t key = i < hi ? src.key(i) : 0u;
            const uint32_t eqm = __ballot_sync(0xFFFFFFFFu, i < hi && key == T);
            const bool keep =
                i < hi && (key > T || (key == T && ee + __popc(eqm & lanemask_lt()) < take_eq));
            const uint32_t km = __ballot_sync(0xFFFFFFFFu, keep);
            if (pass == 0) {
                n_keep += __popc(km);
            } else {
                if (keep) emit(src, i, rank + __popc(km & lanemask_lt()), out_id, out_key);
                rank += __popc(km);
            }
            ee += __popc(eqm);
        }
    }
    __syncthreads();
}

// The k largest of src[0..n) (n > k; ties to the lower index), written in index order to
// out_id (and out_key when non-null).  sel[] has one bit per element (zeroed here).
__device__ __noinline__ void select_topk(const SelSrc src, uint32_t *sel, int n, int k,
                                         int32_t *out_id, uint32_t *out_key) {
    extern __shared__ __align__(16) uint8_t smem[];
    Smem &sh = *reinterpret_cast<Smem *>(smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kBins; i += kThreads) sh.hist[i] = 0;
    for (int i = tid; i < (n + 31) / 32; i += kThreads) sel[i] = 0;
    if (tid == 0) {
        sh.n_cand = 0;
        sh.n_tie = 0;
    }
    __syncthreads();
    // 1. histogram of the top 12 key bits (float4 reads when the score row is aligned)
    if (src.row && (reinterpret_cast<uintptr_t>(src.row) & 15u) == 0) {
        const float4 *r4 = reinterpret_cast<const float4 *>(src.row);
        const int n4 = n >> 2;
        for (int j = tid; j < n4; j += kThreads) {
            const float4 v = __ldg(r4 + j);
            atomicAdd(&sh.hist[order_key(v.x) >> 20], 1);
            atomicAdd(&sh.hist[order_key(v.y) >> 20], 1);
            atomicAdd(&sh.hist[order_key(v.z) >> 20], 1);
            atomicAdd(&sh.hist[order_key(v.w) >> 20], 1);
        }
        for (int j = 4 * n4 + tid; j < n; j += kThreads) atomicAdd(&sh.hist[src.key(j) >> 20], 1);
    } else {
        for (int j = tid; j < n; j += kThreads) atomicAdd(&sh.hist[src.key(j) >> 20], 1);
    }
    __syncthreads();
    find_cut(sh, k);
    const uint32_t cut1 = (uint32_t)sh.cut_bin;
    const int need1 = k - sh.cut_above, n_cut1 = sh.cut_count;
    if (n_cut1 > kMaxCand) {
        radix_select(src, n, k, out_id, out_key);
        return;
    }
    // 2. per-warp counts above the cut bin; gather the cut bin's keys
    const int seg = segment_len(n);
    const int lo = min(n, warp * seg), hi = min(n, lo + seg);
    int n_above = 0;
    for (int b = lo; b < hi; b += 32) {
        const int i = b + lane;
        const uint32_t key = i < hi ? src.key(i) : 0u;
        const uint32_t d = key >> 20;
        n_above += __popc(__ballot_sync(0xFFFFFFFFu, i < hi && d > cut1));
        if (i < hi && d == cut1) {
            const int q = atomicAdd(&sh.n_cand, 1);
            sh.cand_key[q] = key;
            sh.cand_idx[q] = i;
        }
    }
    if (lane == 0) sh.warp_keep[warp] = n_above;
    __syncthreads();
    if (need1 == n_cut1) {
        for (int j = tid; j < n_cut1; j += kThreads) {
            const int i = sh.cand_idx[j];
            atomicOr(&sel[i >> 5], 1u << (i & 31));
            atomicAdd(&sh.warp_keep[i / seg], 1);
        }
    } else {
        // 3. the second digit over the cut bin
        for (int i = tid; i < kBins; i += kThreads) sh.hist[i] = 0;
        __syncthreads();
        for (int j = tid; j < n_cut1; j += kThreads)
            atomicAdd(&sh.hist[(sh.cand_key[j] >> 8) & 0xFFFu], 1);
        __syncthreads();
        find_cut(sh, need1);
        const uint32_t cut2 = (uint32_t)sh.cut_bin;
        const int need2 = need1 - sh.cut_above, n_cut2 = sh.cut_count;
        if (n_cut2 > kMaxTie) {
            radix_select(src, n, k, out_id, out_key);
            return;
        }
        for (int j = tid; j < n_cut1; j += kThreads) {
            const uint32_t key = sh.cand_key[j];
            const uint32_t d2 = (key >> 8) & 0xFFFu;
            const int i = sh.cand_idx[j];
            if (d2 > cut2) {
                atomicOr(&sel[i >> 5], 1u << (i & 31));
                atomicAdd(&sh.warp_keep[i / seg], 1);
            } else if (d2 == cut2) {
                const int t = atomicAdd(&sh.n_tie, 1);
                sh.tie_key[t] = key;
                sh.tie_idx[t] = i;
            }
        }
        __syncthreads();
        for (int t = tid; t < n_cut2; t += kThreads) {
            const uint32_t kt = sh.tie_key[t];
            const int it = sh.tie_idx[t];
            int rank = 0;
            if (need2 < n_cut2) {
                for (int u = 0; u < n_cut2; ++u) {
                    const uint32_t ku = sh.tie_key[u];
                    rank += ku > kt || (ku == kt && sh.tie_idx[u] < it);
                }
            }
            if (rank < need2) {
                atomicOr(&sel[it >> 5], 1u << (it & 31));
                atomicAdd(&sh.warp_keep[it / seg], 1);
            }
        }
    }
    __syncthreads();
    // 4. write the kept elements in index order
    const int my_keep = sh.warp_keep[warp];
    int rank = warp_base_scan(my_keep, sh.warp_tot);
    if (my_keep > 0) {
        for (int b = lo; b < hi; b += 32) {
            const int i = b + lane;
            const bool keep =
                i < hi && ((src.key(i) >> 20) > cut1 || ((sel[i >> 5] >> (i & 31)) & 1u));
            const uint32_t m = __ballot_sync(0xFFFFFFFFu, keep);
            if (keep) emit(src, i, rank + __popc(m & lanemask_lt()), out_id, out_key);
            rank += __popc(m);
        }
    }
    __syncthreads();
}

__device__ __forceinline__ int visible_blocks(const int32_t *q_pos, int i, int cr,
                                              int64_t n_blk_max, int32_t *status) {
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
    uint32_t *cand_key, *merged_key;
    int32_t *cand_id, *merged_id, *cand_n;
    int32_t *status;
    int64_t score_stride, n_blk_max;
    int cr, top_k, chunk, n_chunks;
};

// Persistent over (query, chunk) work items, so that each SM's instruction cache stays warm
// across rows.  Rows that fit the budget, or fit one chunk, are finished here.
__global__ void __launch_bounds__(kThreads, 2) topk_chunk_kernel(const TopkParams p, int n_q) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t *sel = reinterpret_cast<uint32_t *>(smem + sizeof(Smem));
    const int k = p.top_k;
    const int n_items = n_q * p.n_chunks;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int i = item / p.n_chunks, c = item % p.n_chunks;
        const int B = visible_blocks(p.q_pos, i, p.cr, p.n_blk_max,
                                     (c == 0 && threadIdx.x == 0) ? p.status : nullptr);
        int32_t *out = p.blk_idx + (int64_t)i * k;
        if (B <= k) {  // every block fits the budget
            if (c == 0) {
                for (int j = threadIdx.x; j < k; j += kThreads) out[j] = j < B ? j : -1;
                if (threadIdx.x == 0) p.n_sel[i] = B;
            }
            continue;
        }
        const int b0 = c * p.chunk;
        const int n = min(B - b0, p.chunk);
        if (n <= 0) {
            if (threadIdx.x == 0) p.cand_n[(int64_t)i * p.n_chunks + c] = 0;
            continue;
        }
        const SelSrc src{p.scores + (int64_t)i * p.score_stride + b0, nullptr, nullptr, b0};
        if (B <= p.chunk) {
            select_topk(src, sel, n, k, out, nullptr);
            if (threadIdx.x == 0) p.n_sel[i] = k;
            continue;
        }
        uint32_t *ck = p.cand_key + ((int64_t)i * p.n_chunks + c) * k;
        int32_t *ci = p.cand_id + ((int64_t)i * p.n_chunks + c) * k;
        if (n <= k) {
            for (int j = threadIdx.x; j < n; j += kThreads) {
                ck[j] = src.key(j);
                ci[j] = b0 + j;
            }
            if (threadIdx.x == 0) p.cand_n[(int64_t)i * p.n_chunks + c] = n;
        } else {
            select_topk(src, sel, n, k, ci, ck);
            if (threadIdx.x == 0) p.cand_n[(int64_t)i * p.n_chunks + c] = k;
        }
    }
}

// grid (n_q).  Selects among the per-chunk candidates of rows cut into chunks: the chunks'
// slots are compacted in chunk order (ids ascend) into the merge area, then selected.
__global__ void __launch_bounds__(kThreads, 2) topk_merge_kernel(const TopkParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t *sel = reinterpret_cast<uint32_t *>(smem + sizeof(Smem));
    __shared__ int s_off[kMaxChunks + 1];
    const int i = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    const int B = visible_blocks(p.q_pos, i, p.cr, p.n_blk_max, nullptr);
    const int k = p.top_k;
    if (B <= k || B <= p.chunk) return;
    const int nc = (B + p.chunk - 1) / p.chunk;
    if (tid < 32) {  // exclusive scan of the chunks' counts (nc <= 256: 8 per lane)
        int c8[8], local = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = lane * 8 + e;
            c8[e] = c < nc ? p.cand_n[(int64_t)i * p.n_chunks + c] : 0;
            local += c8[e];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        int off = incl - local;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = lane * 8 + e;
            if (c <= nc) s_off[c] = off;
            off += c8[e];
        }
    }
    __syncthreads();
    const int m = s_off[nc];
    uint32_t *mk = p.merged_key + (size_t)i * p.n_chunks * k;
    int32_t *mi = p.merged_id + (size_t)i * p.n_chunks * k;
    for (int f = tid; f < nc * k; f += kThreads) {
        const int c = f / k, j = f % k;
        if (j < s_off[c + 1] - s_off[c]) {
            mk[s_off[c] + j] = p.cand_key[((int64_t)i * p.n_chunks + c) * k + j];
            mi[s_off[c] + j] = p.cand_id[((int64_t)i * p.n_chunks + c) * k + j];
        }
    }
    __syncthreads();
    const SelSrc src{nullptr, mk, mi, 0};
    select_topk(src, sel, m, k, p.blk_idx + (int64_t)i * k, nullptr);
    if (tid == 0) p.n_sel[i] = k;
}

// Chunk length for n_q rows of up to n_blk_max scores (0 when unsupported): at most
// kMaxChunk, and short enough that the chunks of all rows fill the GPU when rows are few.
int chunk_len(int n_q, int64_t n_blk_max, int top_k) {
    const int64_t max_chunks = min(kMaxMerge / top_k, kMaxChunks);
    if (max_chunks < 1) return 0;
    int64_t nc = (n_blk_max + kMaxChunk - 1) / kMaxChunk;
    if (nc > max_chunks) return 0;
    const int64_t want = n_q > 0 ? 2 * device_sm_count() / n_q : 1;
    const int64_t by_size = (n_blk_max + kMinChunk - 1) / kMinChunk;
    int64_t more = want < by_size ? want : by_size;
    if (more > max_chunks) more = max_chunks;
    if (more > nc) nc = more;
    int64_t ch = (n_blk_max + nc - 1) / nc;
    ch = (ch + 1023) / 1024 * 1024;
    return ch > kMaxChunk ? kMaxChunk : (int)ch;
}

}  // namespace
}  // namespace sfa

extern "C" size_t sfa_topk_workspace_bytes(int n_q, int64_t n_blk_max, int top_k) {
    using namespace sfa;
    if (n_q <= 0 || top_k <= 0 || n_blk_max <= 0) return 0;
    const int ch = chunk_len(n_q, n_blk_max, top_k);
    if (ch == 0) return 0;
    const int64_t nc = (n_blk_max + ch - 1) / ch;
    if (nc <= 1) return 0;
    // per row: nc * top_k candidate slots and as many merged entries (key + id each) + counts
    return (size_t)n_q * nc * ((size_t)top_k * 16 + 4) + 256;
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
    const int ch = chunk_len(n_q, nb, top_k);
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
        p.merged_key = reinterpret_cast<uint32_t *>(ws + n_cand * 8);
        p.merged_id = reinterpret_cast<int32_t *>(ws + n_cand * 12);
        p.cand_n = reinterpret_cast<int32_t *>(ws + n_cand * 16);
    }
    const cudaStream_t st = (cudaStream_t)stream;
    static bool attr = false;
    if (!attr) {
        if (!allow_max_dynamic_smem(topk_chunk_kernel) || !allow_max_dynamic_smem(topk_merge_kernel))
            return SFA_ERR_CUDA;
        attr = true;
    }
    // shared memory: the fixed part plus one selection bit per element
    const int64_t ch_used = nb < ch ? nb : ch;
    const size_t smem1 = sizeof(Smem) + ((size_t)ch_used + 31) / 32 * 4 + 16;
    int grid1 = 2 * device_sm_count();
    if ((int64_t)grid1 > (int64_t)nc * n_q) grid1 = nc * n_q;
    topk_chunk_kernel<<<grid1, kThreads, smem1, st>>>(p, n_q);
    SFA_CHECK_LAUNCH();
    if (nc > 1) {
        const size_t m = (size_t)nc * top_k;
        const size_t smem2 = sizeof(Smem) + (m + 31) / 32 * 4 + 16;
        topk_merge_kernel<<<n_q, kThreads, smem2, st>>>(p);
        SFA_CHECK_LAUNCH();
    }
    return SFA_OK;
}
