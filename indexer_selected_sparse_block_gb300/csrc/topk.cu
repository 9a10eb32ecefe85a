// topk.cu -- the budget rule: the indexer_top_k best blocks of each query (sfa_topk_blocks).
//
// The budget holds the indexer_top_k best blocks; the tail that does not fill a block is
// attended anyway, and a query that sees no more blocks than the budget keeps them all
// (llama.cpp commit "model: add Qwen3.8-Flash-Next (qwen4exp)", QSA paragraphs).
// Order: score descending, then block index ascending (the tie rule of this library).  The
// kept ids are written ascending and the row is padded with -1 (the sparse index rows of
// llama.cpp PR #27970 "CUDA + ggml: add sparse-fa for DSV4/GLM" are padded the same way).
//
// Exact and deterministic without sorting.  A 1024-thread CTA takes a piece of at most 36864
// elements and holds it in registers, R consecutive elements per thread, read with 16-byte
// loads; each score becomes its order-preserving 32-bit key.  The k-th largest of the 1024
// per-thread maxima is at most the k-th largest key T (the maxima are a subset), so the floor
// of its 12-bit histogram bin bounds T from below: only the keys at or above it (k and a few
// per cent more on score rows) are compacted, in index order, into shared memory, where a
// radix select (bits 31..20, 19..8, 7..0) finds T and the keys equal to T are ranked lower
// index first.  Kept candidates set their bit in their owner thread's mask; a scan of the
// per-thread kept counts gives each thread its output offset, so the kept ids come out
// ascending with no sort.  Pieces with too many candidates, or many equal keys at the cut,
// run the same digits over the registers and rank the equal keys by a block-wide scan.
// A row longer than one piece is cut into chunks: each chunk keeps its own top k as (score
// bits, id) candidates in chunk order (the global top k lies in their union, the order being
// total), and the next level selects among them the same way, until one piece holds the row.
#include "sfa_common.cuh"

namespace sfa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kPerSm = 1;                 // resident CTAs per SM
constexpr int kBins = 4096;               // 12-bit digits
constexpr int kMaxR = 36;                 // elements per thread
constexpr int kChunk = kMaxR * kThreads;  // 36864: the largest piece
constexpr int kMaxCand = 4096;            // candidates resolved from a compacted list
constexpr int kMaxEqRank = 256;           // keys equal to T that are ranked pairwise
constexpr int kMaxLevels = 8;

// Order-preserving image of a score: larger score -> larger key; -0 == +0; NaN lowest.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// A float bit pattern whose order_key is `key` (candidates are passed on in this form, so that
// every level reads score bits): NaN keys map to a NaN pattern, +0 stands for both zeros.
__device__ __forceinline__ uint32_t key_bits(uint32_t key) {
    return (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
}

struct __align__(16) Smem {
    int hist[kBins];
    uint32_t cand_key[kMaxCand];   // the candidate keys, in index order
    int cand_idx[kMaxCand];
    unsigned long long kept[kThreads];   // candidates kept, one bit per element of a thread
    int wsum[kWarps + 1];
    int cut_bin, cut_above, cut_cnt;
};

// Exclusive scan of one value per thread (thread order); *total gets the sum.
__device__ __forceinline__ int block_scan_excl(int v, Smem &sh, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    __syncthreads();   // earlier readers of wsum are done
    if (lane == 31) sh.wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int t = lane < kWarps ? sh.wsum[lane] : 0;
        int ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, ti, o);
            if (lane >= o) ti += y;
        }
        if (lane < kWarps) sh.wsum[lane] = ti - t;
        if (lane == 31) sh.wsum[kWarps] = ti;
    }
    __syncthreads();
    *total = sh.wsum[kWarps];
    return sh.wsum[warp] + incl - v;
}

// The bin of hist[0..nbins) (ordered by key) holding the rem-th largest counted element,
// with the count above it and its own count, into sh.cut_*.  nbins is 4096 or 256.
__device__ __forceinline__ void find_cut(Smem &sh, int nbins, int rem) {
    const int tid = threadIdx.x;
    const int bpt = nbins >= kThreads ? nbins / kThreads : 1;
    const int top = nbins - 1 - bpt * tid;   // this thread's bins: top, top - 1, ...
    int local = 0;
    if (top >= 0)
        for (int e = 0; e < bpt; ++e) local += sh.hist[top - e];
    int total;
    const int excl = block_scan_excl(local, sh, &total);
    if (top >= 0 && excl < rem && rem <= excl + local) {
        int cum = excl;
        for (int e = 0; e < bpt; ++e) {
            const int h = sh.hist[top - e];
            if (cum + h >= rem) {
                sh.cut_bin = top - e;
                sh.cut_above = cum;
                sh.cut_cnt = h;
                break;
            }
            cum += h;
        }
    }
    __syncthreads();
}

__device__ __forceinline__ void clear_hist(Smem &sh, int nbins) {
    for (int b = threadIdx.x; b < nbins; b += kThreads) sh.hist[b] = 0;
    __syncthreads();
}

struct TopkParams {
    const float *scores;            // level 0 input
    const int32_t *q_pos;
    int32_t *blk_idx, *n_sel;
    const uint32_t *in_bits;        // level >= 1 input: the previous level's candidates
    const int32_t *in_id;
    uint32_t *out_bits;             // chunk stage output: the next level's candidates
    int32_t *out_id;
    int32_t *status;
    int64_t score_stride, n_blk_max;
    int64_t in_stride, out_stride;  // candidate slots per row of the input / output levels
    int cr, top_k, level, final_stage;
};

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

// Elements of a row at the next level after a chunk stage: every chunk but the last passes
// k candidates (a chunk holds more than k), the last min(k, its length).
__host__ __device__ __forceinline__ int64_t next_len(int64_t n, int k) {
    if (n <= 0) return 0;
    const int64_t nc = (n + kChunk - 1) / kChunk;
    const int64_t last = n - (nc - 1) * kChunk;
    return (nc - 1) * k + (last < k ? last : k);
}

// One stage over (row, chunk) items, persistent over the grid; R elements per thread.
template <int R>
__global__ void __launch_bounds__(kThreads, kPerSm) topk_stage_kernel(const TopkParams p, int n_q,
                                                                      int n_chunks) {
    static_assert(R % 4 == 0 && R <= 64, "16-byte loads, one kept bit per element");
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Smem &sh = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x;
    const int k = p.top_k;
    const int n_items = n_q * n_chunks;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int i = item / n_chunks, c = item % n_chunks;
        int64_t len = visible_blocks(p.q_pos, i, p.cr, p.n_blk_max,
                                     (p.level == 0 && c == 0 && tid == 0) ? p.status : nullptr);
        for (int l = 0; l < p.level; ++l) len = next_len(len, k);   // this row at this level
        const int64_t b0 = (int64_t)c * kChunk;
        const int n = (int)(p.final_stage ? len : (len - b0 < kChunk ? len - b0 : kChunk));
        const uint32_t *src = p.level == 0
                                  ? reinterpret_cast<const uint32_t *>(p.scores + (int64_t)i * p.score_stride)
                                  : p.in_bits + (int64_t)i * p.in_stride;   // score bits either way
        const int32_t *in_id = p.level ? p.in_id + (int64_t)i * p.in_stride : nullptr;
        src += b0;
        if (n <= k) {
            if (p.final_stage) {   // every element fits the budget: all of them, in order
                int32_t *out = p.blk_idx + (int64_t)i * k;
                for (int j = tid; j < k; j += kThreads)
                    out[j] = j < n ? (p.level == 0 ? j : in_id[j]) : -1;
                if (tid == 0) p.n_sel[i] = n > 0 ? n : 0;
            } else if (n > 0) {    // a short last chunk passes everything on
                uint32_t *ob = p.out_bits + (int64_t)i * p.out_stride + (int64_t)c * k;
                int32_t *oi = p.out_id + (int64_t)i * p.out_stride + (int64_t)c * k;
                for (int j = tid; j < n; j += kThreads) {
                    ob[j] = src[j];
                    oi[j] = p.level == 0 ? (int)(b0 + j) : in_id[b0 + j];
                }
            }
            continue;
        }
        // ---- this thread's R consecutive elements, as keys (0 past the piece: never kept)
        const int e0 = tid * R;
        const int nv = n - e0 < 0 ? 0 : (n - e0 < R ? n - e0 : R);
        uint32_t key[R];
        const uint32_t *mine = src + e0;
        if (nv == R && (reinterpret_cast<uintptr_t>(mine) & 15u) == 0) {
#pragma unroll
            for (int m = 0; m < R / 4; ++m) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(mine) + m);
                key[4 * m] = order_key(__uint_as_float(v.x));
                key[4 * m + 1] = order_key(__uint_as_float(v.y));
                key[4 * m + 2] = order_key(__uint_as_float(v.z));
                key[4 * m + 3] = order_key(__uint_as_float(v.w));
            }
        } else {
#pragma unroll
            for (int j = 0; j < R; ++j) key[j] = j < nv ? order_key(__uint_as_float(__ldg(mine + j))) : 0u;
        }
        // ---- a lower bound of T: the floor of the cut bin of the k-th largest per-thread
        // maximum (the maxima are a subset of the keys, so their k-th largest is <= T)
        uint32_t lo = 0;
        if (k <= (n + R - 1) / R) {   // at least k threads hold elements, so k maxima exist
            uint32_t mx = 0;
#pragma unroll
            for (int j = 0; j < R; ++j) mx = key[j] > mx ? key[j] : mx;   // 0 past the piece
            clear_hist(sh, kBins);
            if (nv > 0) atomicAdd(&sh.hist[mx >> 20], 1);
            __syncthreads();
            find_cut(sh, kBins, k);
            lo = (uint32_t)sh.cut_bin << 20;
        }
        // ---- candidates: the keys >= lo (at least k), compacted in index order
        uint64_t candm = 0;
        {
            const uint64_t valid = nv ? ~0ull >> (64 - nv) : 0ull;
#pragma unroll
            for (int j = 0; j < R; ++j) candm |= (uint64_t)(key[j] >= lo) << j;
            candm &= valid;
        }
        int nc;
        int cpos = block_scan_excl(__popcll(candm), sh, &nc);
        uint64_t keep = 0;
        bool fallback = nc > kMaxCand;
        if (!fallback) {
            sh.kept[tid] = 0ull;
            for (uint64_t m = candm; m; m &= m - 1) {
                const int j = __ffsll((long long)m) - 1;
                uint32_t kj = 0;
#pragma unroll
                for (int jj = 0; jj < R; ++jj) kj = jj == j ? key[jj] : kj;   // register pick
                sh.cand_key[cpos] = kj;
                sh.cand_idx[cpos] = e0 + j;
                ++cpos;
            }
            // ---- exact radix select over the candidates: T and the keys equal to it to take
            __syncthreads();
            clear_hist(sh, kBins);
            for (int q = tid; q < nc; q += kThreads) atomicAdd(&sh.hist[sh.cand_key[q] >> 20], 1);
            __syncthreads();
            find_cut(sh, kBins, k);
            const uint32_t binA = (uint32_t)sh.cut_bin;
            int rem = k - sh.cut_above;
            uint32_t T = binA << 20;      // keys >= T are kept (all unless take_eq < cnt_eq)
            int take_eq = 0, cnt_eq = 0;  // keys == T to keep (lowest ids first) / present
            if (sh.cut_cnt != rem) {
                __syncthreads();
                clear_hist(sh, kBins);
                for (int q = tid; q < nc; q += kThreads)
                    if ((sh.cand_key[q] >> 20) == binA) atomicAdd(&sh.hist[(sh.cand_key[q] >> 8) & 0xFFFu], 1);
                __syncthreads();
                find_cut(sh, kBins, rem);
                const uint32_t pre24 = (binA << 12) | (uint32_t)sh.cut_bin;
                rem -= sh.cut_above;
                T = pre24 << 8;
                if (sh.cut_cnt != rem) {
                    __syncthreads();
                    clear_hist(sh, 256);
                    for (int q = tid; q < nc; q += kThreads)
                        if ((sh.cand_key[q] >> 8) == pre24) atomicAdd(&sh.hist[sh.cand_key[q] & 0xFFu], 1);
                    __syncthreads();
                    find_cut(sh, 256, rem);
                    T = (pre24 << 8) | (uint32_t)sh.cut_bin;
                    take_eq = rem - sh.cut_above;
                    cnt_eq = sh.cut_cnt;
                }
            }
            const bool rank_eq = take_eq < cnt_eq;
            if (rank_eq && cnt_eq > kMaxEqRank) {
                fallback = true;   // many equal keys at the cut: ranked by a block scan below
            } else {
                for (int q = tid; q < nc; q += kThreads) {
                    const uint32_t kq = sh.cand_key[q];
                    bool kp = kq >= T;
                    if (kq == T && rank_eq) {   // lower index (= list position) first
                        int r = 0;
                        for (int u = 0; u < q; ++u) r += sh.cand_key[u] == T;
                        kp = r < take_eq;
                    }
                    if (kp) {
                        const int iq = sh.cand_idx[q];
                        atomicOr(&sh.kept[iq / R], 1ull << (iq % R));
                    }
                }
                __syncthreads();
                keep = sh.kept[tid];
            }
        }
        if (fallback) {
            // ---- general path: the three digits and the ranking over the registers
            keep = 0;
            __syncthreads();
            clear_hist(sh, kBins);
#pragma unroll
            for (int j = 0; j < R; ++j)
                if (j < nv) atomicAdd(&sh.hist[key[j] >> 20], 1);
            __syncthreads();
            find_cut(sh, kBins, k);
            const uint32_t binA = (uint32_t)sh.cut_bin;
            int rem = k - sh.cut_above;
            uint32_t T = binA << 20;
            int take_eq = 0, cnt_eq = 0;
            if (sh.cut_cnt != rem) {
                __syncthreads();
                clear_hist(sh, kBins);
#pragma unroll
                for (int j = 0; j < R; ++j)
                    if (j < nv && (key[j] >> 20) == binA) atomicAdd(&sh.hist[(key[j] >> 8) & 0xFFFu], 1);
                __syncthreads();
                find_cut(sh, kBins, rem);
                const uint32_t pre24 = (binA << 12) | (uint32_t)sh.cut_bin;
                rem -= sh.cut_above;
                T = pre24 << 8;
                if (sh.cut_cnt != rem) {
                    __syncthreads();
                    clear_hist(sh, 256);
#pragma unroll
                    for (int j = 0; j < R; ++j)
                        if (j < nv && (key[j] >> 8) == pre24) atomicAdd(&sh.hist[key[j] & 0xFFu], 1);
                    __syncthreads();
                    find_cut(sh, 256, rem);
                    T = (pre24 << 8) | (uint32_t)sh.cut_bin;
                    take_eq = rem - sh.cut_above;
                    cnt_eq = sh.cut_cnt;
                }
            }
            const bool rank_eq = take_eq < cnt_eq;
            int eq_rank = 0, tot_eq;
            if (rank_eq) {   // rank of this thread's keys equal to T among all of them
                int c_eq = 0;
#pragma unroll
                for (int j = 0; j < R; ++j) c_eq += (j < nv && key[j] == T) ? 1 : 0;
                eq_rank = block_scan_excl(c_eq, sh, &tot_eq);
            }
#pragma unroll
            for (int j = 0; j < R; ++j) {
                bool kp = false;
                if (j < nv) {
                    if (key[j] > T) {
                        kp = true;
                    } else if (key[j] == T) {
                        kp = !rank_eq || eq_rank < take_eq;
                        ++eq_rank;
                    }
                }
                if (kp) keep |= 1ull << j;
            }
        }
        // ---- output offsets, ascending write-out
        int tot;
        int pos = block_scan_excl(__popcll(keep), sh, &tot);
        if (p.final_stage) {
            int32_t *out = p.blk_idx + (int64_t)i * k;
            for (uint64_t m = keep; m; m &= m - 1) {
                const int j = __ffsll((long long)m) - 1;
                out[pos++] = p.level == 0 ? e0 + j : in_id[e0 + j];
            }
            if (tid == 0) p.n_sel[i] = k;
        } else {
            uint32_t *ob = p.out_bits + (int64_t)i * p.out_stride + (int64_t)c * k;
            int32_t *oi = p.out_id + (int64_t)i * p.out_stride + (int64_t)c * k;
            for (uint64_t m = keep; m; m &= m - 1) {
                const int j = __ffsll((long long)m) - 1;
                uint32_t kj = 0;
#pragma unroll
                for (int jj = 0; jj < R; ++jj) kj = jj == j ? key[jj] : kj;   // register pick
                ob[pos] = key_bits(kj);
                oi[pos] = p.level == 0 ? (int)(b0 + e0 + j) : in_id[b0 + e0 + j];
                ++pos;
            }
        }
        __syncthreads();   // shared memory is reused by the next item
    }
}

// The levels for rows of up to n_blk_max scores: lengths per row at each level (n[0] =
// n_blk_max); the last level is the final select (one piece per row).
struct Plan {
    int levels = 0;   // chunk levels before the final stage; -1: unsupported
    int64_t n[kMaxLevels + 1] = {};
};

Plan make_plan(int64_t n_blk_max, int top_k) {
    Plan pl;
    pl.n[0] = n_blk_max;
    while (pl.n[pl.levels] > kChunk) {
        if (pl.levels == kMaxLevels) {
            pl.levels = -1;
            return pl;
        }
        pl.n[pl.levels + 1] = next_len(pl.n[pl.levels], top_k);
        ++pl.levels;
    }
    return pl;
}

template <int R>
int launch_stage(const TopkParams &p, int n_q, int n_chunks, cudaStream_t st) {
    const int64_t items = (int64_t)n_q * n_chunks;
    if (items > 0x7FFFFFFF) return SFA_ERR_UNSUPPORTED;
    int grid = kPerSm * device_sm_count();
    if (grid < 1) return SFA_ERR_CUDA;
    if (items < grid) grid = (int)items;
    static bool attr = false;   // the shared memory is above the default 48 KB
    if (!attr) {
        if (!allow_max_dynamic_smem(topk_stage_kernel<R>)) return SFA_ERR_CUDA;
        attr = true;
    }
    topk_stage_kernel<R><<<grid, kThreads, sizeof(Smem), st>>>(p, n_q, n_chunks);
    SFA_CHECK_LAUNCH();
    return SFA_OK;
}

// The stage instance that holds n elements per CTA.
int run_stage(const TopkParams &p, int n_q, int n_chunks, int64_t n, cudaStream_t st) {
    if (n <= 8 * kThreads) return launch_stage<8>(p, n_q, n_chunks, st);
    if (n <= 16 * kThreads) return launch_stage<16>(p, n_q, n_chunks, st);
    return launch_stage<kMaxR>(p, n_q, n_chunks, st);
}

}  // namespace
}  // namespace sfa

extern "C" size_t sfa_topk_workspace_bytes(int n_q, int64_t n_blk_max, int top_k) {
    using namespace sfa;
    if (n_q <= 0 || top_k <= 0 || top_k > 2048 || n_blk_max <= 0) return 0;
    const Plan pl = make_plan(n_blk_max, top_k);
    if (pl.levels <= 0) return 0;
    // candidate bits and ids of levels 1..levels, per row
    int64_t slots = 0;
    for (int l = 1; l <= pl.levels; ++l) slots += pl.n[l];
    return (size_t)n_q * (size_t)slots * 8 + 256;
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
    if (n_blk_max > ((int64_t)1 << 21)) return SFA_ERR_UNSUPPORTED;
    if (n_q == 0) return SFA_OK;
    const int64_t nb = n_blk_max > 0 ? n_blk_max : 1;
    const Plan pl = make_plan(nb, top_k);
    if (pl.levels < 0) return SFA_ERR_UNSUPPORTED;
    const size_t need = sfa_topk_workspace_bytes(n_q, nb, top_k);
    if (need > 0 && (!workspace || workspace_bytes < need)) return SFA_ERR_WORKSPACE;
    const cudaStream_t st = (cudaStream_t)stream;
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
    // level l >= 1 candidates: bits [n_q][n[l]] then ids [n_q][n[l]], levels back to back
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    uint32_t *bits[kMaxLevels + 1] = {};
    int32_t *ids[kMaxLevels + 1] = {};
    size_t off = 0;
    for (int l = 1; l <= pl.levels; ++l) {
        bits[l] = reinterpret_cast<uint32_t *>(ws + off);
        off += (size_t)n_q * pl.n[l] * 4;
        ids[l] = reinterpret_cast<int32_t *>(ws + off);
        off += (size_t)n_q * pl.n[l] * 4;
    }
    for (int l = 0; l <= pl.levels; ++l) {
        TopkParams q = p;
        q.level = l;
        q.final_stage = l == pl.levels;
        if (l > 0) {
            q.in_bits = bits[l];
            q.in_id = ids[l];
            q.in_stride = pl.n[l];
        }
        if (!q.final_stage) {
            q.out_bits = bits[l + 1];
            q.out_id = ids[l + 1];
            q.out_stride = pl.n[l + 1];
        }
        const int n_chunks = q.final_stage ? 1 : (int)((pl.n[l] + kChunk - 1) / kChunk);
        const int64_t piece = q.final_stage ? pl.n[l] : kChunk;
        const int rc = run_stage(q, n_q, n_chunks, piece, st);
        if (rc != SFA_OK) return rc;
    }
    return SFA_OK;
}
