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
// elements: coalesced 16-byte loads stage it in shared memory (each element loaded by exactly
// one thread, which keeps the maximum of what it loaded), and each thread then reads R
// consecutive elements back as order-preserving 32-bit keys.  The k-th largest of the 1024
// per-thread maxima is at most the k-th largest key T (the maxima are keys of distinct
// elements), so the floor of its histogram bin bounds T from below; the bins are 12-bit
// windows sized to the range the maxima span, so the bound is tight (while a piece is
// selected, the CTA's next piece is prefetched into L2).  Only the keys at or above it (k and
// a few per cent more on score rows) are compacted, in index order, into shared memory, where a
// radix select whose 12-bit digit windows are again sized to the candidates' range finds T
// (one pass for most rows, at most three).  A single block scan over the candidate list, of
// the counts above T and equal to T packed in one word, then gives every kept candidate its
// output slot, the keys equal to T ranked lower index first, so the kept ids come out
// ascending with no sort.  Pieces with too many candidates (many equal keys, or a budget above
// the thread count) run fixed 12/12/8-bit digits over the registers and rank the keys equal
// to T by a block-wide scan.
// A row longer than one piece is cut into chunks: each chunk keeps its own top k as (score
// bits, id) candidates in chunk order (the global top k lies in their union, the order being
// total), and the next level selects among them the same way, until one piece holds the row.
#include <cooperative_groups.h>

#include "sfa_common.cuh"

namespace sfa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kPerSm = 1;                 // resident CTAs per SM
constexpr int kBins = 4096;               // 12-bit digits
constexpr int kMaxR = 36;                 // elements per thread
constexpr int kChunk = kMaxR * kThreads;  // 36864: the largest piece
constexpr int kMaxCand = 4 * kThreads;    // candidates resolved from a compacted list
constexpr int kMaxLevels = 8;
constexpr int kAllEq = 0x7FFFFFFF;        // Cut::take_eq: every key equal to T is kept
static_assert(kWarps == 32, "one warp reduces the per-warp values");

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
    int cand_idx[kMaxCand];        // their element index within the piece
    int wsum[kWarps + 1];
    uint32_t wred[3][kWarps];      // per-warp extrema
    int cut_bin, cut_above, cut_cnt;
    uint32_t kmin;
};
// The piece is staged right after Smem: R * kThreads words, 16-byte aligned (so is Smem's size).
template <int R>
constexpr size_t smem_bytes() {
    return sizeof(Smem) + (size_t)R * kThreads * 4;
}
__device__ __forceinline__ uint32_t *staged(Smem &sh) {
    return reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(&sh) + sizeof(Smem));
}

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

// Words [0, n) of src into dst (shared memory, 16-byte aligned), n <= R * kThreads: coalesced
// 16-byte loads over the aligned body, single words at its two ends.  Each word is loaded by
// exactly one thread; *mxf is the largest (NaN-skipping) of the scores this thread loaded and
// *n_mine their count, so that the per-thread maxima are maxima of disjoint groups.  Returns
// the number of 16-byte vectors (threads below it hold at least four scores).
template <int R>
__device__ __forceinline__ int stage_piece(const uint32_t *src, int n, uint32_t *dst,
                                           float *mxf, int *n_mine) {
    const int tid = threadIdx.x;
    int head = (int)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(src) & 15u)) & 15u) >> 2);
    head = head < n ? head : n;
    const int nvec = (n - head) >> 2;
    const int tail0 = head + 4 * nvec;
    const uint4 *v = reinterpret_cast<const uint4 *>(src + head);
    uint4 x[R / 4];
#pragma unroll
    for (int m = 0; m < R / 4; ++m) {
        const int q = tid + m * kThreads;
        x[m] = q < nvec ? __ldg(v + q) : make_uint4(0u, 0u, 0u, 0u);
    }
    float mx = __uint_as_float(0x7FFFFFFFu);   // NaN: fmaxf returns the other operand
    int cnt = 0;
    if (tid < head) {
        const uint32_t w = __ldg(src + tid);
        dst[tid] = w;
        mx = fmaxf(mx, __uint_as_float(w));
        ++cnt;
    }
    if (tid < n - tail0) {
        const uint32_t w = __ldg(src + tail0 + tid);
        dst[tail0 + tid] = w;
        mx = fmaxf(mx, __uint_as_float(w));
        ++cnt;
    }
#pragma unroll
    for (int m = 0; m < R / 4; ++m) {
        if (tid + m * kThreads < nvec) {
            mx = fmaxf(mx, fmaxf(fmaxf(__uint_as_float(x[m].x), __uint_as_float(x[m].y)),
                                 fmaxf(__uint_as_float(x[m].z), __uint_as_float(x[m].w))));
            cnt += 4;
        }
    }
    *mxf = mx;
    *n_mine = cnt;
    if (head == 0) {
#pragma unroll
        for (int m = 0; m < R / 4; ++m) {
            const int q = tid + m * kThreads;
            if (q < nvec) reinterpret_cast<uint4 *>(dst)[q] = x[m];
        }
    } else {
#pragma unroll
        for (int m = 0; m < R / 4; ++m) {
            const int q = tid + m * kThreads;
            if (q < nvec) {
                uint32_t *d = dst + head + 4 * q;
                d[0] = x[m].x;
                d[1] = x[m].y;
                d[2] = x[m].z;
                d[3] = x[m].w;
            }
        }
    }
    return nvec;
}

// Key of -inf: keys below it are NaN images only (order_key maps every NaN to 0).
constexpr uint32_t kNegInfKey = 0x007FFFFFu;

// This thread's R staged scores from e0 (a NaN past the nv valid ones: no comparison keeps
// it and fmaxf skips it).
template <int R>
__device__ __forceinline__ void load_vals(const uint32_t *stg, int e0, int nv, float (&v)[R]) {
    if (nv >= R) {   // every thread but the last few: no bounds to apply
#pragma unroll
        for (int m = 0; m < R / 4; ++m) {
            const uint4 w = reinterpret_cast<const uint4 *>(stg + e0)[m];
            v[4 * m] = __uint_as_float(w.x);
            v[4 * m + 1] = __uint_as_float(w.y);
            v[4 * m + 2] = __uint_as_float(w.z);
            v[4 * m + 3] = __uint_as_float(w.w);
        }
        return;
    }
    const float past = __uint_as_float(0x7FFFFFFFu);
#pragma unroll
    for (int m = 0; m < R / 4; ++m) {
        const uint4 w = reinterpret_cast<const uint4 *>(stg + e0)[m];
        v[4 * m] = 4 * m < nv ? __uint_as_float(w.x) : past;
        v[4 * m + 1] = 4 * m + 1 < nv ? __uint_as_float(w.y) : past;
        v[4 * m + 2] = 4 * m + 2 < nv ? __uint_as_float(w.z) : past;
        v[4 * m + 3] = 4 * m + 3 < nv ? __uint_as_float(w.w) : past;
    }
}

// Block-wide maximum of a and minima of b and c (one value of each per thread).
__device__ __forceinline__ void block_extrema(uint32_t a, uint32_t b, uint32_t c, Smem &sh,
                                              uint32_t &amax, uint32_t &bmin, uint32_t &cmin) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    a = __reduce_max_sync(0xFFFFFFFFu, a);
    b = __reduce_min_sync(0xFFFFFFFFu, b);
    c = __reduce_min_sync(0xFFFFFFFFu, c);
    if (lane == 0) {
        sh.wred[0][warp] = a;
        sh.wred[1][warp] = b;
        sh.wred[2][warp] = c;
    }
    __syncthreads();
    amax = __reduce_max_sync(0xFFFFFFFFu, sh.wred[0][lane]);
    bmin = __reduce_min_sync(0xFFFFFFFFu, sh.wred[1][lane]);
    cmin = __reduce_min_sync(0xFFFFFFFFu, sh.wred[2][lane]);
}

// The smallest s with (span >> s) < kBins: 12-bit bins over a range of span + 1 keys.
__device__ __forceinline__ int bin_shift(uint32_t span) {
    const int bits = 32 - __clz((int)span);
    return bits > 12 ? bits - 12 : 0;
}

// The cut at the k-th largest key T: the keys above T are kept, and of the keys equal to T the
// first take_eq in index order (kAllEq: all of them).  nc candidates sit in sh.cand_* in index
// order; nc < 0: they were too many, nothing was compacted.
struct Cut {
    uint32_t T;
    int take_eq;
    int nc;
};

// The cut at the k-th largest of the nc keys in sh.cand_key (1 <= k <= nc), all within
// [lo, kmax]: a radix select whose 12-bit digit windows are sized to the range still open,
// from [lo, kmax] down to single keys (at most three passes).  sh.hist is zero on entry and on
// return; the returned nc is left for the caller.
__device__ Cut cut_candidates(Smem &sh, int nc, int k, uint32_t lo, uint32_t kmax) {
    const int tid = threadIdx.x;
    Cut cut;
    cut.nc = nc;
    uint32_t base = lo;
    uint64_t top = (uint64_t)kmax + 1;
    int s = bin_shift(kmax - lo);
    int rem = k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        for (int q = tid; q < nc; q += kThreads) {
            const uint32_t kq = sh.cand_key[q];
            if (kq >= base && (uint64_t)kq < top) atomicAdd(&sh.hist[(kq - base) >> s], 1);
        }
        __syncthreads();
        find_cut(sh, kBins, rem);
        const int bin = sh.cut_bin, above = sh.cut_above, c = sh.cut_cnt;
        clear_hist(sh, kBins);
        rem -= above;
        base += (uint32_t)bin << s;
        if (c == rem || s == 0) {   // the whole cut bin is kept / the cut bin is one key
            cut.T = base;
            cut.take_eq = c == rem ? kAllEq : rem;
            return cut;
        }
        top = (uint64_t)base + ((uint64_t)1 << s);
        s = s > 12 ? s - 12 : 0;
    }
    cut.T = base;   // not reached: s is 0 by the third pass
    cut.take_eq = rem;
    return cut;
}

// The cut over the block's n staged scores (this thread's nv from element e0; 1 <= k < n),
// from the compacted candidates.  mxf / n_mine: the maximum and the count of the scores this
// thread staged (groups that partition the piece); at least `groups` threads hold some.
// sh.hist is zero on entry and on return.
template <int R>
__device__ Cut select_cut(const uint32_t *stg, int e0, int nv, int n, int k, float mxf,
                          int n_mine, int groups, Smem &sh) {
    const bool has = n_mine > 0;
    const uint32_t mx = has ? order_key(mxf) : 0u;   // all-NaN: 0, like their keys
    uint32_t kmax, mxmin, unused;
    block_extrema(mx, has ? mx : 0xFFFFFFFFu, 0xFFFFFFFFu, sh, kmax, mxmin, unused);
    // ---- a lower bound of T: the floor of the bin of the k-th largest group maximum (the
    // maxima are keys of distinct elements, so their k-th largest is <= T), bins sized to their
    // range
    uint32_t lo = 0;
    if (k <= groups) {   // at least k groups hold elements, so k maxima exist
        const int s = bin_shift(kmax - mxmin);
        if (has) atomicAdd(&sh.hist[(mx - mxmin) >> s], 1);
        __syncthreads();
        find_cut(sh, kBins, k);
        lo = mxmin + ((uint32_t)sh.cut_bin << s);
        clear_hist(sh, kBins);
    }
    // ---- candidates: the keys >= lo (at least k), compacted in index order.  Above the key of
    // -inf, lo is a float's key and the test is a float comparison (NaNs fail it, as their key
    // 0 fails key >= lo); below, it runs on keys.
    uint64_t cm = 0;
    float v[R];   // read again: not held across the barriers above
    load_vals<R>(stg, e0, nv, v);
    if (lo >= kNegInfKey) {
        const float lof = __uint_as_float(key_bits(lo));
#pragma unroll
        for (int j = 0; j < R; ++j) cm |= (uint64_t)(v[j] >= lof) << j;
    } else {
#pragma unroll
        for (int j = 0; j < R; ++j) cm |= (uint64_t)(j < nv && order_key(v[j]) >= lo) << j;
    }
    int nc;
    int pos = block_scan_excl(__popcll(cm), sh, &nc);
    Cut cut;
    cut.T = 0;
    cut.take_eq = 0;
    cut.nc = nc <= kMaxCand ? nc : -1;
    if (cut.nc < 0) return cut;
    for (uint64_t m = cm; m; m &= m - 1) {
        const int j = __ffsll((long long)m) - 1;
        sh.cand_key[pos] = order_key(__uint_as_float(stg[e0 + j]));
        sh.cand_idx[pos] = e0 + j;
        ++pos;
    }
    __syncthreads();
    const Cut c = cut_candidates(sh, nc, k, lo, kmax);
    cut.T = c.T;
    cut.take_eq = c.take_eq;
    return cut;
}

// Calls f(slot, key, idx) for every kept candidate, slot = its place among the kept ones in
// index order: one block scan of the counts above T and equal to T (packed in one word; each
// thread takes four consecutive candidates).
template <class F>
__device__ __forceinline__ void for_each_kept(const Cut &cut, Smem &sh, F f) {
    const int q0 = threadIdx.x * 4;
    uint32_t kk[4];
    int ngt = 0, neq = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const bool ok = q0 + u < cut.nc;
        kk[u] = ok ? sh.cand_key[q0 + u] : 0u;
        ngt += (ok && kk[u] > cut.T) ? 1 : 0;
        neq += (ok && kk[u] == cut.T) ? 1 : 0;
    }
    int tot;
    const int ex = block_scan_excl(ngt | (neq << 16), sh, &tot);   // fields stay below 2^13
    int gt = ex & 0xFFFF, eq = ex >> 16;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        if (q0 + u < cut.nc) {
            if (kk[u] > cut.T) {
                f(gt + (eq < cut.take_eq ? eq : cut.take_eq), kk[u], sh.cand_idx[q0 + u]);
                ++gt;
            } else if (kk[u] == cut.T) {
                if (eq < cut.take_eq) f(gt + eq, kk[u], sh.cand_idx[q0 + u]);
                ++eq;
            }
        }
    }
}

// The key of this thread's staged element j (0 past the nv valid ones).
__device__ __forceinline__ uint32_t staged_key(const uint32_t *stg, int e0, int nv, int j) {
    return j < nv ? order_key(__uint_as_float(stg[e0 + j])) : 0u;
}

// The cut over the staged piece when the candidates do not fit: fixed digits (bits 31..20,
// 19..8, 7..0) down to the exact key T; take_eq of the cnt_eq keys equal to T are kept.
// sh.hist is zero on entry and on return.
struct RegCut {
    uint32_t T;
    int take_eq, cnt_eq;
};
template <int R>
__device__ RegCut cut_staged(const uint32_t *stg, int e0, int nv, int k, Smem &sh) {
    uint32_t prefix = 0;
    int rem = k, cnt = 0;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 20 : (pass == 1 ? 8 : 0);
        const int fixed = pass == 1 ? 20 : 8;   // the bits above this digit, fixed by now
        const uint32_t mask = pass == 2 ? 0xFFu : 0xFFFu;
#pragma unroll 4
        for (int j = 0; j < nv; ++j) {
            const uint32_t kj = staged_key(stg, e0, nv, j);
            if (pass == 0 || (kj >> fixed) == (prefix >> fixed))
                atomicAdd(&sh.hist[(kj >> shift) & mask], 1);
        }
        __syncthreads();
        find_cut(sh, (int)mask + 1, rem);
        prefix |= (uint32_t)sh.cut_bin << shift;
        rem -= sh.cut_above;
        cnt = sh.cut_cnt;
        clear_hist(sh, (int)mask + 1);
    }
    return RegCut{prefix, rem, cnt};
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

__device__ __forceinline__ int visible_blocks_at(int pos, int cr, int64_t n_blk_max,
                                                 int32_t *status) {
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
__device__ __forceinline__ int visible_blocks(const int32_t *q_pos, int i, int cr,
                                              int64_t n_blk_max, int32_t *status) {
    return visible_blocks_at(q_pos[i], cr, n_blk_max, status);
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
    uint32_t *stg = staged(sh);
    const int tid = threadIdx.x;
    const int k = p.top_k;
    const int n_items = n_q * n_chunks;
    clear_hist(sh, kBins);   // kept zero between items from here on
    pdl_wait();              // global memory from here on
    // The piece of item `it`: its first word and its length (no status is raised here).
    auto piece_of = [&](int it, const uint32_t *&src, int &n) {
        const int i = it / n_chunks, c = it % n_chunks;
        int64_t len = visible_blocks(p.q_pos, i, p.cr, p.n_blk_max, nullptr);
        for (int l = 0; l < p.level; ++l) len = next_len(len, k);   // this row at this level
        const int64_t b0 = (int64_t)c * kChunk;
        n = (int)(p.final_stage ? len : (len - b0 < kChunk ? len - b0 : kChunk));
        src = (p.level == 0
                   ? reinterpret_cast<const uint32_t *>(p.scores + (int64_t)i * p.score_stride)
                   : p.in_bits + (int64_t)i * p.in_stride) + b0;   // score bits either way
    };
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
        // The CTA's next piece starts towards L2 now, so that its staging reads L2 rather than
        // DRAM (pp2048's top-k: 158 -> 149 us): the piece's 16-byte-aligned interior, 16 KB per
        // bulk prefetch, issued by warp 0.
        if (tid < 32 && item + (int)gridDim.x < n_items) {
            const uint32_t *nsrc;
            int nn;
            piece_of(item + (int)gridDim.x, nsrc, nn);
            if (nn > k) {
                const uintptr_t a0 = (reinterpret_cast<uintptr_t>(nsrc) + 15u) & ~uintptr_t(15);
                const uintptr_t a1 = reinterpret_cast<uintptr_t>(nsrc + nn) & ~uintptr_t(15);
                constexpr uintptr_t kPiece = 16384;
                for (uintptr_t a = a0 + (uintptr_t)tid * kPiece; a < a1; a += 32 * kPiece) {
                    const uintptr_t e = a + kPiece < a1 ? a + kPiece : a1;
                    prefetch_l2_bulk(reinterpret_cast<const void *>(a), (uint32_t)(e - a));
                }
            }
        }
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
        float mxf;
        int n_mine;
        const int nvec = stage_piece<R>(src, n, stg, &mxf, &n_mine);
        __syncthreads();
        const int e0 = tid * R;
        const int nv = n - e0 < 0 ? 0 : (n - e0 < R ? n - e0 : R);
        const int groups = min(kThreads, nvec);   // threads holding a 16-byte vector each
        const Cut cut = select_cut<R>(stg, e0, nv, n, k, mxf, n_mine, groups, sh);
        if (cut.nc >= 0) {
            // ---- ascending write-out from the candidate list
            if (p.final_stage) {
                int32_t *out = p.blk_idx + (int64_t)i * k;
                for_each_kept(cut, sh, [&](int slot, uint32_t, int idx) {
                    if (slot < k) out[slot] = p.level == 0 ? idx : in_id[idx];
                });
            } else {
                uint32_t *ob = p.out_bits + (int64_t)i * p.out_stride + (int64_t)c * k;
                int32_t *oi = p.out_id + (int64_t)i * p.out_stride + (int64_t)c * k;
                for_each_kept(cut, sh, [&](int slot, uint32_t kq, int idx) {
                    if (slot < k) {
                        ob[slot] = key_bits(kq);
                        oi[slot] = p.level == 0 ? (int)(b0 + idx) : in_id[b0 + idx];
                    }
                });
            }
        } else {
            // ---- general path: the three digits over the staged piece, and the ranking of the
            // keys equal to T by a block scan
            const RegCut rc = cut_staged<R>(stg, e0, nv, k, sh);
            const bool rank_eq = rc.take_eq < rc.cnt_eq;
            int eq_rank = 0, tot_eq;
            if (rank_eq) {   // rank of this thread's keys equal to T among all of them
                int c_eq = 0;
                for (int j = 0; j < nv; ++j) c_eq += staged_key(stg, e0, nv, j) == rc.T ? 1 : 0;
                eq_rank = block_scan_excl(c_eq, sh, &tot_eq);
            }
            uint64_t keep = 0;
            for (int j = 0; j < nv; ++j) {
                const uint32_t kj = staged_key(stg, e0, nv, j);
                bool kp = kj > rc.T;
                if (kj == rc.T) {
                    kp = !rank_eq || eq_rank < rc.take_eq;
                    ++eq_rank;
                }
                if (kp) keep |= 1ull << j;
            }
            int tot;
            int pos = block_scan_excl(__popcll(keep), sh, &tot);
            if (p.final_stage) {
                int32_t *out = p.blk_idx + (int64_t)i * k;
                for (uint64_t m = keep; m && pos < k; m &= m - 1) {
                    const int j = __ffsll((long long)m) - 1;
                    out[pos++] = p.level == 0 ? e0 + j : in_id[e0 + j];
                }
            } else {
                uint32_t *ob = p.out_bits + (int64_t)i * p.out_stride + (int64_t)c * k;
                int32_t *oi = p.out_id + (int64_t)i * p.out_stride + (int64_t)c * k;
                for (uint64_t m = keep; m && pos < k; m &= m - 1) {
                    const int j = __ffsll((long long)m) - 1;
                    ob[pos] = key_bits(staged_key(stg, e0, nv, j));
                    oi[pos] = p.level == 0 ? (int)(b0 + e0 + j) : in_id[b0 + e0 + j];
                    ++pos;
                }
            }
        }
        if (tid == 0 && p.final_stage) p.n_sel[i] = k;
        __syncthreads();   // shared memory is reused by the next item
    }
}

namespace cg = cooperative_groups;

// Loads group g of a row (elements 4g .. 4g+3, those below B; NaN past B).
__device__ __forceinline__ float4 load_group(const float *row, int g, int B, bool vec) {
    const float nan = __uint_as_float(0x7FFFFFFFu);
    const int e = 4 * g;
    if (vec && e + 3 < B) return __ldg(reinterpret_cast<const float4 *>(row) + g);
    float4 v;
    v.x = e < B ? __ldg(row + e) : nan;
    v.y = e + 1 < B ? __ldg(row + e + 1) : nan;
    v.z = e + 2 < B ? __ldg(row + e + 2) : nan;
    v.w = e + 3 < B ? __ldg(row + e + 3) : nan;
    return v;
}

// The top k of a list of n > k exact-score bits in global memory whose ids are ascending, by
// fixed digits (bits 31..20, 19..8, 7..0) over the keys and packed scans over chunks of 4096
// for the kept ids in order.  The path for candidate lists too long for shared memory.
// sh.hist is zero on entry and on return.
__device__ void select_global_list(const uint32_t *bits, const int32_t *ids, int n, int k,
                                   int32_t *out, Smem &sh) {
    const int tid = threadIdx.x;
    uint32_t prefix = 0;
    int rem = k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 20 : (pass == 1 ? 8 : 0);
        const int fixed = pass == 1 ? 20 : 8;
        const uint32_t mask = pass == 2 ? 0xFFu : 0xFFFu;
        for (int q = tid; q < n; q += kThreads) {
            const uint32_t kq = order_key(__uint_as_float(bits[q]));
            if (pass == 0 || (kq >> fixed) == (prefix >> fixed))
                atomicAdd(&sh.hist[(kq >> shift) & mask], 1);
        }
        __syncthreads();
        find_cut(sh, (int)mask + 1, rem);
        prefix |= (uint32_t)sh.cut_bin << shift;
        rem -= sh.cut_above;
        clear_hist(sh, (int)mask + 1);
    }
    const uint32_t T = prefix;
    const int take_eq = rem;
    int G = 0, E = 0;   // keys above T / equal to T in the chunks before
#pragma unroll 1
    for (int c0 = 0; c0 < n; c0 += kMaxCand) {
        const int q0 = c0 + 4 * tid;
        uint32_t kk[4];
        int ngt = 0, neq = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const bool ok = q0 + u < n;
            kk[u] = ok ? order_key(__uint_as_float(bits[q0 + u])) : 0u;
            ngt += (ok && kk[u] > T) ? 1 : 0;
            neq += (ok && kk[u] == T) ? 1 : 0;
        }
        int tot;
        const int ex = block_scan_excl(ngt | (neq << 16), sh, &tot);
        int gt = G + (ex & 0xFFFF), eq = E + (ex >> 16);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (q0 + u < n) {
                if (kk[u] > T) {
                    const int slot = gt + (eq < take_eq ? eq : take_eq);
                    if (slot < k) out[slot] = ids[q0 + u];
                    ++gt;
                } else if (kk[u] == T) {
                    if (eq < take_eq && gt + eq < k) out[gt + eq] = ids[q0 + u];
                    ++eq;
                }
            }
        }
        G += tot & 0xFFFF;
        E += tot >> 16;
    }
}

// ---------------------------------------------------------------------------------------
// The bounded selection (sfa_topk_blocks_refine), one cluster per row (4 CTAs, or 8 for rows
// past one selection piece).  With lower and upper bounds lo_b <= s_b <= up_b of the exact
// (hi + lo) score s_b, each CTA takes an equal share of the row's blocks:
//   1. the maxima of groups of four lower bounds (each bounds a distinct block from below) and
//      their histogram in the CTA's own shared memory; X_r is the floor of the bin of the CTA's
//      k_r-th largest group maximum, with quotas k_r proportional to the shares' groups and
//      summing to at least k; L = min_r X_r is a lower bound of the k-th largest score;
//   2. the candidates up_b >= L of the share, in ascending order; every block of the exact
//      top k is one (s_b >= s_(k) >= L), and so is every block tied with s_(k);
//   3. their exact scores from the hi + lo pooled keys (mma.sync, fp32 sums), by the share's
//      own CTA, written as keys with the block ids into the leader's candidate list at the
//      share's offset;
//   4. the leader selects the top k of the list.
// Lists longer than 4096 go through global memory (select_global_list).
// A row's cluster: 4 CTAs for rows of up to one selection piece (36864 blocks), each taking
// 3 rounds of 4 * kThreads elements; 8 CTAs of 4 rounds each for rows of up to 131072 blocks.
constexpr int kCl = 4;
constexpr int kClRoundsShort = (kChunk / kCl + 4 * kThreads - 1) / (4 * kThreads);   // 3
constexpr int kClLong = 8;
constexpr int kClRoundsLong = 4;
constexpr int64_t kRefineMaxLong = (int64_t)kClLong * kClRoundsLong * 4 * kThreads;   // 131072
static_assert(kClRoundsShort * 4 * kThreads >= kChunk / kCl, "a quarter of a piece fits the rounds");
static_assert(4 * kClRoundsLong <= 32, "one candidate bit per element in a 32-bit mask");

struct RefineParams {
    const float *lower, *upper;
    int64_t stride;
    const __nv_bfloat16 *q_idx;   // [n_q][H][D]
    const float *w;               // [n_q][H]
    const int32_t *q_seq, *q_pos;
    const __nv_bfloat16 *kbar;    // [n_seq][blk_cap][2 D]
    int64_t kbar_seq_stride;
    int64_t n_blk_max;
    uint32_t *cand_bits;          // [n_q][n_blk_max] exact-score bits (long lists)
    int32_t *cand_id, *cand_n;    // [n_q][n_blk_max], [n_q] (-1: within the budget)
    int32_t *blk_idx, *n_sel;
    int32_t *status;
    int n_seq, cr, H, D, top_k;
};

// The query's index heads as mma.sync B fragments (m16n8k16, bf16): entry ((nt * kPq + pq) * 2
// + h) * 32 + lane holds the pair of registers for heads 8 nt .. 8 nt + 7 and the k-step (pair
// pq, half h) of the column order the A loads use (see rescore_tile).
constexpr int kPq = 4;   // q dims / 32 (D <= 128)
template <int R, int CL>
struct BoundedSmem {
    Smem sh;                        // the leader's candidate list serves the cluster
    float up[R * 4 * kThreads];     // this share's upper bounds (cp.async)
    uint2 qf[2 * kPq * 2 * 32];
    float w[16];
    int woff[R * kWarps];           // per (round, warp): this CTA's candidates before it
    uint32_t cut_x[CL];             // leader slots, per rank: the share's cut X_r
    int cnt[CL];
};

// Exact scores of ROWS (16, or 8 with rows 8..15 of the MMA zero) candidates on the tensor
// cores: S[16 x heads] = [hi | lo] rows x [q ; q], K = 2D, fp32 accumulation, then
// sum_j w_j ReLU(S_j) per row.  Lane (g, t) loads 16 bytes of rows g and g + 8 at element
// 32 pp + 8 t of each 32-element piece pp of the 2D-wide row: the first four elements are its A
// columns (2t, 2t+1, 2t+8, 2t+9) of k-step (pp, 0), the last four those of (pp, 1).  The B table
// pairs the same columns with q (dims mod D), so each k-step sums over 16 distinct columns and
// the pieces cover all 2D.  With 8 rows every piece of a row is loaded at once (one memory round
// trip); with 16, four pieces at a time.  Returns the score of row g (lanes with t == 0) and of
// row g + 8 through s0, s1.
template <int D, int ROWS, typename BS>
__device__ __forceinline__ void rescore_tile(const __nv_bfloat16 *r0, const __nv_bfloat16 *r1,
                                             const BS &bs, int H, float &s0, float &s1) {
    static_assert(ROWS == 8 || ROWS == 16, "tile rows");
    constexpr int kPieces = 2 * D / 32;   // 8 or 4
    constexpr int kG = ROWS == 8 ? kPieces : (kPieces < 4 ? kPieces : 4);   // pieces in flight
    const int lane = threadIdx.x & 31, t = lane & 3;
    const int nt_n = (H + 7) / 8;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int p0 = 0; p0 < kPieces; p0 += kG) {
        uint4 a0[kG], a1[kG];
#pragma unroll
        for (int u = 0; u < kG; ++u) {
            a0[u] = __ldg(reinterpret_cast<const uint4 *>(r0 + 32 * (p0 + u) + 8 * t));
            if constexpr (ROWS == 16)
                a1[u] = __ldg(reinterpret_cast<const uint4 *>(r1 + 32 * (p0 + u) + 8 * t));
            else
                a1[u] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kG; ++u) {
            const int pq = (p0 + u) % (D / 32);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t a[4] = {h ? a0[u].z : a0[u].x, h ? a1[u].z : a1[u].x,
                                       h ? a0[u].w : a0[u].y, h ? a1[u].w : a1[u].y};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    if (nt < nt_n) {
                        const uint2 b = bs.qf[((nt * kPq + pq) * 2 + h) * 32 + lane];
                        mma_bf16_16816(acc[nt], a, b.x, b.y);
                    }
                }
            }
        }
    }
    float p0s = 0.f, p1s = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int h0 = 8 * nt + 2 * t;
        const float w0 = h0 < H ? bs.w[h0] : 0.f, w1 = h0 + 1 < H ? bs.w[h0 + 1] : 0.f;
        p0s = fmaf(w0, fmaxf(acc[nt][0], 0.f), p0s);
        p0s = fmaf(w1, fmaxf(acc[nt][1], 0.f), p0s);
        p1s = fmaf(w0, fmaxf(acc[nt][2], 0.f), p1s);
        p1s = fmaf(w1, fmaxf(acc[nt][3], 0.f), p1s);
    }
    p0s += __shfl_xor_sync(0xFFFFFFFFu, p0s, 1);
    p0s += __shfl_xor_sync(0xFFFFFFFFu, p0s, 2);
    p1s += __shfl_xor_sync(0xFFFFFFFFu, p1s, 1);
    p1s += __shfl_xor_sync(0xFFFFFFFFu, p1s, 2);
    s0 = p0s;
    s1 = p1s;
}

template <int D, int R, int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(kThreads, 1)
    bounded_select_kernel(const RefineParams p, int n_q) {
    constexpr int kClRounds = R;
    constexpr int kCl = CL;
    using BS = BoundedSmem<R, CL>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    BS &bs = *reinterpret_cast<BS *>(smem_raw);
    Smem &sh = bs.sh;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    BS &lead = *cluster.map_shared_rank(&bs, 0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = p.top_k, H = p.H;
    const int n_cl = gridDim.x / kCl;
    clear_hist(sh, kBins);   // kept zero between rows from here on
    // Every CTA of the cluster is running before any remote access: arrive here, wait just
    // before the first one, so that the first row's loads overlap the barrier.
    cluster_arrive_relaxed();
    bool started = false;
    pdl_wait();              // global memory from here on
    // This CTA's groups of four blocks, [g0, g1): a share of the widest row (n_blk_max), fixed
    // before any row's metadata is read, so that the bound loads of a row do not wait for its
    // position.  Elements at or past the row's own length B are masked after the loads.
    const int nbm = (int)p.n_blk_max;
    const int ngm = (nbm + 3) / 4;
    const int per = (ngm + kCl - 1) / kCl;
    const int g0 = rank * per < ngm ? rank * per : ngm;
    const int g1 = g0 + per < ngm ? g0 + per : ngm;
    for (int i = blockIdx.x / kCl; i < n_q; i += n_cl) {
        // the row's metadata, its query's B-fragment table entry and head weight, and the
        // share's bounds: every load of the row is issued before any of them is used
        const int seq = p.q_seq[i];
        const int pos = p.q_pos[i];
        uint2 qb = make_uint2(0u, 0u);
        if (tid < 2 * kPq * 2 * 32) {   // the B fragment table of this query
            const int ln = tid & 31, h = (tid >> 5) & 1, pq = (tid >> 6) % kPq, nt = tid / (64 * kPq);
            const int n = 8 * nt + (ln >> 2), d0 = 32 * pq + 8 * (ln & 3) + 4 * h;
            if (n < H && d0 < D) {
                const uint32_t *qr = reinterpret_cast<const uint32_t *>(p.q_idx + ((int64_t)i * H + n) * D + d0);
                qb = make_uint2(qr[0], qr[1]);
            }
        }
        const float wv = tid < H ? p.w[(int64_t)i * H + tid] : 0.f;
        const float *lp = p.lower + (int64_t)i * p.stride;
        const float *up = p.upper + (int64_t)i * p.stride;
        // lower bounds into registers, upper bounds into shared memory (cp.async), all within
        // the n_blk_max columns of the row
        float4 lv[kClRounds];
        {
            const bool lvec = (reinterpret_cast<uintptr_t>(lp) & 15u) == 0;
#pragma unroll
            for (int m = 0; m < kClRounds; ++m) {
                const int g = g0 + tid + kThreads * m;
                if (g < g1) lv[m] = load_group(lp, g, nbm, lvec);
            }
            const bool vec = (reinterpret_cast<uintptr_t>(up) & 15u) == 0;
#pragma unroll
            for (int m = 0; m < kClRounds; ++m) {
                const int lg = tid + kThreads * m, g = g0 + lg;
                if (g < g1) {
                    if (vec && 4 * g + 3 < nbm) {
                        cp_async16(smem_u32(&bs.up[4 * lg]), up + 4 * g, 16);
                    } else {
                        const float4 v = load_group(up, g, nbm, false);
                        bs.up[4 * lg] = v.x;
                        bs.up[4 * lg + 1] = v.y;
                        bs.up[4 * lg + 2] = v.z;
                        bs.up[4 * lg + 3] = v.w;
                    }
                }
            }
            cp_async_commit();
        }
        int B = visible_blocks_at(pos, p.cr, p.n_blk_max, (rank == 0 && tid == 0) ? p.status : nullptr);
        if (seq < 0 || seq >= p.n_seq) {
            if (rank == 0 && tid == 0) set_status(p.status, SFA_DEV_BAD_QUERY);
            B = 0;
        }
        if (B <= k) {   // every block fits the budget (the same for the whole cluster)
            if (rank == 0) {
                int32_t *out = p.blk_idx + (int64_t)i * k;
                for (int j = tid; j < k; j += kThreads) out[j] = j < B ? j : -1;
                if (tid == 0) {
                    p.n_sel[i] = B;
                    p.cand_n[i] = -1;
                }
            }
            cp_async_wait<0>();   // no copy of this row lands in a later row's buffer
            continue;
        }
        if (tid < 2 * kPq * 2 * 32) bs.qf[tid] = qb;
        if (tid < H) bs.w[tid] = wv;
        // ---- 1. group maxima of the row's lower bounds -> this CTA's cut X_r -> L
        const int ng = (B + 3) / 4;                       // groups of the row
        const int gv = ng < g1 ? ng : g1;                 // this share's groups in the row: [g0, gv)
        const int n_loc = gv > g0 ? gv - g0 : 0;
        uint32_t gm[kClRounds];
        uint32_t mx = 0, mn = 0xFFFFFFFFu;
#pragma unroll
        for (int m = 0; m < kClRounds; ++m) {
            const int g = g0 + tid + kThreads * m;
            gm[m] = 0;
            if (g < gv) {
                const float nan = __uint_as_float(0x7FFFFFFFu);
                const int e = 4 * g;
                const float a = lv[m].x, b = e + 1 < B ? lv[m].y : nan;
                const float c = e + 2 < B ? lv[m].z : nan, d = e + 3 < B ? lv[m].w : nan;
                gm[m] = order_key(fmaxf(fmaxf(a, b), fmaxf(c, d)));
                mx = gm[m] > mx ? gm[m] : mx;
                mn = gm[m] < mn ? gm[m] : mn;
            }
        }
        // This CTA's quota k_r = ceil(k n_loc / ng) (the quotas sum to at least k) and X_r, the
        // floor of the bin of its k_r-th largest group maximum: at least k_r of its group maxima
        // are >= X_r.  L = min_r X_r then has at least k group maxima >= L in the row, each the
        // lower bound of a distinct block, so the k-th largest score is >= L.  A share with no
        // group of the row takes no part (X_r = the largest key); k > ng: L = the lowest key.
        uint32_t X = 0xFFFFFFFFu;
        if (k > ng) {
            X = 0;
        } else if (n_loc > 0) {
            const int k_r = (int)(((int64_t)k * n_loc + ng - 1) / ng);
            uint32_t bmax, bmin, unused;
            block_extrema(mx, mn, 0xFFFFFFFFu, sh, bmax, bmin, unused);
            const int sft = bin_shift(bmax - bmin);
#pragma unroll
            for (int m = 0; m < kClRounds; ++m)
                if (g0 + tid + kThreads * m < gv) atomicAdd(&sh.hist[(gm[m] - bmin) >> sft], 1);
            __syncthreads();
            find_cut(sh, kBins, k_r);
            X = bmin + ((uint32_t)sh.cut_bin << sft);
            clear_hist(sh, kBins);
        }
        if (!started) {   // the first remote access of this CTA
            cluster_wait();
            started = true;
        }
        if (tid == 0) lead.cut_x[rank] = X;
        cluster.sync();   // (a) every share's X_r is in the leader
        uint32_t lo = 0xFFFFFFFFu;
#pragma unroll
        for (int r = 0; r < kCl; ++r) {
            const uint32_t x = lead.cut_x[r];
            lo = x < lo ? x : lo;
        }
        // ---- 2. candidates up_b >= L (as keys: >= lo); bit 4m + r for element 4g + r
        uint32_t cm = 0;
        cp_async_wait<0>();
        __syncthreads();   // the share's upper bounds have landed
        {
            const bool fcmp = lo >= kNegInfKey;   // lo is a float's key: compare floats
            const float L = __uint_as_float(key_bits(lo));
#pragma unroll
            for (int m = 0; m < kClRounds; ++m) {
                const int lg = tid + kThreads * m, g = g0 + lg;
                if (g < gv) {
                    const float4 v = *reinterpret_cast<const float4 *>(&bs.up[4 * lg]);
                    const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const bool c = 4 * g + r < B && (fcmp ? f[r] >= L : order_key(f[r]) >= lo);
                        cm |= (uint32_t)c << (4 * m + r);
                    }
                }
            }
        }
        // ascending order within the share = (round, warp, lane, r)
        int incl[kClRounds];
#pragma unroll
        for (int m = 0; m < kClRounds; ++m) {
            const int c = __popc((cm >> (4 * m)) & 0xFu);
            int x = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            incl[m] = x - c;
            if (lane == 31) bs.woff[m * kWarps + warp] = x;
        }
        __syncthreads();
        if (warp == 0) {   // scan of the kClRounds * 32 totals: kClRounds per lane
            int loc[kClRounds], sum = 0;
#pragma unroll
            for (int e = 0; e < kClRounds; ++e) {
                loc[e] = bs.woff[lane * kClRounds + e];
                sum += loc[e];
            }
            int x = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            int run = x - sum;
#pragma unroll
            for (int e = 0; e < kClRounds; ++e) {
                bs.woff[lane * kClRounds + e] = run;
                run += loc[e];
            }
            if (lane == 31) lead.cnt[rank] = x;
        }
        cluster.sync();   // (d) every share's count is in the leader
        int off = 0, total = 0;
#pragma unroll
        for (int r = 0; r < kCl; ++r) {
            const int c = lead.cnt[r];
            off += r < rank ? c : 0;
            total += c;
        }
        const int mine = lead.cnt[rank];
        const bool in_smem = total <= kMaxCand;   // the same in every CTA
        int32_t *gid = p.cand_id + (int64_t)i * p.n_blk_max;
        uint32_t *gbits = p.cand_bits + (int64_t)i * p.n_blk_max;
        // this share's list: local shared memory, or the row's global list at its offset
#pragma unroll
        for (int m = 0; m < kClRounds; ++m) {
            int pos = bs.woff[m * kWarps + warp] + incl[m];
            const int g = g0 + tid + kThreads * m;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if ((cm >> (4 * m + r)) & 1u) {
                    if (in_smem)
                        sh.cand_idx[pos] = 4 * g + r;
                    else
                        gid[off + pos] = 4 * g + r;
                    ++pos;
                }
        }
        __syncthreads();
        // ---- 3. exact scores of this share's candidates: a warp takes 8 at a time, every
        // piece of their rows in flight at once.  (Spreading all shares' candidates evenly
        // over the CTAs needs each share's list visible to the others first: one more cluster
        // barrier, which cost more than the balance gained -- decode_32x131072's selection
        // 26.9 -> 28.6 us, the 1M-token decode's 24.5 -> 26.5.)
        {
            constexpr int kTR = 8;
            const int32_t *lid = in_smem ? sh.cand_idx : gid + off;
            const __nv_bfloat16 *kseq = p.kbar + (int64_t)seq * p.kbar_seq_stride;
            const int g = lane >> 2;
            for (int c0 = warp * kTR; c0 < mine; c0 += kWarps * kTR) {
                const int ra = c0 + g;
                int ba = lid[ra < mine ? ra : c0];
                if ((unsigned)ba >= (unsigned)B) {   // never a candidate: flagged, row 0 read
                    if ((lane & 3) == 0) set_status(p.status, SFA_DEV_BAD_BLOCK);
                    ba = 0;
                }
                float sa, unused;
                const __nv_bfloat16 *ka = kseq + (int64_t)ba * 2 * D;
                rescore_tile<D, kTR>(ka, ka, bs, H, sa, unused);
                if ((lane & 3) == 0 && ra < mine) {
                    if (in_smem) {
                        // the leader's own list is this array's head: the id written at a
                        // position of it is the one already there
                        lead.sh.cand_key[off + ra] = order_key(sa);
                        lead.sh.cand_idx[off + ra] = ba;
                    } else {
                        gbits[off + ra] = __float_as_uint(sa);
                    }
                }
            }
        }
        if (!in_smem) __threadfence();   // the global list is complete before the leader reads it
        cluster.sync();   // (e) the list is complete
        // ---- 4. the leader selects the top k of the list
        if (rank == 0) {
            int32_t *out = p.blk_idx + (int64_t)i * k;
            if (in_smem) {
                uint32_t kx = 0, kn = 0xFFFFFFFFu;
                for (int q = tid; q < total; q += kThreads) {
                    const uint32_t kq = sh.cand_key[q];
                    kx = kq > kx ? kq : kx;
                    kn = kq < kn ? kq : kn;
                }
                uint32_t kmax, kmin, unused;
                block_extrema(kx, kn, 0xFFFFFFFFu, sh, kmax, kmin, unused);
                const Cut cut = cut_candidates(sh, total, k, kmin, kmax);
                for_each_kept(cut, sh, [&](int slot, uint32_t, int idx) {
                    if (slot < k) out[slot] = idx;
                });
            } else {
                select_global_list(gbits, gid, total, k, out, sh);
            }
            if (tid == 0) {
                p.n_sel[i] = k;
                p.cand_n[i] = total;
            }
            __syncthreads();
        }
    }
    if (!started) cluster_wait();   // the arrival above is matched before the CTA exits
    // The CTAs of a cluster leave together.  (Letting the other CTAs leave while the leader
    // still selects -- which no remote access needs -- made the whole step slower: the next
    // kernel's CTAs took their SMs early.)
    cluster.sync();
}

template <int D, int R, int CL>
int launch_bounded_d(const RefineParams &p, int n_q, cudaStream_t st) {
    if (!ensure_max_dynamic_smem(bounded_select_kernel<D, R, CL>)) return SFA_ERR_CUDA;
    int clusters = device_sm_count() / CL;
    if (clusters < 1) return SFA_ERR_CUDA;
    if (n_q < clusters) clusters = n_q;
    if (launch_pdl(bounded_select_kernel<D, R, CL>, dim3(clusters * CL), dim3(kThreads),
                   sizeof(BoundedSmem<R, CL>), st, p, n_q) != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

// Rows of up to one selection piece take 4-CTA clusters of 3 rounds per CTA; longer rows (up
// to 131072 blocks) take 8-CTA clusters of 4 rounds, an eighth of the row's upper bounds (64 KB)
// in each CTA's shared memory.
int launch_bounded(const RefineParams &p, int n_q, cudaStream_t st) {
    if (p.n_blk_max <= kChunk)
        return p.D == 64 ? launch_bounded_d<64, kClRoundsShort, kCl>(p, n_q, st)
                         : launch_bounded_d<128, kClRoundsShort, kCl>(p, n_q, st);
    return p.D == 64 ? launch_bounded_d<64, kClRoundsLong, kClLong>(p, n_q, st)
                     : launch_bounded_d<128, kClRoundsLong, kClLong>(p, n_q, st);
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
    if (!ensure_max_dynamic_smem(topk_stage_kernel<R>)) return SFA_ERR_CUDA;
    if (launch_pdl(topk_stage_kernel<R>, dim3(grid), dim3(kThreads), smem_bytes<R>(), st, p, n_q,
                   n_chunks) != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
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

extern "C" size_t sfa_topk_refine_workspace_bytes(int n_q, int64_t n_blk_max) {
    if (n_q <= 0 || n_blk_max <= 0) return 0;
    // candidate score bits and ids [n_q][n_blk_max], counts [n_q]
    return (size_t)n_q * (size_t)n_blk_max * 8 + (size_t)n_q * 4 + 256;
}

extern "C" int sfa_topk_blocks_refine(const float *lower, const float *upper,
                                      int64_t score_stride, const void *q_idx, const float *w,
                                      const int32_t *q_seq, const int32_t *q_pos, int n_q,
                                      int h_idx, int d_idx, const void *Kbar,
                                      int64_t kbar_seq_stride, int n_seq, int compress_ratio,
                                      int top_k, int64_t n_blk_max, int32_t *blk_idx,
                                      int32_t *n_sel, void *workspace, size_t workspace_bytes,
                                      int32_t *dev_status, sfa_stream_t stream) {
    using namespace sfa;
    if (!q_pos || !q_seq || !blk_idx || !n_sel || !q_idx || !w || !Kbar || n_q < 0 ||
        compress_ratio < 1 || n_blk_max < 0 || n_seq < 1)
        return SFA_ERR_INVALID_ARG;
    if (top_k < 1 || top_k > 2048) return SFA_ERR_UNSUPPORTED;
    if (d_idx != 64 && d_idx != 128) return SFA_ERR_UNSUPPORTED;
    if (h_idx < 1 || h_idx > 16) return SFA_ERR_UNSUPPORTED;
    if (n_blk_max > kRefineMaxLong) return SFA_ERR_UNSUPPORTED;   // 8 CTAs x 4 rounds
    if (n_blk_max > 0 && (!lower || !upper || score_stride < n_blk_max))
        return SFA_ERR_INVALID_ARG;
    if (kbar_seq_stride < n_blk_max * 2 * d_idx) return SFA_ERR_INVALID_ARG;
    // 16-byte loads of pooled-key rows, 4-byte loads of index-query pairs
    if (!aligned16(Kbar) || kbar_seq_stride % 8 != 0 || (reinterpret_cast<uintptr_t>(q_idx) & 3u))
        return SFA_ERR_INVALID_ARG;
    if (n_q == 0) return SFA_OK;
    const int64_t nb = n_blk_max > 0 ? n_blk_max : 1;
    const size_t need = sfa_topk_refine_workspace_bytes(n_q, nb);
    if (!workspace || workspace_bytes < need) return SFA_ERR_WORKSPACE;
    const cudaStream_t st = (cudaStream_t)stream;
    uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
    RefineParams r{};
    r.lower = lower;
    r.upper = upper;
    r.stride = score_stride;
    r.q_idx = reinterpret_cast<const __nv_bfloat16 *>(q_idx);
    r.w = w;
    r.q_seq = q_seq;
    r.q_pos = q_pos;
    r.kbar = reinterpret_cast<const __nv_bfloat16 *>(Kbar);
    r.kbar_seq_stride = kbar_seq_stride;
    r.n_blk_max = nb;
    r.cand_bits = reinterpret_cast<uint32_t *>(ws);
    r.cand_id = reinterpret_cast<int32_t *>(ws + (size_t)n_q * nb * 4);
    r.cand_n = reinterpret_cast<int32_t *>(ws + (size_t)n_q * nb * 8);
    r.status = dev_status;
    r.blk_idx = blk_idx;
    r.n_sel = n_sel;
    r.n_seq = n_seq;
    r.cr = compress_ratio;
    r.H = h_idx;
    r.D = d_idx;
    r.top_k = top_k;
    return launch_bounded(r, n_q, st);
}
