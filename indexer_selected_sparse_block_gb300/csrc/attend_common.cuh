// attend_common.cuh -- the attended list of a query and the launch parameters shared by the
// attention kernels of libsfa (attend.cu: the warp-level, tcgen05 and fp32 kernels;
// attend_ws.cu: the warp-specialised bulk-copy kernel).
//
// llama.cpp PR #27970 "CUDA + ggml: add sparse-fa for DSV4/GLM" gathers the K/V rows of each
// query through a per-query index list.  Here the list is built on the fly from the kept block
// ids: list position j maps to token
//   j < n_sel*cr : blk[j / cr]*cr + j % cr       (kept blocks, ascending)
//   otherwise     : B*cr + (j - n_sel*cr)          (the tail, always attended)
// and the dense case is the identity j -> j over 0..p.
#pragma once

#include "sfa_common.cuh"

namespace sfa {

constexpr int kT = 32;          // tokens per tile
constexpr int kThreads = 128;   // 4 warps
constexpr int kMaxBlkList = 2056;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
    const void *Q, *K, *V;
    const int32_t *q_seq, *q_pos, *blk_idx, *n_sel;
    float *O, *lse, *part_o, *part_ml;
    int32_t *status;
    int64_t k_tok_stride, k_seq_stride, v_tok_stride, v_seq_stride, n_tok_cap;
    const int32_t *cell_of;   // paged layout: [n_seq][n_tok_cap] cell of each position, or null
    int64_t n_cells;          // rows of the paged K (and V) arrays
    int n_seq, n_q, h_q, h_kv, G, top_k, cr, dense, n_split, split_tokens, stages;
    int cluster_merge;   // 1: the n_split CTAs of an item form one cluster and merge in place
    int n_items;         // n_q * h_kv * n_split work items (query, KV head, split)
    int64_t n_kv_max;    // the caller's bound on every list's length
    int64_t window;      // > 0: the window positions p - window + 1 .. p are attended too
    int part;            // SFA_PART_*: the whole list, its kept part, or its window part
    int tail_fold;       // 1: the splits cover the kept tokens and the last one also the tail
                         // (the warp-level bf16 kernel, V = K, in-cluster merge, no window)
    float scale_log2;
};

// Row of position tok of sequence seq in the K (and V) arrays, in units of k_tok_stride
// (v_tok_stride) from the sequence's base: the position itself in the per-sequence layout, the
// cell the map gives in the paged one (where the sequence bases are all zero).  Padding
// (tok < 0) and a cell outside [0, n_cells) give -1: the position is left out of the softmax,
// and a bad cell raises SFA_DEV_BAD_CELL.
__device__ __forceinline__ int64_t checked_cell(const AttnParams &p, int32_t c) {
    if (c < 0 || (int64_t)c >= p.n_cells) {
        set_status(p.status, SFA_DEV_BAD_CELL);
        return -1;
    }
    return c;
}
__device__ __forceinline__ int64_t kv_row(const AttnParams &p, int seq, int tok) {
    if (tok < 0 || !p.cell_of) return tok;
    return checked_cell(p, __ldg(p.cell_of + (int64_t)seq * p.n_tok_cap + tok));
}

// Per-CTA view of the attended list of one query.
struct ListInfo {
    int ok;        // 0: the query is outside the caches (skipped)
    int seq, pos;
    int len;       // list length
    int n_blk_tok; // n_sel * cr: positions [0, n_blk_tok) come from kept blocks
    int tail0;     // first token of the suffix attended in full: the tail (B * cr), or the
                   // window's first position when a window reaches further back; kept
                   // tokens from here on are left out of the kept part (padding)
};

__device__ __forceinline__ ListInfo list_info(const AttnParams &p, int i, bool flag) {
    ListInfo L{};
    L.seq = p.q_seq[i];
    L.pos = p.q_pos[i];
    L.ok = L.seq >= 0 && L.seq < p.n_seq && L.pos >= 0 && (int64_t)L.pos < p.n_tok_cap;
    if (!L.ok) {
        if (flag) set_status(p.status, SFA_DEV_BAD_QUERY);
        return L;
    }
    if (p.dense) {
        L.len = L.pos + 1;
        L.n_blk_tok = 0;
        L.tail0 = 0;
        // a dense query longer than the bound the call was planned with: its keys past the
        // bound are not attended, and the query is flagged
        if (L.len > p.n_kv_max) {
            if (flag) set_status(p.status, SFA_DEV_BAD_QUERY);
            L.len = (int)p.n_kv_max;
        }
        return L;
    }
    const int B = (L.pos + 1) / p.cr;
    int ns = p.n_sel[i];
    const int ns_max = min(p.top_k, B);
    if (ns < 0 || ns > ns_max) {
        if (flag) set_status(p.status, SFA_DEV_BAD_NSEL);
        ns = ns < 0 ? 0 : ns_max;
    }
    // the suffix attended in full: the tail, or the window when it starts earlier
    int64_t s0 = (int64_t)B * p.cr;
    if (p.window > 0) {
        const int64_t w0 = (int64_t)L.pos - p.window + 1;
        s0 = min(s0, w0 < 0 ? (int64_t)0 : w0);
    }
    L.tail0 = (int)s0;
    L.n_blk_tok = p.part == SFA_PART_WINDOW ? 0 : ns * p.cr;
    L.len = L.n_blk_tok + (p.part == SFA_PART_SELECTED ? 0 : L.pos + 1 - L.tail0);
    return L;
}

// Loads the validated block ids that list positions [j0, j1) need into s_blk (from jb0), the
// threads first, first + stride, ... sharing the entries.
__device__ __forceinline__ int load_block_list(const AttnParams &p, int i, const ListInfo &L,
                                               int j0, int j1, int *s_blk, bool flag,
                                               int first, int stride) {
    if (p.dense || L.n_blk_tok == 0 || j0 >= L.n_blk_tok) return 0;
    const int jb0 = j0 / p.cr;
    const int jb1 = (min(j1, L.n_blk_tok) + p.cr - 1) / p.cr;
    const int B = (L.pos + 1) / p.cr;
    const int32_t *row = p.blk_idx + (int64_t)i * p.top_k;
    for (int jb = jb0 + first; jb < jb1; jb += stride) {
        const int b = row[jb];
        const bool ok = b >= 0 && b < B && (jb == 0 || b > row[jb - 1]);
        if (!ok && flag) set_status(p.status, SFA_DEV_BAD_BLOCK);
        s_blk[jb - jb0] = ok ? b : -1;
    }
    return jb0;
}
__device__ __forceinline__ int load_block_list(const AttnParams &p, int i, const ListInfo &L,
                                               int j0, int j1, int *s_blk, bool flag) {
    return load_block_list(p, i, L, j0, j1, s_blk, flag, threadIdx.x, blockDim.x);
}

__device__ __forceinline__ int token_at(const AttnParams &p, const ListInfo &L, int j, int j1,
                                        const int *s_blk, int jb0) {
    if (j >= j1) return -1;
    if (p.dense) return j;
    if (j < L.n_blk_tok) {
        const int jb = j / p.cr;
        const int b = s_blk[jb - jb0];
        const int t = b * p.cr + (j - jb * p.cr);
        return b < 0 || t >= L.tail0 ? -1 : t;   // kept tokens inside the suffix: padding
    }
    return L.tail0 + (j - L.n_blk_tok);
}

// ---- the warp-specialised bulk-copy kernel (attend_ws.cu)
// Launch plan of one attention call on that kernel: the list of each (query, KV head) is cut
// into n_split pieces of split_tokens positions; grid CTAs (one per SM at most) take the
// n_q * h_kv * n_split work items; cluster > 1: the n_split CTAs of an item form one cluster and
// merge in place; otherwise, with n_split > 1, combine_kernel merges the partials.
struct WsPlan {
    int n_split, split_tokens, cluster, grid;
};
// false: the warp-specialised kernel has no instantiation for this shape (or it does not fit).
bool ws_make_plan(int n_q, int h_kv, int dkq, int dv, bool has_v, int64_t n_kv_max, int cr,
                  int dense, WsPlan *out);
int ws_launch(const AttnParams &p, const WsPlan &plan, int dkq, int dv, bool has_v,
              cudaStream_t st);
// The gather alone (the K/V rows of every attended list into shared memory, no arithmetic):
// the data-movement ceiling of the attention on the same lists (attend_ws.cu).
int ws_gather_launch(const AttnParams &p, const WsPlan &plan, int dkq, int dv, bool has_v,
                     uint32_t *checksum, cudaStream_t st);

}  // namespace sfa
