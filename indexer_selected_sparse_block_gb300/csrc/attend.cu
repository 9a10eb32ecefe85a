// attend.cu -- gathered flash attention over the kept cells (sfa_gather_attend) and its
// below-budget dense twin (sfa_dense_attend).
//
// llama.cpp PR #27970 "CUDA + ggml: add sparse-fa for DSV4/GLM" gathers the K/V tiles of the
// flash-attention loop through a per-query index list, with V a view of the first 512 dims
// of K for the MLA-shaped heads (576/512) and separate V for 512/512; no ALiBi, no softcap.
// Here the list is built on the fly from the kept block ids: list position j maps to token
//   j < n_sel*cr : blk[j / cr]*cr + j % cr       (kept blocks, ascending)
//   otherwise     : B*cr + (j - n_sel*cr)          (the tail, always attended)
// and the dense case is the identity j -> j over 0..p.
//
// bf16 kernel (one CTA = one query x one KV head x one split of its list, 4 warps):
//   * cp.async 16-byte gathers of 32 selected token rows per stage (each kept block is cr
//     contiguous rows), XOR-swizzled rows so that ldmatrix is conflict-free, 2-4 stages;
//   * S = Q K^T on tensor cores (mma.sync m16n8k16, M = the 16 query heads of the KV head),
//     the head dim split over the 4 warps and the partial sums reduced through shared memory;
//   * online softmax (base 2) over the 32 tokens; P is carried as two bf16 halves
//     (hi = bf16(p), lo = bf16(p - hi)), so P V is accurate to ~2^-17 instead of the 2^-9 of
//     a single bf16 rounding (which alone uses up a 2e-3 output tolerance);
//   * O += P_hi V + P_lo V on tensor cores, the 512 value dims split over the 4 warps; V = K
//     reuses the K tile in shared memory.
// Decode has few queries, so each list is split over several CTAs (flash-decoding) and the
// partial (O, m, l) are merged by combine_kernel.  fp32 inputs take a plain SIMT kernel with
// the same split/merge structure (accuracy reference path).
#include <math.h>

#include <mutex>

#include "sfa_common.cuh"

namespace sfa {
namespace {

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
    int n_seq, n_q, h_q, h_kv, G, top_k, cr, dense, n_split, split_tokens, stages;
    float scale_log2;
};

// Per-CTA view of the attended list of one query.
struct ListInfo {
    int ok;        // 0: the query is outside the caches (skipped)
    int seq, pos;
    int len;       // list length
    int n_blk_tok; // n_sel * cr: positions [0, n_blk_tok) come from kept blocks
    int tail0;     // first tail token (B * cr)
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
        return L;
    }
    const int B = (L.pos + 1) / p.cr;
    int ns = p.n_sel[i];
    const int ns_max = min(p.top_k, B);
    if (ns < 0 || ns > ns_max) {
        if (flag) set_status(p.status, SFA_DEV_BAD_NSEL);
        ns = ns < 0 ? 0 : ns_max;
    }
    L.n_blk_tok = ns * p.cr;
    L.tail0 = B * p.cr;
    L.len = L.n_blk_tok + (L.pos + 1 - L.tail0);
    return L;
}

// Loads the validated block ids that list positions [j0, j1) need into s_blk (from jb0).
__device__ __forceinline__ int load_block_list(const AttnParams &p, int i, const ListInfo &L,
                                               int j0, int j1, int *s_blk, bool flag) {
    if (p.dense || L.n_blk_tok == 0 || j0 >= L.n_blk_tok) return 0;
    const int jb0 = j0 / p.cr;
    const int jb1 = (min(j1, L.n_blk_tok) + p.cr - 1) / p.cr;
    const int B = (L.pos + 1) / p.cr;
    const int32_t *row = p.blk_idx + (int64_t)i * p.top_k;
    for (int jb = jb0 + threadIdx.x; jb < jb1; jb += blockDim.x) {
        const int b = row[jb];
        const bool ok = b >= 0 && b < B && (jb == 0 || b > row[jb - 1]);
        if (!ok && flag) set_status(p.status, SFA_DEV_BAD_BLOCK);
        s_blk[jb - jb0] = ok ? b : -1;
    }
    return jb0;
}

__device__ __forceinline__ int token_at(const AttnParams &p, const ListInfo &L, int j, int j1,
                                        const int *s_blk, int jb0) {
    if (j >= j1) return -1;
    if (p.dense) return j;
    if (j < L.n_blk_tok) {
        const int jb = j / p.cr;
        const int b = s_blk[jb - jb0];
        return b < 0 ? -1 : b * p.cr + (j - jb * p.cr);
    }
    return L.tail0 + (j - L.n_blk_tok);
}

__device__ __forceinline__ uint32_t swz(int c, int r) { return (uint32_t)((c & ~7) | ((c ^ r) & 7)); }

template <int DKQ, int DV, bool V_IS_K>
__global__ void __launch_bounds__(kThreads, 1) attend_bf16_kernel(const AttnParams p) {
    constexpr int KROW = DKQ * 2;                 // bytes of a K row in shared memory
    constexpr int VROW = V_IS_K ? KROW : DV * 2;  // bytes of a V row
    constexpr int KCH = DKQ / 8, VCH = DV / 8;    // 16-byte chunks per row
    constexpr int KS = DKQ / 64;                  // k16 steps of S per warp
    constexpr int NTV = DV / 32;                  // n8 tiles of O per warp
    constexpr int SP_PITCH = kT + 8;              // fp32 S-partial row pitch
    constexpr int P_PITCH = kT + 8;               // bf16 P row pitch
    constexpr int STAGE_BYTES = kT * KROW + (V_IS_K ? 0 : kT * VROW);

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sStage = smem;                                              // stages x STAGE_BYTES
    uint8_t *sQ = sStage + (size_t)p.stages * STAGE_BYTES;               // 16 x KROW
    float *sSP = reinterpret_cast<float *>(sQ + 16 * KROW);              // 4 x 16 x SP_PITCH
    __nv_bfloat16 *sP = reinterpret_cast<__nv_bfloat16 *>(sSP + 4 * 16 * SP_PITCH);  // hi, lo
    float *sAlpha = reinterpret_cast<float *>(sP + 2 * 16 * P_PITCH);    // 16
    float *sL = sAlpha + 16;                                             // 16
    float *sM = sL + 16;                                                 // 16
    int *sTok = reinterpret_cast<int *>(sM + 16);                        // stages x kT
    int *sBlk = sTok + p.stages * kT;                                    // block list

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, g = blockIdx.y, i = blockIdx.z;
    const bool lead = split == 0 && g == 0;
    const ListInfo L = list_info(p, i, lead && tid == 0);
    const int j0 = split * p.split_tokens;
    const int j1 = L.ok ? min(L.len, j0 + p.split_tokens) : 0;
    const int G = p.G;

    if (j0 >= j1) {  // nothing to attend in this split
        for (int e = tid; e < G * DV; e += kThreads) {
            const int row = e / DV, d = e % DV;
            const int h = g * G + row;
            if (p.n_split == 1) {
                p.O[((int64_t)i * p.h_q + h) * DV + d] = 0.f;
                if (d == 0 && p.lse) p.lse[(int64_t)i * p.h_q + h] = -INFINITY;
            } else {
                const int64_t base = (((int64_t)i * p.h_kv + g) * p.n_split + split) * G + row;
                p.part_o[base * DV + d] = 0.f;
                if (d == 0) {
                    p.part_ml[base * 2] = -INFINITY;
                    p.part_ml[base * 2 + 1] = 0.f;
                }
            }
        }
        return;
    }
    // Q rows of this KV head (rows >= G zero-filled), swizzled like the K tile: copied
    // asynchronously as the oldest cp.async group, so the copy overlaps the block-list reads
    // and the first K/V tiles.
    {
        const __nv_bfloat16 *Qg = reinterpret_cast<const __nv_bfloat16 *>(p.Q) +
                                  ((int64_t)i * p.h_q + (int64_t)g * G) * DKQ;
        const uint32_t qs = smem_u32(sQ);
        for (int e = tid; e < 16 * KCH; e += kThreads) {
            const int r = e / KCH, c = e % KCH;
            const bool live = r < G;
            cp_async16(qs + r * KROW + swz(c, r) * 16, live ? Qg + (int64_t)r * DKQ + c * 8 : Qg,
                       live ? 16u : 0u);
        }
        cp_async_commit();
    }
    const int jb0 = load_block_list(p, i, L, j0, j1, sBlk, g == 0);
    __syncthreads();

    const __nv_bfloat16 *Kseq = reinterpret_cast<const __nv_bfloat16 *>(p.K) +
                                (int64_t)L.seq * p.k_seq_stride + (int64_t)g * DKQ;
    const __nv_bfloat16 *Vseq = V_IS_K ? Kseq
                                       : reinterpret_cast<const __nv_bfloat16 *>(p.V) +
                                             (int64_t)L.seq * p.v_seq_stride + (int64_t)g * DV;
    const int n_tiles = (j1 - j0 + kT - 1) / kT;

    auto issue_tile = [&](int t) {
        const int st = t % p.stages;
        uint8_t *dstK = sStage + (size_t)st * STAGE_BYTES;
        const int r = tid >> 2, sub = tid & 3;
        const int tok = token_at(p, L, j0 + t * kT + r, j1, sBlk, jb0);
        if (sub == 0) sTok[st * kT + r] = tok;
        const __nv_bfloat16 *srcK = tok >= 0 ? Kseq + (int64_t)tok * p.k_tok_stride : Kseq;
        const uint32_t nbytes = tok >= 0 ? 16u : 0u;
        const uint32_t rowK = smem_u32(dstK) + r * KROW;
#pragma unroll 6
        for (int c = sub; c < KCH; c += 4) cp_async16(rowK + swz(c, r) * 16, srcK + c * 8, nbytes);
        if constexpr (!V_IS_K) {
            const __nv_bfloat16 *srcV = tok >= 0 ? Vseq + (int64_t)tok * p.v_tok_stride : Vseq;
            const uint32_t rowV = smem_u32(dstK + kT * KROW) + r * VROW;
#pragma unroll 4
            for (int c = sub; c < VCH; c += 4)
                cp_async16(rowV + swz(c, r) * 16, srcV + c * 8, nbytes);
        }
    };

    // prologue: stages-1 tiles in flight (behind the Q group)
    for (int t = 0; t < p.stages - 1; ++t) {
        if (t < n_tiles) issue_tile(t);
        cp_async_commit();
    }
    // Q has landed once at most stages-1 younger groups are pending
    if (p.stages == 2) cp_async_wait<1>();
    else if (p.stages == 3) cp_async_wait<2>();
    else cp_async_wait<3>();
    __syncthreads();

    // Q fragments of this warp's head-dim slice (A operand, kept in registers)
    uint32_t qa[KS][4];
    {
        const uint32_t q_base = smem_u32(sQ);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int kg = warp * KS + ks;
            const int r = lane & 15, c = kg * 2 + (lane >> 4);
            ldsm_x4(q_base + r * KROW + swz(c, r) * 16, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
        }
    }

    float o[NTV][4];
#pragma unroll
    for (int n = 0; n < NTV; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;   // of row (tid >> 3), kept by its 8 threads

    const int gq = lane >> 2, tq = lane & 3;
    for (int t = 0; t < n_tiles; ++t) {
        // tile t has landed once at most stages-2 younger groups are pending
        if (p.stages == 2) cp_async_wait<0>();
        else if (p.stages == 3) cp_async_wait<1>();
        else cp_async_wait<2>();
        __syncthreads();
        if (t + p.stages - 1 < n_tiles) issue_tile(t + p.stages - 1);
        cp_async_commit();

        const int st = t % p.stages;
        const uint32_t kbase = smem_u32(sStage + (size_t)st * STAGE_BYTES);
        const uint32_t vbase = V_IS_K ? kbase : kbase + kT * KROW;

        // ---- S partial over this warp's head-dim slice
        float acc[kT / 8][4];
#pragma unroll
        for (int n = 0; n < kT / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
        for (int np = 0; np < kT / 16; ++np) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int kg = warp * KS + ks;
                const int mi = lane >> 3, r8 = lane & 7;
                const int n = np * 16 + (mi >> 1) * 8 + r8;
                const int c = kg * 2 + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + n * KROW + swz(c, n) * 16, b0, b1, b2, b3);
                mma_bf16_16816(acc[2 * np], qa[ks], b0, b1);
                mma_bf16_16816(acc[2 * np + 1], qa[ks], b2, b3);
            }
        }
        float *sp = sSP + warp * 16 * SP_PITCH;
#pragma unroll
        for (int n = 0; n < kT / 8; ++n) {
            *reinterpret_cast<float2 *>(sp + gq * SP_PITCH + n * 8 + 2 * tq) = make_float2(acc[n][0], acc[n][1]);
            *reinterpret_cast<float2 *>(sp + (gq + 8) * SP_PITCH + n * 8 + 2 * tq) = make_float2(acc[n][2], acc[n][3]);
        }
        __syncthreads();

        // ---- online softmax: thread -> row tid/8, columns 4*(tid%8) .. +3
        {
            const int row = tid >> 3, c0 = (tid & 7) * 4;
            float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float4 v = *reinterpret_cast<const float4 *>(sSP + (w * 16 + row) * SP_PITCH + c0);
                s[0] += v.x; s[1] += v.y; s[2] += v.z; s[3] += v.w;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[e] = sTok[st * kT + c0 + e] >= 0 ? s[e] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[e]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
            float ph[4], pl[4], rs = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float pe = m_new == -INFINITY ? 0.f : exp2f(s[e] - m_new);
                ph[e] = __bfloat162float(__float2bfloat16_rn(pe));
                pl[e] = pe - ph[e];
                rs += pe;
            }
            rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 1);
            rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 2);
            rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 4);
            l_run = l_run * alpha + rs;
            m_run = m_new;
            *reinterpret_cast<uint2 *>(sP + row * P_PITCH + c0) =
                make_uint2(pack_bf16(ph[0], ph[1]), pack_bf16(ph[2], ph[3]));
            *reinterpret_cast<uint2 *>(sP + (16 + row) * P_PITCH + c0) =
                make_uint2(pack_bf16(pl[0], pl[1]), pack_bf16(pl[2], pl[3]));
            if ((tid & 7) == 0) sAlpha[row] = alpha;
        }
        __syncthreads();

        // ---- O = O * alpha + P V over this warp's value-dim slice
        {
            const float a0 = sAlpha[gq], a1 = sAlpha[gq + 8];
#pragma unroll
            for (int n = 0; n < NTV; ++n) {
                o[n][0] *= a0; o[n][1] *= a0; o[n][2] *= a1; o[n][3] *= a1;
            }
            const uint32_t pbase = smem_u32(sP);
#pragma unroll
            for (int ks = 0; ks < kT / 16; ++ks) {
                uint32_t pa[4], pb[4];
                {
                    const int r = lane & 15, col = ks * 16 + (lane >> 4) * 8;
                    const uint32_t a = pbase + r * (P_PITCH * 2) + col * 2;
                    ldsm_x4(a, pa[0], pa[1], pa[2], pa[3]);
                    ldsm_x4(a + 16 * P_PITCH * 2, pb[0], pb[1], pb[2], pb[3]);
                }
#pragma unroll
                for (int np = 0; np < NTV / 2; ++np) {
                    const int mi = lane >> 3, r8 = lane & 7;
                    const int k = ks * 16 + (mi & 1) * 8 + r8;
                    const int c = (warp * (DV / 4)) / 8 + np * 2 + (mi >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vbase + k * VROW + swz(c, k) * 16, b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * np], pa, b0, b1);
                    mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
                    mma_bf16_16816(o[2 * np], pb, b0, b1);
                    mma_bf16_16816(o[2 * np + 1], pb, b2, b3);
                }
            }
        }
    }
    cp_async_wait<0>();

    // ---- epilogue
    if ((tid & 7) == 0) {
        sL[tid >> 3] = l_run;
        sM[tid >> 3] = m_run;
    }
    __syncthreads();
    const int dv0 = warp * (DV / 4);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int row = gq + half * 8;
        if (row >= G) continue;
        const int h = g * G + row;
        const float l = sL[row], m = sM[row];
        if (p.n_split == 1) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float *dst = p.O + ((int64_t)i * p.h_q + h) * DV + dv0;
#pragma unroll
            for (int n = 0; n < NTV; ++n)
                *reinterpret_cast<float2 *>(dst + n * 8 + 2 * tq) =
                    make_float2(o[n][2 * half] * inv, o[n][2 * half + 1] * inv);
            if (p.lse && tq == 0 && warp == 0)
                p.lse[(int64_t)i * p.h_q + h] = l > 0.f ? (m + log2f(l)) / kLog2e : -INFINITY;
        } else {
            const int64_t base = (((int64_t)i * p.h_kv + g) * p.n_split + split) * G + row;
            float *dst = p.part_o + base * DV + dv0;
#pragma unroll
            for (int n = 0; n < NTV; ++n)
                *reinterpret_cast<float2 *>(dst + n * 8 + 2 * tq) =
                    make_float2(o[n][2 * half], o[n][2 * half + 1]);
            if (tq == 0 && warp == 0) {
                p.part_ml[base * 2] = m;
                p.part_ml[base * 2 + 1] = l;
            }
        }
    }
}

// fp32 inputs: plain SIMT online softmax, one head per 8 threads (accuracy path).
template <int DKQ, int DV>
__global__ void __launch_bounds__(kThreads) attend_f32_kernel(const AttnParams p) {
    constexpr int QE = DKQ / 8, OE = DV / 8;
    __shared__ int sBlk[kMaxBlkList];
    const int tid = threadIdx.x;
    const int split = blockIdx.x, g = blockIdx.y, i = blockIdx.z;
    const int row = tid >> 3, part = tid & 7;
    const ListInfo L = list_info(p, i, split == 0 && g == 0 && tid == 0);
    const int j0 = split * p.split_tokens;
    const int j1 = L.ok ? min(L.len, j0 + p.split_tokens) : 0;
    const int jb0 = j0 < j1 ? load_block_list(p, i, L, j0, j1, sBlk, g == 0) : 0;
    __syncthreads();
    const int G = p.G;
    const bool active = row < G;
    const int h = g * G + (active ? row : 0);
    float q[QE], o[OE];
    const float *Qh = reinterpret_cast<const float *>(p.Q) + ((int64_t)i * p.h_q + h) * DKQ;
#pragma unroll
    for (int e = 0; e < QE; ++e) q[e] = Qh[part + 8 * e];
#pragma unroll
    for (int e = 0; e < OE; ++e) o[e] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    const float *Kseq = reinterpret_cast<const float *>(p.K) + (int64_t)(L.ok ? L.seq : 0) * p.k_seq_stride + (int64_t)g * DKQ;
    const float *Vseq = p.V ? reinterpret_cast<const float *>(p.V) + (int64_t)(L.ok ? L.seq : 0) * p.v_seq_stride + (int64_t)g * DV
                            : Kseq;
    const int64_t vstride = p.V ? p.v_tok_stride : p.k_tok_stride;
    for (int j = j0; j < j1; ++j) {
        const int tok = token_at(p, L, j, j1, sBlk, jb0);
        if (tok < 0) continue;
        const float *kr = Kseq + (int64_t)tok * p.k_tok_stride;
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < QE; ++e) s = fmaf(q[e], kr[part + 8 * e], s);
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 4);
        s *= p.scale_log2;
        const float m_new = fmaxf(m_run, s);
        const float corr = exp2f(m_run - m_new);
        const float pe = exp2f(s - m_new);
        l_run = l_run * corr + pe;
        m_run = m_new;
        const float *vr = Vseq + (int64_t)tok * vstride;
#pragma unroll
        for (int e = 0; e < OE; ++e) o[e] = fmaf(pe, vr[part + 8 * e], o[e] * corr);
    }
    if (!active) return;
    if (p.n_split == 1) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        float *dst = p.O + ((int64_t)i * p.h_q + h) * DV;
#pragma unroll
        for (int e = 0; e < OE; ++e) dst[part + 8 * e] = o[e] * inv;
        if (p.lse && part == 0)
            p.lse[(int64_t)i * p.h_q + h] = l_run > 0.f ? (m_run + log2f(l_run)) / kLog2e : -INFINITY;
    } else {
        const int64_t base = (((int64_t)i * p.h_kv + g) * p.n_split + split) * G + row;
        float *dst = p.part_o + base * DV;
#pragma unroll
        for (int e = 0; e < OE; ++e) dst[part + 8 * e] = o[e];
        if (part == 0) {
            p.part_ml[base * 2] = m_run;
            p.part_ml[base * 2 + 1] = l_run;
        }
    }
}

// Merges the split partials of one (query, head): grid (n_q * h_q), 128 threads.  Warp 0
// turns the splits' (m, l) into merge weights in shared memory; then each thread owns 4
// consecutive value dims and sums the weighted partials with 16-byte loads.
__global__ void __launch_bounds__(128) combine_kernel(const AttnParams p, int dv) {
    extern __shared__ float s_w[];  // [n_split] weights, then 1/L and M
    const int i = blockIdx.x / p.h_q, h = blockIdx.x % p.h_q;
    const int g = h / p.G, row = h % p.G;
    const int64_t base0 = ((int64_t)i * p.h_kv + g) * p.n_split * p.G + row;
    const int ns = p.n_split;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        float M = -INFINITY;
        for (int s = lane; s < ns; s += 32) M = fmaxf(M, p.part_ml[(base0 + (int64_t)s * p.G) * 2]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        float L = 0.f;
        for (int s = lane; s < ns; s += 32) {
            const int64_t b = base0 + (int64_t)s * p.G;
            const float m = p.part_ml[b * 2];
            const float w = m == -INFINITY ? 0.f : exp2f(m - M);
            s_w[s] = w;
            L += w * p.part_ml[b * 2 + 1];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
        if (lane == 0) {
            s_w[ns] = L > 0.f ? 1.f / L : 0.f;
            s_w[ns + 1] = M;
            if (p.lse) p.lse[(int64_t)i * p.h_q + h] = L > 0.f ? (M + log2f(L)) / kLog2e : -INFINITY;
        }
    }
    __syncthreads();
    const float inv = s_w[ns];
    const int64_t stride4 = (int64_t)p.G * dv / 4;   // float4 step between splits
    const float4 *src = reinterpret_cast<const float4 *>(p.part_o + base0 * dv);
    float4 *dst = reinterpret_cast<float4 *>(p.O + ((int64_t)i * p.h_q + h) * dv);
    for (int d4 = threadIdx.x; d4 < dv / 4; d4 += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int s = 0; s < ns; ++s) {
            const float w = s_w[s];
            const float4 v = __ldg(src + s * stride4 + d4);
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        dst[d4] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

// ------------------------------------------------------------------------------ host side
struct SplitPlan {
    int n_split, split_tokens;
};

// Few (query, KV head) items -> split each list so that the CTAs fill one wave (one CTA per
// SM: each streams a long run of tiles, so its fixed start-up cost is amortised); many items
// -> one CTA per item.
SplitPlan plan_split(int n_q, int h_kv, int64_t n_kv_max, int per_sm = 2) {
    const int64_t items = (int64_t)n_q * h_kv;
    const int64_t tiles = (n_kv_max + kT - 1) / kT;
    const int64_t target = (int64_t)per_sm * device_sm_count();
    int64_t ns = target / items;
    if (ns > tiles) ns = tiles;
    if (ns < 1) ns = 1;
    const int64_t per = (tiles + ns - 1) / ns;
    SplitPlan sp;
    sp.split_tokens = (int)(per * kT);
    sp.n_split = (int)((tiles + per - 1) / per);
    if (sp.n_split < 1) sp.n_split = 1;
    return sp;
}

bool shape_supported(int dkq, int dv) {
    return (dkq == 576 && dv == 512) || (dkq == 512 && dv == 512) || (dkq == 128 && dv == 128) ||
           (dkq == 64 && dv == 64);
}

// Shared memory of one bf16 CTA: the K/V stages plus Q, the S partials, P (hi, lo), the
// softmax statistics, the token ids and the block list of its split.
template <int DKQ, int DV, bool VK>
size_t bf16_smem(int stages, int blk_list) {
    constexpr int KROW = DKQ * 2, VROW = VK ? KROW : DV * 2;
    constexpr int STAGE = kT * KROW + (VK ? 0 : kT * VROW);
    return (size_t)stages * STAGE + 16 * KROW + 4 * 16 * (kT + 8) * 4 + 2 * 16 * (kT + 8) * 2 +
           48 * 4 + (size_t)stages * kT * 4 + (size_t)blk_list * 4 + 16;
}

// Two CTAs per SM when two stages fit in half the shared memory (more warps to hide the
// latency of each tile's dependent steps), else one CTA with up to four stages.
template <int DKQ, int DV, bool VK>
int bf16_per_sm(int blk_list) {
    return bf16_smem<DKQ, DV, VK>(2, blk_list) <= 113 * 1024 ? 2 : 1;
}

template <int DKQ, int DV, bool VK>
int launch_bf16(const AttnParams &p, dim3 grid, cudaStream_t st, int blk_list) {
    int stages = 2;
    if (bf16_per_sm<DKQ, DV, VK>(blk_list) == 1) {
        stages = 4;
        while (stages > 2 && bf16_smem<DKQ, DV, VK>(stages, blk_list) > 227 * 1024) --stages;
    }
    if (bf16_smem<DKQ, DV, VK>(stages, blk_list) > 227 * 1024) return SFA_ERR_UNSUPPORTED;
    AttnParams q = p;
    q.stages = stages;
    const size_t smem = bf16_smem<DKQ, DV, VK>(stages, blk_list);
    static bool attr = false;
    if (!attr) {
        if (!allow_max_dynamic_smem(attend_bf16_kernel<DKQ, DV, VK>)) return SFA_ERR_CUDA;
        attr = true;
    }
    attend_bf16_kernel<DKQ, DV, VK><<<grid, kThreads, smem, st>>>(q);
    SFA_CHECK_LAUNCH();
    return SFA_OK;
}

int run_attend(const void *Q, const void *K, const void *V, int dtype, int n_seq,
               int64_t n_tok_cap, int n_q, int h_q, int h_kv, int dkq, int dv, float scale,
               const int32_t *q_seq, const int32_t *q_pos, const int32_t *blk_idx,
               const int32_t *n_sel, int top_k, int cr, int dense, int64_t n_kv_max, float *O,
               float *lse, void *ws, size_t ws_bytes, int32_t *status, cudaStream_t st) {
    if (!Q || !K || !q_seq || !q_pos || !O) return SFA_ERR_INVALID_ARG;
    if (dtype != SFA_BF16 && dtype != SFA_F32) return SFA_ERR_INVALID_ARG;
    if (n_seq < 1 || n_tok_cap < 1 || n_q < 0 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0)
        return SFA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return SFA_ERR_INVALID_ARG;
    if (!dense && (!blk_idx || !n_sel || cr < 1 || top_k < 1)) return SFA_ERR_INVALID_ARG;
    if (!dense && top_k > 2048) return SFA_ERR_UNSUPPORTED;
    if (n_kv_max < 1) return SFA_ERR_INVALID_ARG;
    if (dv > dkq && !V) return SFA_ERR_INVALID_ARG;
    if (!shape_supported(dkq, dv) || h_q / h_kv > 16) return SFA_ERR_UNSUPPORTED;
    if (!aligned16(Q) || !aligned16(K) || (V && !aligned16(V)) || !aligned16(O))
        return SFA_ERR_INVALID_ARG;
    if (n_q == 0) return SFA_OK;
    if (n_q > 65535 || h_kv > 65535 || n_kv_max > 0x7FFFFFFF) return SFA_ERR_UNSUPPORTED;
    // resident CTAs per SM of the kernel this shape takes (the split plan fills them once)
    int per_sm = 1;
    if (dtype == SFA_BF16) {
        const int bl_max = dense ? 0 : (int)(n_kv_max / cr + 2);
        if (dkq == 576) per_sm = bf16_per_sm<576, 512, true>(bl_max);
        else if (dkq == 512) per_sm = V ? bf16_per_sm<512, 512, false>(bl_max) : bf16_per_sm<512, 512, true>(bl_max);
        else if (dkq == 128) per_sm = V ? bf16_per_sm<128, 128, false>(bl_max) : bf16_per_sm<128, 128, true>(bl_max);
        else per_sm = V ? bf16_per_sm<64, 64, false>(bl_max) : bf16_per_sm<64, 64, true>(bl_max);
    }
    const SplitPlan sp = plan_split(n_q, h_kv, n_kv_max, per_sm);
    const size_t need = sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv_max);
    if (need > 0 && (!ws || ws_bytes < need)) return SFA_ERR_WORKSPACE;

    AttnParams p{};
    p.Q = Q; p.K = K; p.V = V;
    p.q_seq = q_seq; p.q_pos = q_pos; p.blk_idx = blk_idx; p.n_sel = n_sel;
    p.O = O; p.lse = lse; p.status = status;
    p.k_tok_stride = (int64_t)h_kv * dkq;
    p.k_seq_stride = n_tok_cap * p.k_tok_stride;
    p.v_tok_stride = V ? (int64_t)h_kv * dv : p.k_tok_stride;
    p.v_seq_stride = V ? n_tok_cap * p.v_tok_stride : p.k_seq_stride;
    p.n_tok_cap = n_tok_cap;
    p.n_seq = n_seq; p.n_q = n_q; p.h_q = h_q; p.h_kv = h_kv; p.G = h_q / h_kv;
    p.top_k = top_k; p.cr = cr; p.dense = dense;
    p.n_split = sp.n_split; p.split_tokens = sp.split_tokens;
    p.scale_log2 = scale * kLog2e;
    if (sp.n_split > 1) {
        const size_t n_rows = (size_t)n_q * h_q * sp.n_split;
        p.part_o = reinterpret_cast<float *>(ws);
        p.part_ml = p.part_o + n_rows * dv;
    }
    if (!dense && (int64_t)sp.split_tokens / cr + 2 > kMaxBlkList) return SFA_ERR_UNSUPPORTED;
    const int bl = dense ? 0 : sp.split_tokens / cr + 2;   // block-list entries a split needs
    const dim3 grid(sp.n_split, h_kv, n_q);
    int rc;
    if (dtype == SFA_BF16) {
        if (dkq == 576) rc = V ? SFA_ERR_UNSUPPORTED : launch_bf16<576, 512, true>(p, grid, st, bl);
        else if (dkq == 512) rc = V ? launch_bf16<512, 512, false>(p, grid, st, bl) : launch_bf16<512, 512, true>(p, grid, st, bl);
        else if (dkq == 128) rc = V ? launch_bf16<128, 128, false>(p, grid, st, bl) : launch_bf16<128, 128, true>(p, grid, st, bl);
        else rc = V ? launch_bf16<64, 64, false>(p, grid, st, bl) : launch_bf16<64, 64, true>(p, grid, st, bl);
    } else {
        if (dkq == 576) attend_f32_kernel<576, 512><<<grid, kThreads, 0, st>>>(p);
        else if (dkq == 512) attend_f32_kernel<512, 512><<<grid, kThreads, 0, st>>>(p);
        else if (dkq == 128) attend_f32_kernel<128, 128><<<grid, kThreads, 0, st>>>(p);
        else attend_f32_kernel<64, 64><<<grid, kThreads, 0, st>>>(p);
        rc = cudaGetLastError() == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
    }
    if (rc != SFA_OK) return rc;
    if (sp.n_split > 1) {
        combine_kernel<<<n_q * h_q, 128, (sp.n_split + 2) * sizeof(float), st>>>(p, dv);
        SFA_CHECK_LAUNCH();
    }
    return SFA_OK;
}

}  // namespace
}  // namespace sfa

extern "C" size_t sfa_attend_workspace_bytes(int n_q, int h_q, int h_kv, int dv, int64_t n_kv_max) {
    if (n_q <= 0 || h_q <= 0 || h_kv <= 0 || dv <= 0 || n_kv_max <= 0) return 0;
    const sfa::SplitPlan sp = sfa::plan_split(n_q, h_kv, n_kv_max, 2);  // the largest plan
    if (sp.n_split <= 1) return 0;
    return (size_t)n_q * h_q * sp.n_split * ((size_t)dv + 2) * sizeof(float);
}

extern "C" int sfa_gather_attend(const void *Q, const void *K, const void *V, int dtype,
                                 int n_seq, int64_t n_tok_cap, int n_q, int h_q, int h_kv,
                                 int dkq, int dv, float scale, const int32_t *q_seq,
                                 const int32_t *q_pos, const int32_t *blk_idx,
                                 const int32_t *n_sel, int top_k, int compress_ratio, float *O,
                                 float *lse, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, sfa_stream_t stream) {
    if (compress_ratio < 1 || top_k < 1) return SFA_ERR_INVALID_ARG;
    const int64_t n_kv_max = (int64_t)top_k * compress_ratio + compress_ratio - 1;
    return sfa::run_attend(Q, K, V, dtype, n_seq, n_tok_cap, n_q, h_q, h_kv, dkq, dv, scale,
                           q_seq, q_pos, blk_idx, n_sel, top_k, compress_ratio, 0, n_kv_max, O,
                           lse, workspace, workspace_bytes, dev_status, (cudaStream_t)stream);
}

extern "C" int sfa_dense_attend(const void *Q, const void *K, const void *V, int dtype,
                                int n_seq, int64_t n_tok_cap, int n_q, int h_q, int h_kv,
                                int dkq, int dv, float scale, const int32_t *q_seq,
                                const int32_t *q_pos, int64_t n_kv_max, float *O, float *lse,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                sfa_stream_t stream) {
    return sfa::run_attend(Q, K, V, dtype, n_seq, n_tok_cap, n_q, h_q, h_kv, dkq, dv, scale,
                           q_seq, q_pos, nullptr, nullptr, 0, 1, 1, n_kv_max, O, lse, workspace,
                           workspace_bytes, dev_status, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------------------
// sfa_gather_attend_noalloc: the split-KV scratch lives in this file-scope device array, so
// the call allocates nothing.  Host code may not use the array's name as a device address:
// the address is looked up once per device with cudaGetSymbolAddress and cached.
namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[SFA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64] = {nullptr};

// Device address of g_noalloc_scratch on the current device (nullptr on failure).
void *noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}
}  // namespace

extern "C" int sfa_gather_attend_noalloc(const void *Q, const void *K, const void *V, int dtype,
                                         int n_seq, int64_t n_tok_cap, int n_q, int h_q,
                                         int h_kv, int dkq, int dv, float scale,
                                         const int32_t *q_seq, const int32_t *q_pos,
                                         const int32_t *blk_idx, const int32_t *n_sel,
                                         int top_k, int compress_ratio, float *O, float *lse,
                                         int32_t *dev_status, sfa_stream_t stream) {
    if (compress_ratio < 1 || top_k < 1) return SFA_ERR_INVALID_ARG;
    const int64_t n_kv_max = (int64_t)top_k * compress_ratio + compress_ratio - 1;
    const size_t need = sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv_max);
    if (need > SFA_NOALLOC_SCRATCH_BYTES) return SFA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        scratch = noalloc_scratch();
        if (!scratch) return SFA_ERR_CUDA;
    }
    return sfa::run_attend(Q, K, V, dtype, n_seq, n_tok_cap, n_q, h_q, h_kv, dkq, dv, scale,
                           q_seq, q_pos, blk_idx, n_sel, top_k, compress_ratio, 0, n_kv_max, O,
                           lse, scratch, need, dev_status, (cudaStream_t)stream);
}
