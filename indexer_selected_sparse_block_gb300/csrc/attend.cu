// attend.cu -- gathered flash attention over the kept cells (sfa_gather_attend) and its
// below-budget dense twin (sfa_dense_attend): the warp-level kernel (the default for bf16 and
// q8_0 caches), the tcgen05 kernel (opt-in), the fp32 SIMT kernel, combine_kernel, the launch
// plans and the C entry points.  The attended list of a query and the shared parameters are in
// attend_common.cuh; the warp-specialised bulk-copy kernel (opt-in) is in attend_ws.cu.
//
// bf16 kernel (one CTA = one query x one KV head x one split of its list, 4 warps, two CTAs
// per SM):
//   * cp.async 16-byte gathers of the selected token rows, 32 rows per stage (each kept block
//     is cr contiguous rows), XOR-swizzled rows so that ldmatrix is conflict-free;
//   * S = Q K^T on tensor cores (mma.sync m16n8k16, M = the 16 query heads of the KV head),
//     the head dim split over the 4 warps and the partial sums reduced through shared memory;
//   * online softmax (base 2) over the tile; P is carried as two bf16 halves
//     (hi = bf16(p), lo = bf16(p - hi)), so P V is accurate to ~2^-17 instead of the 2^-9 of
//     a single bf16 rounding (which alone uses up a 2e-3 output tolerance);
//   * O += P_hi V + P_lo V on tensor cores, the 512 value dims split over the 4 warps; V = K
//     reuses the K tile in shared memory.
// Decode has few queries, so each list is split over several CTAs (flash-decoding); the
// partial (O, m, l) merge inside a thread-block cluster or through combine_kernel.  With an
// in-cluster merge and V = K, the splits cover the kept tokens only and the last one attends
// the few tail tokens as a 16-token tile loaded into the Q buffer at its start (AttnParams::
// tail_fold), so that no split spends a whole 32-token tile on them.  fp32 inputs
// take a plain SIMT kernel with the same split/merge structure (accuracy reference path).
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include <cooperative_groups.h>

#include "attend_common.cuh"

namespace sfa {
namespace {

namespace cg = cooperative_groups;

__device__ __forceinline__ uint32_t swz(int c, int r) { return (uint32_t)((c & ~7) | ((c ^ r) & 7)); }

// The merge of the splits of one (query, KV head) inside their cluster (flash-decoding without
// a second kernel): each CTA holds its unnormalised O rows sPart[G][DV] and their (m, l) in
// sM, sL (base-2 maxima and sums); CTA r of the n_split writes the value dims [r DV/ns,
// (r+1) DV/ns) of every row as sum_c w_c O_c / sum_c w_c l_c with w_c = 2^(m_c - M), reading
// the other CTAs' shared memory.  sW (n_split * 16 + 32 floats) is this CTA's scratch.
template <int DV>
__device__ void cluster_merge(const AttnParams &p, float *sPart, float *sL, float *sM, float *sW,
                              int i, int g) {
    cg::cluster_group cl = cg::this_cluster();
    const int tid = threadIdx.x, G = p.G, ns = p.n_split;
    cl.sync();   // every CTA's partial rows and statistics are in its shared memory
    const int r = (int)cl.block_rank();
    // Every remote load of a step is issued before any is used (the split count is at most 8,
    // unrolled with predicates): one round trip over distributed shared memory per step
    // instead of one per split.
    constexpr int kMaxNs = 8;
    if (tid < G) {
        float mv[kMaxNs], lv[kMaxNs];
#pragma unroll
        for (int c = 0; c < kMaxNs; ++c) {
            mv[c] = c < ns ? cl.map_shared_rank(sM, c)[tid] : -INFINITY;
            lv[c] = c < ns ? cl.map_shared_rank(sL, c)[tid] : 0.f;
        }
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kMaxNs; ++c) M = fmaxf(M, mv[c]);
        float Lsum = 0.f, wv[kMaxNs];
#pragma unroll
        for (int c = 0; c < kMaxNs; ++c) {
            wv[c] = mv[c] == -INFINITY ? 0.f : exp2f(mv[c] - M);
            Lsum += wv[c] * lv[c];
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
        for (int c = 0; c < kMaxNs; ++c)
            if (c < ns) sW[c * 16 + tid] = wv[c] * inv;
        if (r == 0 && p.lse)
            p.lse[(int64_t)i * p.h_q + g * G + tid] = Lsum > 0.f ? (M + log2f(Lsum)) / kLog2e : -INFINITY;
    }
    __syncthreads();
    const int dq = DV / ns / 4;   // float4 per row in this CTA's slice
    const int d0 = r * (DV / ns);
    for (int e = tid; e < G * dq; e += kThreads) {
        const int row = e / dq, d = d0 + 4 * (e % dq);
        float wc[kMaxNs];
        float4 v[kMaxNs];
#pragma unroll
        for (int c = 0; c < kMaxNs; ++c) {
            wc[c] = c < ns ? sW[c * 16 + row] : 0.f;
            // an empty split (weight 0) wrote no rows: not read
            v[c] = wc[c] != 0.f
                       ? *reinterpret_cast<const float4 *>(cl.map_shared_rank(sPart, c) + row * DV + d)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kMaxNs; ++c) {
            acc.x = fmaf(wc[c], v[c].x, acc.x);
            acc.y = fmaf(wc[c], v[c].y, acc.y);
            acc.z = fmaf(wc[c], v[c].z, acc.z);
            acc.w = fmaf(wc[c], v[c].w, acc.w);
        }
        *reinterpret_cast<float4 *>(p.O + ((int64_t)i * p.h_q + g * G + row) * DV + d) = acc;
    }
    cl.sync();   // no CTA leaves while another may still read its shared memory
}

// m16n8k16 MMA, packing and rounding of the 16-bit operand type: bf16, or binary16 (F16).
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (F16) mma_f16_16816(d, a, b0, b1);
    else mma_bf16_16816(d, a, b0, b1);
}
template <bool F16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
    if constexpr (F16) return pack_f16(lo, hi);
    else return pack_bf16(lo, hi);
}
template <bool F16>
__device__ __forceinline__ float round16(float x) {
    if constexpr (F16) return __half2float(__float2half_rn(x));
    else return __bfloat162float(__float2bfloat16_rn(x));
}

// Dequantizes TT q8_0 rows of D elements (pitch SROW bytes: D codes, then D/32 binary16 scales)
// into binary16 rows of the swizzled tile layout (pitch 2*D bytes): element j of a row is
// scale(j / 32) * code_j, exact in fp32, then rounded to binary16.  Zero-filled rows (padding)
// give zeros.  Returns false when a value exceeds binary16's range.
// Four int8 codes (one 32-bit word) -> two pairs of binary16 values, exactly: each biased code
// c + 128 becomes the low byte of binary16 1024 + (c + 128) (a byte permute), and subtracting
// 1152 leaves c.
__device__ __forceinline__ void codes_to_f16(uint32_t w, __half2 &c01, __half2 &c23) {
    const uint32_t b = w ^ 0x80808080u;
    const uint32_t h01 = __byte_perm(b, 0x64646464u, 0x5140u);
    const uint32_t h23 = __byte_perm(b, 0x64646464u, 0x7362u);
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480u));   // 1152
    c01 = __hsub2(*reinterpret_cast<const __half2 *>(&h01), bias);
    c23 = __hsub2(*reinterpret_cast<const __half2 *>(&h23), bias);
}

// Chunks [c0, c0 + NC) of 8 elements of every row of the tile, by the threads first, first +
// stride, ...
template <int D, int SROW, int TT, int NC>
__device__ __forceinline__ bool dequant_tile(const uint8_t *src, uint8_t *dst, int c0, int first,
                                             int stride) {
    bool ok = true;
    for (int e = first; e < TT * NC; e += stride) {
        const int r = e / NC, c = c0 + (e - r * NC);
        const uint8_t *row = src + r * SROW;
        const uint2 w = *reinterpret_cast<const uint2 *>(row + c * 8);
        const __half s = *reinterpret_cast<const __half *>(row + D + (c >> 2) * 2);
        uint4 out;
        if (fabsf(__half2float(s)) * 127.f < 65520.f) {
            // scale * code is exact in binary32 (11 x 8 significant bits) and one binary16
            // multiply rounds that exact product once, as the conversion of the binary32
            // product does
            const __half2 s2 = __half2half2(s);
            __half2 c0, c1, c2, c3;
            codes_to_f16(w.x, c0, c1);
            codes_to_f16(w.y, c2, c3);
            const __half2 v0 = __hmul2(c0, s2), v1 = __hmul2(c1, s2), v2 = __hmul2(c2, s2),
                          v3 = __hmul2(c3, s2);
            out = make_uint4(*reinterpret_cast<const uint32_t *>(&v0),
                             *reinterpret_cast<const uint32_t *>(&v1),
                             *reinterpret_cast<const uint32_t *>(&v2),
                             *reinterpret_cast<const uint32_t *>(&v3));
        } else {   // a scale that can overflow binary16: the binary32 path, with the range check
            const float sc = __half2float(s);
            float v[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[k] = sc * (float)(int8_t)(w.x >> (8 * k));
                v[4 + k] = sc * (float)(int8_t)(w.y >> (8 * k));
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) ok &= fabsf(v[k]) < 65520.f;
            out = make_uint4(pack_f16(v[0], v[1]), pack_f16(v[2], v[3]), pack_f16(v[4], v[5]),
                             pack_f16(v[6], v[7]));
        }
        *reinterpret_cast<uint4 *>(dst + r * (2 * D) + swz(c, r) * 16) = out;
    }
    return ok;
}

// Waits until at most n of this thread's cp.async groups are pending (n in 0 .. 5).
__device__ __forceinline__ void cp_async_wait_n(int n) {
    switch (n) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        default: cp_async_wait<5>(); break;
    }
}

// Shared memory of one CTA of the warp-level kernel with TT-token tiles: the K/V stages (Q8:
// quantized rows, plus one binary16 tile), Q, the S partials, P (hi, lo), the softmax
// statistics, the token ids and the block list of its split.  The layout is attend_mma_body's.
template <int DKQ, int DV, bool VK, bool Q8, int TT>
__host__ __device__ constexpr size_t mma_smem_bytes(int stages, int blk_list) {
    return (size_t)stages * (Q8 ? TT * q8_row_bytes(DKQ) + (VK ? 0 : TT * q8_row_bytes(DV))
                                : TT * DKQ * 2 + (VK ? 0 : TT * DV * 2)) +
           (Q8 ? TT * DKQ * 2 + (VK ? 0 : TT * DV * 2) : 0) + 16 * DKQ * 2 + 4 * 16 * (TT + 8) * 4 +
           2 * 16 * (TT + 8) * 2 + 48 * 4 + (size_t)stages * TT * 4 + (size_t)blk_list * 4 + 16;
}

// Gathered attention on warp-level MMAs: the body of attend_bf16_kernel (bf16 K/V) and of
// attend_q8_kernel (Q8: q8_0 K/V rows, gathered as such, dequantized per tile in shared memory
// to binary16, with Q converted to binary16 and every tensor-core product on binary16).
// Tiles of TT tokens (16 or 32) stream through a ring of p.stages stages: tile t + stages - 1
// is issued while tile t is scored, so stages - 1 tiles are in flight behind the one in use.
template <int DKQ, int DV, bool V_IS_K, bool Q8, int TT, bool FOLD = false>
__device__ __forceinline__ void attend_mma_body(const AttnParams &p) {
    static_assert(!FOLD || (!Q8 && V_IS_K && TT == 32), "the folded tail: bf16, V = K, TT 32");
    constexpr int KROW = DKQ * 2;                 // bytes of a K row in shared memory
    constexpr int VROW = V_IS_K ? KROW : DV * 2;  // bytes of a V row
    constexpr int KCH = DKQ / 8, VCH = DV / 8;    // 16-byte chunks per row
    constexpr int KS = DKQ / 64;                  // k16 steps of S per warp
    constexpr int NTV = DV / 32;                  // n8 tiles of O per warp
    constexpr int SP_PITCH = TT + 8;              // fp32 S-partial row pitch
    constexpr int P_PITCH = TT + 8;               // 16-bit P row pitch
    constexpr int TPR = kThreads / TT;            // copying threads per tile row
    constexpr int SPT = TT / 8;                   // softmax columns per thread
    static_assert(TT == 16 || TT == 32, "tile sizes");
    constexpr int QKROW = q8_row_bytes(DKQ), QVROW = q8_row_bytes(DV);   // q8_0 rows (Q8)
    constexpr int STAGE_BYTES = Q8 ? TT * QKROW + (V_IS_K ? 0 : TT * QVROW)
                                   : TT * KROW + (V_IS_K ? 0 : TT * VROW);
    constexpr int DEQ_BYTES = Q8 ? TT * KROW + (V_IS_K ? 0 : TT * VROW) : 0;
    using KElem = std::conditional_t<Q8, uint8_t, __nv_bfloat16>;   // element of a cache row
    constexpr int KG = Q8 ? QKROW : DKQ, VG = Q8 ? QVROW : DV;       // its elements per row

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sStage = smem;                                              // stages x STAGE_BYTES
    uint8_t *sDeq = sStage + (size_t)p.stages * STAGE_BYTES;             // Q8: DEQ_BYTES
    uint8_t *sQ = sDeq + DEQ_BYTES;                                      // 16 x KROW
    float *sSP = reinterpret_cast<float *>(sQ + 16 * KROW);              // 4 x 16 x SP_PITCH
    __nv_bfloat16 *sP = reinterpret_cast<__nv_bfloat16 *>(sSP + 4 * 16 * SP_PITCH);  // hi, lo
    float *sAlpha = reinterpret_cast<float *>(sP + 2 * 16 * P_PITCH);    // 16
    float *sL = sAlpha + 16;                                             // 16
    float *sM = sL + 16;                                                 // 16
    int *sTok = reinterpret_cast<int *>(sM + 16);                        // stages x TT
    int *sBlk = sTok + p.stages * TT;                                    // block list

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int split = blockIdx.x, g = blockIdx.y, i = blockIdx.z;
    const bool lead = split == 0 && g == 0;
    const int G = p.G;
    pdl_wait();   // global memory from here on
    const ListInfo L = list_info(p, i, lead && tid == 0);
    const int j0 = split * p.split_tokens;
    int j1 = L.ok ? min(L.len, j0 + p.split_tokens) : 0;
    // p.tail_fold: the splits cover the kept tokens only, and the last split also attends the
    // tail (positions n_blk_tok .. len - 1, at most 15 tokens) as a 16-token tile loaded into
    // the Q buffer at its start, so that no split spends a whole tile on a few tail tokens
    int tail_n = 0;
    if constexpr (FOLD) {
        if (p.tail_fold && L.ok) {
            j1 = max(j0, min(L.n_blk_tok, j0 + p.split_tokens));
            if (split == p.n_split - 1) tail_n = min(L.len - L.n_blk_tok, 16);
        }
    }

    if (j0 >= j1 && tail_n == 0) {  // nothing to attend in this split
        if (p.cluster_merge) {   // it still takes its part in the cluster's merge
            if (tid < 16) {
                sL[tid] = 0.f;
                sM[tid] = -INFINITY;
            }
            cluster_merge<DV>(p, reinterpret_cast<float *>(sStage), sL, sM,
                              reinterpret_cast<float *>(sStage) + 16 * DV, i, g);
            return;
        }
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

    const KElem *Kseq = reinterpret_cast<const KElem *>(p.K) + (int64_t)L.seq * p.k_seq_stride +
                        (int64_t)g * KG;
    const KElem *Vseq = V_IS_K ? Kseq
                               : reinterpret_cast<const KElem *>(p.V) +
                                     (int64_t)L.seq * p.v_seq_stride + (int64_t)g * VG;
    const int n_tiles = (j1 - j0 + TT - 1) / TT;

    // The token (and, paged, the map entry) of this thread's row is looked up one tile ahead
    // of the copy that uses it: tiles are issued in order, so the lookup for tile t + 1 is
    // made while tile t is issued, and its latency overlaps a tile of compute.
    int nx_tok = -1;
    int32_t nx_cell = 0;
    auto lookup = [&](int t) {
        nx_tok = t < n_tiles ? token_at(p, L, j0 + t * TT + tid / TPR, j1, sBlk, jb0) : -1;
        if (p.cell_of && nx_tok >= 0)
            nx_cell = __ldg(p.cell_of + (int64_t)L.seq * p.n_tok_cap + nx_tok);
    };
    lookup(0);

    auto issue_tile = [&](int t) {
        const int st = t % p.stages;
        uint8_t *dstK = sStage + (size_t)st * STAGE_BYTES;
        const int r = tid / TPR, sub = tid % TPR;
        const int tok = nx_tok;
        const int64_t row = p.cell_of && tok >= 0 ? checked_cell(p, nx_cell) : tok;
        lookup(t + 1);
        if (sub == 0) sTok[st * TT + r] = row >= 0 ? tok : -1;
        const KElem *srcK = row >= 0 ? Kseq + row * p.k_tok_stride : Kseq;
        const uint32_t nbytes = row >= 0 ? 16u : 0u;
        if constexpr (Q8) {   // the quantized rows as they are (the tile is dequantized later)
            const uint32_t rowK = smem_u32(dstK) + r * QKROW;
#pragma unroll 4
            for (int c = sub; c < QKROW / 16; c += TPR) cp_async16(rowK + c * 16, srcK + c * 16, nbytes);
            if constexpr (!V_IS_K) {
                const KElem *srcV = row >= 0 ? Vseq + row * p.v_tok_stride : Vseq;
                const uint32_t rowV = smem_u32(dstK + TT * QKROW) + r * QVROW;
#pragma unroll 4
                for (int c = sub; c < QVROW / 16; c += TPR)
                    cp_async16(rowV + c * 16, srcV + c * 16, nbytes);
            }
        } else {
            const uint32_t rowK = smem_u32(dstK) + r * KROW;
#pragma unroll 6
            for (int c = sub; c < KCH; c += TPR) cp_async16(rowK + swz(c, r) * 16, srcK + c * 8, nbytes);
            if constexpr (!V_IS_K) {
                const KElem *srcV = row >= 0 ? Vseq + row * p.v_tok_stride : Vseq;
                const uint32_t rowV = smem_u32(dstK + TT * KROW) + r * VROW;
#pragma unroll 4
                for (int c = sub; c < VCH; c += TPR)
                    cp_async16(rowV + swz(c, r) * 16, srcV + c * 8, nbytes);
            }
        }
    };

    // prologue: stages-1 tiles in flight (behind the Q group)
    for (int t = 0; t < p.stages - 1; ++t) {
        if (t < n_tiles) issue_tile(t);
        cp_async_commit();
    }
    // Q has landed once at most stages-1 younger groups are pending
    cp_async_wait_n(p.stages - 1);
    __syncthreads();
    if constexpr (Q8) {   // Q to binary16 in place: this path's tensor-core operand type
        bool ok = true;
        for (int e = tid; e < 16 * KCH; e += kThreads) {
            const int r = e / KCH, c = e % KCH;
            uint4 *q4 = reinterpret_cast<uint4 *>(sQ + r * KROW + swz(c, r) * 16);
            const uint4 u = *q4;
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            uint32_t h[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xFFFF0000u);
                ok &= fabsf(lo) < 65520.f && fabsf(hi) < 65520.f;
                h[k] = pack_f16(lo, hi);
            }
            *q4 = make_uint4(h[0], h[1], h[2], h[3]);
        }
        if (!ok) set_status(p.status, SFA_DEV_FP16_RANGE);
        __syncthreads();
    }
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
    // the folded tail's rows into the Q buffer (free once every warp holds its fragments), laid
    // out like a tile's rows, as the youngest copy group; rows past the tail are zero
    if constexpr (FOLD) {
        if (tail_n > 0) {
            __syncthreads();
            const uint32_t qs = smem_u32(sQ);
            for (int e = tid; e < 16 * KCH; e += kThreads) {
                const int r = e / KCH, c = e % KCH;
                const int64_t row = r < tail_n ? kv_row(p, L.seq, L.tail0 + r) : -1;
                const KElem *src = row >= 0 ? Kseq + row * p.k_tok_stride + c * 8 : Kseq;
                cp_async16(qs + r * KROW + swz(c, r) * 16, src, row >= 0 ? 16u : 0u);
            }
            cp_async_commit();
        }
    }

    float o[NTV][4];
#pragma unroll
    for (int n = 0; n < NTV; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;   // of row (tid >> 3), kept by its 8 threads

    for (int t = 0; t < n_tiles; ++t) {
        // tile t has landed once at most stages-2 younger groups are pending
        cp_async_wait_n(p.stages - 2 + (FOLD && tail_n > 0 && t <= p.stages - 2 ? 1 : 0));
        __syncthreads();
        if (t + p.stages - 1 < n_tiles) issue_tile(t + p.stages - 1);
        cp_async_commit();

        const int st = t % p.stages;
        if constexpr (Q8) {
            // tile t from its q8_0 rows into the binary16 tile: each warp converts the K
            // columns of its own head-dim slice (all it reads for S) and, with a separate V,
            // the V columns of its value-dim slice; the block barrier after the S partials
            // publishes the whole tile before any warp reads V columns of another's slice
            const uint8_t *stg = sStage + (size_t)st * STAGE_BYTES;
            bool ok = dequant_tile<DKQ, QKROW, TT, DKQ / 32>(stg, sDeq, warp * (DKQ / 32), lane, 32);
            if constexpr (!V_IS_K)
                ok &= dequant_tile<DV, QVROW, TT, DV / 32>(stg + TT * QKROW, sDeq + TT * KROW,
                                                            warp * (DV / 32), lane, 32);
            if (!ok) set_status(p.status, SFA_DEV_FP16_RANGE);
            __syncwarp();
        }
        const uint32_t kbase = Q8 ? smem_u32(sDeq) : smem_u32(sStage + (size_t)st * STAGE_BYTES);
        const uint32_t vbase = V_IS_K ? kbase : kbase + TT * KROW;

        // ---- S partial over this warp's head-dim slice
        float acc[TT / 8][4];
#pragma unroll
        for (int n = 0; n < TT / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
        for (int np = 0; np < TT / 16; ++np) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int kg = warp * KS + ks;
                const int mi = lane >> 3, r8 = lane & 7;
                const int n = np * 16 + (mi >> 1) * 8 + r8;
                const int c = kg * 2 + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + n * KROW + swz(c, n) * 16, b0, b1, b2, b3);
                mma16816<Q8>(acc[2 * np], qa[ks], b0, b1);
                mma16816<Q8>(acc[2 * np + 1], qa[ks], b2, b3);
            }
        }
        float *sp = sSP + warp * 16 * SP_PITCH;
#pragma unroll
        for (int n = 0; n < TT / 8; ++n) {
            *reinterpret_cast<float2 *>(sp + gq * SP_PITCH + n * 8 + 2 * tq) = make_float2(acc[n][0], acc[n][1]);
            *reinterpret_cast<float2 *>(sp + (gq + 8) * SP_PITCH + n * 8 + 2 * tq) = make_float2(acc[n][2], acc[n][3]);
        }
        __syncthreads();

        // ---- online softmax: thread -> row tid/8, columns SPT*(tid%8) .. +SPT-1
        {
            const int row = tid >> 3, c0 = (tid & 7) * SPT;
            float s[SPT];
#pragma unroll
            for (int e = 0; e < SPT; ++e) s[e] = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float *src = sSP + (w * 16 + row) * SP_PITCH + c0;
                if constexpr (SPT == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(src);
                    s[0] += v.x; s[1] += v.y; s[2] += v.z; s[3] += v.w;
                } else {
                    const float2 v = *reinterpret_cast<const float2 *>(src);
                    s[0] += v.x; s[1] += v.y;
                }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int e = 0; e < SPT; ++e) {
                s[e] = sTok[st * TT + c0 + e] >= 0 ? s[e] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[e]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
            float ph[SPT], pl[SPT], rs = 0.f;
#pragma unroll
            for (int e = 0; e < SPT; ++e) {
                const float pe = m_new == -INFINITY ? 0.f : exp2f(s[e] - m_new);
                ph[e] = round16<Q8>(pe);
                pl[e] = pe - ph[e];
                rs += pe;
            }
            rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 1);
            rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 2);
            rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 4);
            l_run = l_run * alpha + rs;
            m_run = m_new;
            if constexpr (SPT == 4) {
                *reinterpret_cast<uint2 *>(sP + row * P_PITCH + c0) =
                    make_uint2(pack16<Q8>(ph[0], ph[1]), pack16<Q8>(ph[2], ph[3]));
                *reinterpret_cast<uint2 *>(sP + (16 + row) * P_PITCH + c0) =
                    make_uint2(pack16<Q8>(pl[0], pl[1]), pack16<Q8>(pl[2], pl[3]));
            } else {
                *reinterpret_cast<uint32_t *>(sP + row * P_PITCH + c0) = pack16<Q8>(ph[0], ph[1]);
                *reinterpret_cast<uint32_t *>(sP + (16 + row) * P_PITCH + c0) = pack16<Q8>(pl[0], pl[1]);
            }
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
            for (int ks = 0; ks < TT / 16; ++ks) {
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
                    mma16816<Q8>(o[2 * np], pa, b0, b1);
                    mma16816<Q8>(o[2 * np + 1], pa, b2, b3);
                    mma16816<Q8>(o[2 * np], pb, b0, b1);
                    mma16816<Q8>(o[2 * np + 1], pb, b2, b3);
                }
            }
        }
    }
    if constexpr (FOLD) {
        if (tail_n > 0) {   // the folded tail, its rows long since in the Q buffer
        // The loop's tile step for NT tokens from K rows at kbase and V rows at vbase (S over
        // this warp's head-dim slice, the online softmax, O += P V over its value-dim slice;
        // tokv[c] < 0 leaves column c out), here for the 16-token tail tile.  The loop keeps
        // its own copy: routing it through this lambda made the plain kernel's dense prefill
        // 1.3% slower (decode_32x131072 unchanged).
        auto tile_step = [&](auto nt, const uint32_t kbase, const uint32_t vbase, const int *tokv) {
            constexpr int NT = decltype(nt)::value;
            constexpr int NSPT = NT / 8;   // softmax columns per thread
            // ---- S partial over this warp's head-dim slice
            float acc[NT / 8][4];
    #pragma unroll
            for (int n = 0; n < NT / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    #pragma unroll
            for (int np = 0; np < NT / 16; ++np) {
    #pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int kg = warp * KS + ks;
                    const int mi = lane >> 3, r8 = lane & 7;
                    const int n = np * 16 + (mi >> 1) * 8 + r8;
                    const int c = kg * 2 + (mi & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kbase + n * KROW + swz(c, n) * 16, b0, b1, b2, b3);
                    mma16816<Q8>(acc[2 * np], qa[ks], b0, b1);
                    mma16816<Q8>(acc[2 * np + 1], qa[ks], b2, b3);
                }
            }
            float *sp = sSP + warp * 16 * SP_PITCH;
    #pragma unroll
            for (int n = 0; n < NT / 8; ++n) {
                *reinterpret_cast<float2 *>(sp + gq * SP_PITCH + n * 8 + 2 * tq) = make_float2(acc[n][0], acc[n][1]);
                *reinterpret_cast<float2 *>(sp + (gq + 8) * SP_PITCH + n * 8 + 2 * tq) = make_float2(acc[n][2], acc[n][3]);
            }
            __syncthreads();

            // ---- online softmax: thread -> row tid/8, columns NSPT*(tid%8) .. +NSPT-1
            {
                const int row = tid >> 3, c0 = (tid & 7) * NSPT;
                float s[NSPT];
    #pragma unroll
                for (int e = 0; e < NSPT; ++e) s[e] = 0.f;
    #pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float *src = sSP + (w * 16 + row) * SP_PITCH + c0;
                    if constexpr (NSPT == 4) {
                        const float4 v = *reinterpret_cast<const float4 *>(src);
                        s[0] += v.x; s[1] += v.y; s[2] += v.z; s[3] += v.w;
                    } else {
                        const float2 v = *reinterpret_cast<const float2 *>(src);
                        s[0] += v.x; s[1] += v.y;
                    }
                }
                float mx = -INFINITY;
    #pragma unroll
                for (int e = 0; e < NSPT; ++e) {
                    s[e] = tokv[c0 + e] >= 0 ? s[e] * p.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, s[e]);
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
                const float m_new = fmaxf(m_run, mx);
                const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
                float ph[NSPT], pl[NSPT], rs = 0.f;
    #pragma unroll
                for (int e = 0; e < NSPT; ++e) {
                    const float pe = m_new == -INFINITY ? 0.f : exp2f(s[e] - m_new);
                    ph[e] = round16<Q8>(pe);
                    pl[e] = pe - ph[e];
                    rs += pe;
                }
                rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 1);
                rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 2);
                rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 4);
                l_run = l_run * alpha + rs;
                m_run = m_new;
                if constexpr (NSPT == 4) {
                    *reinterpret_cast<uint2 *>(sP + row * P_PITCH + c0) =
                        make_uint2(pack16<Q8>(ph[0], ph[1]), pack16<Q8>(ph[2], ph[3]));
                    *reinterpret_cast<uint2 *>(sP + (16 + row) * P_PITCH + c0) =
                        make_uint2(pack16<Q8>(pl[0], pl[1]), pack16<Q8>(pl[2], pl[3]));
                } else {
                    *reinterpret_cast<uint32_t *>(sP + row * P_PITCH + c0) = pack16<Q8>(ph[0], ph[1]);
                    *reinterpret_cast<uint32_t *>(sP + (16 + row) * P_PITCH + c0) = pack16<Q8>(pl[0], pl[1]);
                }
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
                for (int ks = 0; ks < NT / 16; ++ks) {
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
                        mma16816<Q8>(o[2 * np], pa, b0, b1);
                        mma16816<Q8>(o[2 * np + 1], pa, b2, b3);
                        mma16816<Q8>(o[2 * np], pb, b0, b1);
                        mma16816<Q8>(o[2 * np + 1], pb, b2, b3);
                    }
                }
            }
        };

            cp_async_wait<0>();
            if (tid < 16) sTok[tid] = tid < tail_n ? 0 : -1;
            __syncthreads();
            tile_step(std::integral_constant<int, 16>{}, smem_u32(sQ), smem_u32(sQ), sTok);
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
    if (p.cluster_merge) {   // the unnormalised rows into this CTA's (now idle) stage memory
        float *sPart = reinterpret_cast<float *>(sStage);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int row = gq + half * 8;
            if (row >= G) continue;
#pragma unroll
            for (int n = 0; n < NTV; ++n)
                *reinterpret_cast<float2 *>(sPart + row * DV + dv0 + n * 8 + 2 * tq) =
                    make_float2(o[n][2 * half], o[n][2 * half + 1]);
        }
        cluster_merge<DV>(p, sPart, sL, sM, sPart + 16 * DV, i, g);
        return;
    }
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

template <int DKQ, int DV, bool V_IS_K, int TT>
__global__ void __launch_bounds__(kThreads, 1) attend_bf16_kernel(const AttnParams p) {
    attend_mma_body<DKQ, DV, V_IS_K, false, TT>(p);
}
template <int DKQ, int DV, bool V_IS_K, int TT>
__global__ void __launch_bounds__(kThreads, 1) attend_q8_kernel(const AttnParams p) {
    attend_mma_body<DKQ, DV, V_IS_K, true, TT>(p);
}
// The bf16 kernel with the list's tail folded into the last split (AttnParams::tail_fold):
// its own instance, so that the other plans keep the plain kernel's code and registers.
template <int DKQ, int DV>
__global__ void __launch_bounds__(kThreads, 1) attend_bf16_fold_kernel(const AttnParams p) {
    attend_mma_body<DKQ, DV, true, false, 32, true>(p);
}

// ---------------------------------------------------------------------------------------
// tcgen05 kernel for the MLA / 512-wide heads (DKQ 576 or 512, DV 512).  One CTA = one query x
// one KV head x one split of its list; the list is cut into 32-token tiles that stream
// through a ring of NR stages (NR = 4, or 2 when V is separate and the stages are twice as
// large).  Within each 64-wide slab of the head dim the ring's rows are contiguous (tile t
// sits at rows 32 * (t % NR) ...), so one M = 128 MMA over the ring scores every tile in it
// at once.  Warp roles (9 warps):
//   warps 5-8   producers (one per SM sub-partition): Q once (cp.async), then 8 rows of
//               every tile each, as 4-row groups: a group of 4 consecutive tokens (a kept
//               block of cr = 4, half of one of cr = 8, the tail, the dense case) is one TMA
//               box per 64-wide slab, landing 128-byte-swizzled in the K-major layout with
//               its bytes counted on the stage's barrier; any other group (the ragged end of
//               the list, a dropped block) is copied row by row with zero-filling cp.async,
//               waited for and fenced into the async proxy by the producer itself;
//   warp 4      tensor-memory owner and single-thread MMA issuer.  It groups the landed,
//               not yet scored tiles into a batch (two at least, unless the list ends;
//               the whole ring at most) and issues
//                 S^T[128 ring rows x 16 heads] = ring (A, K-major) x Q^T (B, K-major),
//               then, once the batch's P is ready, for each 128-wide slice of DV
//                 O^T[128 dv x 32] = V^T (A, MN-major; the K rows when V is the first 512
//                                    dims of K) x [P_hi | P_lo]^T (B, K-major, N = 32),
//               P carried as bf16 hi + lo in one MMA and the halves summed on read-out;
//               the stages of a batch are released when its PV MMAs complete;
//   warps 0-3   softmax and correction.  Warp s reads the S rows of ring stage s (TMEM lanes
//               32s ..); per-head max and sum are reduced across the batch through shared
//               memory and P^T hi/lo is written at the tokens' ring positions.  The same
//               warps own the value dims 32s .. of every 128-wide slice of O (TMEM lanes of
//               the PV result) and keep O in registers: after the softmax of batch b they
//               fold in batch b - 1 (O = O * alpha + P_hi V + P_lo V) while the tensor cores
//               run the PV of batch b; O is normalised at the end (or written as a split
//               partial).
// S, P and O are double-buffered per batch, so the MMAs of batch b + 1 overlap the softmax
// and correction of batch b.  Staging the ring through TMA (the async proxy) keeps generic
// copies out of flight, so the proxy fence that publishes P stays cheap.  Every wait is
// bounded.
namespace tc {
constexpr int kThreads = 288;
constexpr int kMmaWarp = 4, kProdWarp0 = 5;
constexpr int kProdThreads = 128;
constexpr int kTT = 32;          // tokens per tile (ring stage)
constexpr int kBatchMin = 2;     // tiles an S / PV batch waits for (at most the whole ring)
constexpr int kTmemCols = 512;   // S: 2 x 16, O: 2 x (4 x 32); one CTA per SM
}  // namespace tc

template <int DKQ, int DV, bool V_IS_K>
struct TcLayout {
    static constexpr int kNR = V_IS_K ? 4 : 2;                // ring stages
    static constexpr int kRingRows = kNR * tc::kTT;
    static constexpr int kSlabK = DKQ / 64;                   // 64-wide slabs of K
    static constexpr int kSlabV = V_IS_K ? 0 : DV / 64;       // separate V slabs
    static constexpr int kSlabBytes = kRingRows * 128;        // ring rows x 128 B
    static constexpr int kRingBytes = (kSlabK + kSlabV) * kSlabBytes;
    static constexpr int kQBytes = kSlabK * 16 * 128;         // B operand: 16 rows per slab
    static constexpr int kPRegion = 32 * 128;                 // 32 rows (hi, lo) x 64 tokens
    static constexpr int kPBuf = ((kRingRows + 63) / 64) * kPRegion;
    // the S MMA reads 128 rows from each slab start; past the ring they fall in Q and P
    static_assert(kQBytes + 2 * kPBuf >= (128 - kRingRows) * 128, "over-read stays in the CTA");
    static constexpr int kOffRing = 0;
    static constexpr int kOffQ = kRingBytes;
    static constexpr int kOffP = kOffQ + kQBytes;                         // [2][kPBuf]
    static constexpr int kOffRed = kOffP + 2 * kPBuf;                     // max, sum [4][16]
    static constexpr int kOffAlpha = kOffRed + 2 * 4 * 16 * 4;            // [2][16]
    static constexpr int kOffL = kOffAlpha + 2 * 16 * 4;                  // running sums [16]
    static constexpr int kOffM = kOffL + 16 * 4;                          // running maxima [2][16]
    static constexpr int kOffBat = kOffM + 2 * 16 * 4;                    // [2] x (t0, n)
    static constexpr int kOffBar = kOffBat + 16;                          // mbarriers
    static constexpr int kNumBars = 2 * kNR + 2 * 7 + 3;
    static constexpr int kOffTok = kOffBar + kNumBars * 8 + 16;           // [ring rows]
    static constexpr int kOffBlk = kOffTok + kRingRows * 4;
    static constexpr size_t bytes(int blk_list) { return 1024 + kOffBlk + (size_t)blk_list * 4 + 16; }
};

// Reduces v[0..15] (one value per head) over the 32 lanes with op: afterwards lanes 2h and
// 2h + 1 hold the reduction of head h.  16 shuffles (a transposing butterfly).
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(float (&v)[16], int lane) {
    auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
    float a8[8], a4[4], a2[2];
    const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float keep = u16 ? v[i + 8] : v[i], send = u16 ? v[i] : v[i + 8];
        a8[i] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 16));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float keep = u8 ? a8[i + 4] : a8[i], send = u8 ? a8[i] : a8[i + 4];
        a4[i] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 8));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float keep = u4 ? a4[i + 2] : a4[i], send = u4 ? a4[i] : a4[i + 2];
        a2[i] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 4));
    }
    const float keep = u2 ? a2[1] : a2[0], send = u2 ? a2[0] : a2[1];
    const float a1 = op(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 2));
    return op(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, 1));
}

// O = O * alpha + (P_hi V + P_lo V) of batch bb, whose PV result sits in O buffer bb & 1
// (32 columns per 128-wide slice of DV: the hi half, then the lo half).
template <int DV>
__device__ __forceinline__ bool tc_fold(float (&o)[DV / 128][16], const float *al, int bb,
                                        uint64_t *o_full, uint64_t *o_empty, uint32_t tO,
                                        uint32_t lane_addr, int lane, uint64_t deadline) {
    const int x = bb & 1;
    if (!mbar_wait(&o_full[x], (bb >> 1) & 1, deadline)) return false;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const float a = al[c];
#pragma unroll
        for (int mt = 0; mt < DV / 128; ++mt) o[mt][c] *= a;
    }
#pragma unroll
    for (int mt = 0; mt < DV / 128; ++mt) {
        uint32_t r[16];
        tmem_ld16(tO + x * 128 + mt * 32 + lane_addr, r);          // P_hi V
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c) o[mt][c] += __uint_as_float(r[c]);
        tmem_ld16(tO + x * 128 + mt * 32 + 16 + lane_addr, r);     // P_lo V
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c) o[mt][c] += __uint_as_float(r[c]);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&o_empty[x]);
    return true;
}

template <int DKQ, int DV, bool V_IS_K>
__global__ void __launch_bounds__(tc::kThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
    using Lay = TcLayout<DKQ, DV, V_IS_K>;
    constexpr int NR = Lay::kNR, TT = tc::kTT;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-aligned base, derived by pointer arithmetic so accesses stay shared-space ones
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sRing = smem + Lay::kOffRing;
    uint8_t *sQ = smem + Lay::kOffQ;
    uint8_t *sP = smem + Lay::kOffP;
    float *sMax = reinterpret_cast<float *>(smem + Lay::kOffRed);   // [4 warps][16 heads]
    float *sSum = sMax + 64;
    float *sAlpha = reinterpret_cast<float *>(smem + Lay::kOffAlpha);  // per batch buffer
    float *sL = reinterpret_cast<float *>(smem + Lay::kOffL);          // running sums per head
    float *sM = reinterpret_cast<float *>(smem + Lay::kOffM);          // running maxima; after
                                                                       // batch b in [b & 1]
    int *sBat = reinterpret_cast<int *>(smem + Lay::kOffBat);        // [2] x (first tile, n)
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kOffBar);
    uint64_t *full = bars, *empty = bars + NR;
    uint64_t *bat_ready = bars + 2 * NR, *s_full = bat_ready + 2, *s_empty = s_full + 2;
    uint64_t *p_full = s_empty + 2, *p_empty = p_full + 2;
    uint64_t *o_full = p_empty + 2, *o_empty = o_full + 2;
    uint64_t *q_ready = o_empty + 2, *drain = q_ready + 1;
    uint64_t *soft_bar = q_ready + 2;   // the softmax threads' own (bounded) barrier
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Lay::kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *sTok = reinterpret_cast<int *>(smem + Lay::kOffTok);
    int *sBlk = reinterpret_cast<int *>(smem + Lay::kOffBlk);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, g = blockIdx.y, i = blockIdx.z;
    pdl_wait();   // global memory from here on
    const ListInfo L = list_info(p, i, split == 0 && g == 0 && tid == 0);
    const int j0 = split * p.split_tokens;
    const int j1 = L.ok ? min(L.len, j0 + p.split_tokens) : 0;
    const int G = p.G;

    if (j0 >= j1) {  // nothing to attend in this split
        for (int e = tid; e < G * DV; e += tc::kThreads) {
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
    const int n_tiles = (j1 - j0 + TT - 1) / TT;
    const uint64_t deadline = global_timer_ns() + kWaitLimitNs;

    // ------------------------------------------------------------------ set-up
    if (tid == tc::kProdWarp0 * 32) {
        prefetch_tensormap(&kmap);
        if constexpr (!V_IS_K) prefetch_tensormap(&vmap);
    }
    if (tid == 0) {
        for (int s = 0; s < NR; ++s) {
            mbar_init(&full[s], tc::kProdThreads / 32);   // one expect-tx arrival per warp
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bat_ready[b], 1);
            mbar_init(&s_full[b], 1);
            mbar_init(&s_empty[b], 4);      // the four softmax warps
            mbar_init(&p_full[b], 4);
            mbar_init(&p_empty[b], 1);      // the PV commit
            mbar_init(&o_full[b], 1);
            mbar_init(&o_empty[b], 4);
        }
        mbar_init(q_ready, 128);   // the softmax warps load Q
        mbar_init(drain, 1);
        mbar_init(soft_bar, 128);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == tc::kMmaWarp) {
        tmem_alloc(tmem_slot, tc::kTmemCols);
        tmem_relinquish();
    }
    const int jb0 = load_block_list(p, i, L, j0, j1, sBlk, g == 0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + 32;  // S: cols [0, 32), O: cols [32, 288)

    auto fail = [&]() {
        set_status(p.status, SFA_DEV_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp >= tc::kProdWarp0) {
        // ------------------------------------------------------------ producers
        constexpr int KCH = DKQ / 8, VCH = DV / 8;
        const __nv_bfloat16 *Kseq = reinterpret_cast<const __nv_bfloat16 *>(p.K) +
                                    (int64_t)L.seq * p.k_seq_stride + (int64_t)g * DKQ;
        const __nv_bfloat16 *Vseq = V_IS_K ? Kseq
                                           : reinterpret_cast<const __nv_bfloat16 *>(p.V) +
                                                 (int64_t)L.seq * p.v_seq_stride + (int64_t)g * DV;
        // warp pw owns tile rows 8pw .. 8pw + 7: two 4-row groups
        const int pw = warp - tc::kProdWarp0;
        constexpr int NSL = Lay::kSlabK + Lay::kSlabV;
        static_assert(2 * NSL <= 32, "one box per lane");
        static_assert((4 * KCH) % 32 == 0 && (4 * VCH) % 32 == 0, "uniform row-copy loops");
        const int64_t zseq = (int64_t)L.seq * p.n_tok_cap;   // TMA row of the sequence's token 0
        const uint32_t ring = smem_u32(sRing);
        for (int t = 0; t < n_tiles; ++t) {
            const int st = t % NR;
            if (*abort_flag) break;
            if (!mbar_wait(&empty[st], ((t / NR) & 1) ^ 1, deadline)) { fail(); break; }
            const int row0 = st * TT + pw * 8;                  // ring row of this warp's row 0
            int tok_l = -1;
            if (lane < 8) {
                tok_l = token_at(p, L, j0 + t * TT + pw * 8 + lane, j1, sBlk, jb0);
                sTok[row0 + lane] = tok_l;
            }
            int tk[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) tk[k] = __shfl_sync(0xFFFFFFFFu, tok_l, k);
            bool box[2];
#pragma unroll
            for (int gi = 0; gi < 2; ++gi)
                box[gi] = tk[4 * gi] >= 0 && tk[4 * gi + 1] == tk[4 * gi] + 1 &&
                          tk[4 * gi + 2] == tk[4 * gi] + 2 && tk[4 * gi + 3] == tk[4 * gi] + 3;
            if (!box[0] || !box[1]) {
                // row-by-row copies (zero rows for masked positions), landed and fenced here
#pragma unroll
                for (int gi = 0; gi < 2; ++gi) {
                    if (box[gi]) continue;
#pragma unroll 1
                    for (int e = lane; e < 4 * KCH; e += 32) {
                        const int k = e / KCH, c = e - k * KCH, r = row0 + 4 * gi + k;
                        const int tok = tk[4 * gi + k];
                        cp_async16(ring + (c >> 3) * Lay::kSlabBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4),
                                   tok >= 0 ? Kseq + (int64_t)tok * p.k_tok_stride + c * 8 : Kseq,
                                   tok >= 0 ? 16u : 0u);
                    }
                    if constexpr (!V_IS_K) {
                        const uint32_t v0 = ring + Lay::kSlabK * Lay::kSlabBytes;
#pragma unroll 1
                        for (int e = lane; e < 4 * VCH; e += 32) {
                            const int k = e / VCH, c = e - k * VCH, r = row0 + 4 * gi + k;
                            const int tok = tk[4 * gi + k];
                            cp_async16(v0 + (c >> 3) * Lay::kSlabBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4),
                                       tok >= 0 ? Vseq + (int64_t)tok * p.v_tok_stride + c * 8 : Vseq,
                                       tok >= 0 ? 16u : 0u);
                        }
                    }
                }
                cp_async_commit();
                cp_async_wait<0>();
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive_expect_tx(&full[st], (uint32_t)((box[0] ? 1 : 0) + (box[1] ? 1 : 0)) * NSL * 512u);
            __syncwarp();
            if (lane < 2 * NSL) {   // lane -> (group, slab): one 4-row x 128-byte box each
                const int gi = lane / NSL, sl = lane - gi * NSL;
                if (box[gi]) {
                    const bool is_v = !V_IS_K && sl >= Lay::kSlabK;
                    tma_load_3d(sRing + sl * Lay::kSlabBytes + (row0 + 4 * gi) * 128,
                                is_v ? &vmap : &kmap, (is_v ? sl - Lay::kSlabK : sl) * 64, g,
                                (int32_t)(zseq + tk[4 * gi]), &full[st]);
                }
            }
        }
    } else if (warp == tc::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(128, 16);
            const uint32_t idPV = idesc_bf16_f32(128, 32) | (1u << 15);   // A (V^T) MN-major
            const uint32_t ring = smem_u32(sRing), q0 = smem_u32(sQ), p0 = smem_u32(sP);
            const uint64_t aS = sw128_desc(ring, 16, 1024);
            const uint64_t bq = sw128_desc(q0, 16, 1024);
            const uint32_t vbase = ring + (V_IS_K ? 0 : Lay::kSlabK * Lay::kSlabBytes);
            // V^T (MN-major): 64-dim atoms one slab apart, 8-token groups 1024 B apart
            const uint64_t av0 = sw128_desc(vbase, Lay::kSlabBytes, 1024);
            const uint64_t bp0 = sw128_desc(p0, 16, 1024);
            static_assert((NR & (NR - 1)) == 0, "ring size is a power of two");
            bool ok = mbar_wait(q_ready, 0, deadline);
            int t_next = 0, nb = 0, np = 0;      // next tile to score, batches formed, PV'd
            int bt0[2] = {0, 0}, btn[2] = {0, 0};
            // PV of the oldest batch whose P is ready (it releases stages); also called
            // between the chunks of an S issue so that PV never waits behind a whole S
            auto try_pv = [&]() -> bool {
                if (np >= nb) return false;
                const int x = np & 1;
                if (!mbar_try_wait(smem_u32(&p_full[x]), (np >> 1) & 1) ||
                    !mbar_try_wait(smem_u32(&o_empty[x]), ((np >> 1) & 1) ^ 1))
                    return false;
                tc_fence_after();
                // u outer, the slices of DV inner: the first tile starts each slice
#pragma unroll 1
                for (int u = 0; u < btn[x]; ++u) {
                    const int st = (bt0[x] + u) & (NR - 1);
                    const uint64_t a_u = av0 + (uint64_t)((st * TT * 128) >> 4);
                    const uint64_t b_u = bp0 + (uint64_t)((x * Lay::kPBuf + (st >> 1) * Lay::kPRegion +
                                                           (st & 1) * 64) >> 4);
#pragma unroll
                    for (int mt = 0; mt < DV / 128; ++mt) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf)
                            tc_mma_bf16(tO + x * 128 + mt * 32,
                                        a_u + (uint64_t)((2 * mt * Lay::kSlabBytes + hf * 2048) >> 4),
                                        b_u + (uint64_t)(hf * 2), idPV, (u > 0 || hf > 0) ? 1u : 0u);
                    }
                }
                tc_commit(&o_full[x]);
                tc_commit(&p_empty[x]);
                for (int u = 0; u < btn[x]; ++u) tc_commit(&empty[(bt0[x] + u) & (NR - 1)]);
                ++np;
                return true;
            };
            uint32_t spin = 0;
            while (ok && (t_next < n_tiles || np < nb)) {
                if (*abort_flag) { ok = false; break; }
                bool progressed = try_pv();
                // S for the landed, unscored tiles (a batch), when an S buffer is free
                if (t_next < n_tiles && nb - np < 2) {
                    const int x = nb & 1;
                    // at least kBatchMin landed tiles (fewer only at the end), then every
                    // further landed one up to the whole ring: S costs the same for all of them
                    const int n_min = min(tc::kBatchMin, n_tiles - t_next);
                    bool ready = mbar_try_wait(smem_u32(&s_empty[x]), ((nb >> 1) & 1) ^ 1);
                    for (int u = 0; ready && u < n_min; ++u)
                        ready = mbar_try_wait(smem_u32(&full[(t_next + u) % NR]), ((t_next + u) / NR) & 1);
                    if (ready) {
                        int n = n_min;
                        while (n < NR && t_next + n < n_tiles &&
                               mbar_try_wait(smem_u32(&full[(t_next + n) % NR]), ((t_next + n) / NR) & 1))
                            ++n;
                        bt0[x] = t_next;
                        btn[x] = n;
                        sBat[2 * x] = t_next;
                        sBat[2 * x + 1] = n;
                        mbar_arrive(&bat_ready[x]);
                        tc_fence_after();
#pragma unroll 1
                        for (int sl = 0; sl < Lay::kSlabK; ++sl) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc_mma_bf16(tS + x * 16, aS + (uint64_t)((sl * Lay::kSlabBytes + kk * 32) >> 4),
                                            bq + (uint64_t)((sl * 2048 + kk * 32) >> 4), idS,
                                            (sl > 0 || kk > 0) ? 1u : 0u);
                            if (sl % 3 == 2 && sl + 1 < Lay::kSlabK) try_pv();   // PV cuts in
                        }
                        tc_commit(&s_full[x]);
                        t_next += n;
                        ++nb;
                        progressed = true;
                    }
                }
                if (!progressed && (++spin & 63u) == 0 && global_timer_ns() > deadline) ok = false;
            }
            if (!ok) fail();
        }
    } else {
        // ------------------------------------------------- softmax + correction (4 warps)
        {   // Q^T operand: 16 rows (heads; rows >= G zero) x DKQ, one slab per 64 dims
            constexpr int KCH = DKQ / 8;
            const __nv_bfloat16 *Qg = reinterpret_cast<const __nv_bfloat16 *>(p.Q) +
                                      ((int64_t)i * p.h_q + (int64_t)g * G) * DKQ;
            const uint32_t qs = smem_u32(sQ);
            for (int e = tid; e < 16 * KCH; e += 128) {
                const int r = e / KCH, c = e % KCH;
                const bool live = r < G;
                cp_async16(qs + (c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4),
                           live ? Qg + (int64_t)r * DKQ + c * 8 : Qg, live ? 16u : 0u);
            }
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(q_ready);
        }
        const int sq = warp;                       // ring stage / TMEM lane quarter
        const int rrow = sq * TT + lane;           // ring row = TMEM lane of this thread
        const uint32_t lane_addr = (uint32_t)(sq * 32) << 16;
        // the running maxima and sums live in sM / sL; lanes 0-15 of warp 0 update them
        float o[DV / 128][16];
        if (tid < 16) {
            sL[tid] = 0.f;
            sM[16 + tid] = -INFINITY;   // "after batch -1"
        }
#pragma unroll
        for (int mt = 0; mt < DV / 128; ++mt)
#pragma unroll
            for (int c = 0; c < 16; ++c) o[mt][c] = 0.f;
        uint32_t soft_phase = 0;
        auto soft_sync = [&]() -> bool {   // the 128 threads of warps 0-3, bounded
            mbar_arrive(soft_bar);
            const bool done = mbar_wait(soft_bar, soft_phase, deadline);
            soft_phase ^= 1;
            return done;
        };
        bool ok = true;
        int done_tiles = 0, b = 0;
        for (; done_tiles < n_tiles; ++b) {
            const int x = b & 1;
            const uint32_t par = (b >> 1) & 1;
            if (*abort_flag) { ok = false; break; }
            if (!mbar_wait(&bat_ready[x], par, deadline)) { ok = false; break; }
            const int t0 = sBat[2 * x], n = sBat[2 * x + 1];
            const int u = ((sq - t0 % NR) + NR) % NR;      // this stage's place in the batch
            const bool part = sq < NR && u < n;
            const int tq = t0 + u;
            if (!mbar_wait(&s_full[x], par, deadline) ||
                (part && !mbar_wait(&full[sq], (tq / NR) & 1, deadline))) { ok = false; break; }
            tc_fence_after();
            float s[16];
            if (part) {
                uint32_t r[16];
                tmem_ld16(tS + x * 16 + lane_addr, r);
                tmem_ld_wait();
                const bool valid = sTok[rrow] >= 0;
#pragma unroll
                for (int h = 0; h < 16; ++h) s[h] = valid ? __uint_as_float(r[h]) * p.scale_log2 : -INFINITY;
            } else {
#pragma unroll
                for (int h = 0; h < 16; ++h) s[h] = -INFINITY;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[x]);
            {
                float v[16];
#pragma unroll
                for (int h = 0; h < 16; ++h) v[h] = s[h];
                const float mx = warp_reduce16<true>(v, lane);
                if ((lane & 1) == 0) sMax[sq * 16 + (lane >> 1)] = mx;
            }
            if (!soft_sync()) { ok = false; break; }
            // P^T (ring row rrow) into buffer x once the PV two batches back is done with it
            if (!mbar_wait(&p_empty[x], par ^ 1, deadline)) { ok = false; break; }
            // new running max mn; l and (through sAlpha, at the fold) O are rescaled by alpha
            uint8_t *pb = sP + x * Lay::kPBuf + (rrow >> 6) * Lay::kPRegion;
            const int col = rrow & 63;
            const float *mold = sM + (x ^ 1) * 16;
            // every shared load first (the P stores below could alias them for the compiler)
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                const float4 m4 = make_float4(sMax[h], sMax[16 + h], sMax[32 + h], sMax[48 + h]);
                const float mn = fmaxf(mold[h], fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w)));
                s[h] = (!part || mn == -INFINITY) ? -INFINITY : s[h] - mn;   // exponent of p
            }
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                const float pe = exp2f(s[h]);
                s[h] = pe;
                if (part) {
                    const __nv_bfloat16 hi = __float2bfloat16_rn(pe);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(pe - __bfloat162float(hi));
                    const int off = ((((col >> 3) ^ (h & 7))) << 4) + (col & 7) * 2;
                    *reinterpret_cast<__nv_bfloat16 *>(pb + h * 128 + off) = hi;
                    *reinterpret_cast<__nv_bfloat16 *>(pb + (16 + h) * 128 + off) = lo;
                }
            }
            {
                const float rs = warp_reduce16<false>(s, lane);
                if ((lane & 1) == 0) sSum[sq * 16 + (lane >> 1)] = rs;
            }
            if (warp == 0 && lane < 16) {   // running max / alpha / rescaled sum of head lane
                const int h = lane;
                const float mx = fmaxf(fmaxf(sMax[h], sMax[16 + h]), fmaxf(sMax[32 + h], sMax[48 + h]));
                const float mo = mold[h], mn = fmaxf(mo, mx);
                const float alpha = mn == -INFINITY ? 1.f : exp2f(mo - mn);
                sAlpha[x * 16 + h] = alpha;
                sL[h] *= alpha;
                sM[x * 16 + h] = mn;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
            // while the PV of this batch runs: fold the previous batch into O
            if (b > 0 && !tc_fold<DV>(o, sAlpha + ((b - 1) & 1) * 16, b - 1, o_full, o_empty, tO,
                                      lane_addr, lane, deadline)) {
                ok = false;
                break;
            }
            if (!soft_sync()) { ok = false; break; }
            if (warp == 0 && lane < 16)
                sL[lane] += (sSum[lane] + sSum[16 + lane]) + (sSum[32 + lane] + sSum[48 + lane]);
            done_tiles = t0 + n;
        }
        if (ok && b > 0 &&
            !tc_fold<DV>(o, sAlpha + ((b - 1) & 1) * 16, b - 1, o_full, o_empty, tO, lane_addr, lane, deadline))
            ok = false;
        if (ok && !soft_sync()) ok = false;   // thread 0's last update of sL is visible
        if (!ok) {
            fail();
        } else {
            const int dv_base = sq * 32 + lane;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                if (c >= G) break;
                const int h = g * G + c;
                const float m = sM[((b - 1) & 1) * 16 + c], l = sL[c];
                if (p.n_split == 1) {
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    float *dst = p.O + ((int64_t)i * p.h_q + h) * DV + dv_base;
#pragma unroll
                    for (int mt = 0; mt < DV / 128; ++mt) dst[mt * 128] = o[mt][c] * inv;
                    if (p.lse && dv_base == 0)
                        p.lse[(int64_t)i * p.h_q + h] = l > 0.f ? (m + log2f(l)) / kLog2e : -INFINITY;
                } else {
                    const int64_t base = (((int64_t)i * p.h_kv + g) * p.n_split + split) * G + c;
                    float *dst = p.part_o + base * DV + dv_base;
#pragma unroll
                    for (int mt = 0; mt < DV / 128; ++mt) dst[mt * 128] = o[mt][c];
                    if (dv_base == 0) {
                        p.part_ml[base * 2] = m;
                        p.part_ml[base * 2 + 1] = l;
                    }
                }
            }
        }
    }

    // ------------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == tc::kMmaWarp) {
        if (*abort_flag && lane == 0) {   // all issued MMAs must finish before TMEM goes
            tc_commit(drain);
            mbar_wait(drain, 0, global_timer_ns() + kWaitLimitNs);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, tc::kTmemCols);
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
    pdl_wait();   // global memory from here on
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
        const int64_t row = kv_row(p, L.seq, token_at(p, L, j, j1, sBlk, jb0));
        if (row < 0) continue;
        const float *kr = Kseq + row * p.k_tok_stride;
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
        const float *vr = Vseq + row * vstride;
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

// Merges the split partials of one (query, head): grid (n_q * h_q), 512 threads.  Warp 0
// reads every split's (m, l) in one pass, keeps them in shared memory and turns them into
// merge weights; then four groups of 128 threads each sum the weighted partials of every
// fourth split with 16-byte loads (four value dims per thread), and the first group adds the
// other three's sums (a 17-split merge of the 1M-token decode took 2 µs less than with one
// group over every split).
__global__ void __launch_bounds__(512) combine_kernel(const AttnParams p, int dv) {
    __shared__ float4 s_acc[3][128];   // groups 1..3's sums
    extern __shared__ float s_w[];  // [n_split] weights, then 1/L and M, then [n_split] l
    pdl_wait();   // the partials of the attention kernel
    const int i = blockIdx.x / p.h_q, h = blockIdx.x % p.h_q;
    const int g = h / p.G, row = h % p.G;
    const int64_t base0 = ((int64_t)i * p.h_kv + g) * p.n_split * p.G + row;
    const int ns = p.n_split;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        float *s_l = s_w + ns + 2;
        float M = -INFINITY;
        for (int s = lane; s < ns; s += 32) {
            const int64_t b = base0 + (int64_t)s * p.G;
            const float m = p.part_ml[b * 2];
            s_w[s] = m;
            s_l[s] = p.part_ml[b * 2 + 1];
            M = fmaxf(M, m);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        float L = 0.f;
        for (int s = lane; s < ns; s += 32) {   // the lane's own entries: no other lane's writes
            const float m = s_w[s];
            const float w = m == -INFINITY ? 0.f : exp2f(m - M);
            s_w[s] = w;
            L += w * s_l[s];
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
    // four groups of 128 threads, group q over the splits q, q + 4, ...; thread t of a group
    // owns value dims 4t .. 4t + 3 (dv <= 512)
    const int grp = threadIdx.x >> 7, d4 = threadIdx.x & 127;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (d4 < dv / 4) {
#pragma unroll 4
        for (int s = grp; s < ns; s += 4) {
            const float w = s_w[s];
            const float4 v = __ldg(src + s * stride4 + d4);
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        if (grp > 0) s_acc[grp - 1][d4] = acc;
    }
    __syncthreads();
    if (grp == 0 && d4 < dv / 4) {
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const float4 v = s_acc[q][d4];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        dst[d4] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

// The attention over the union of two disjoint key sets from the attentions over each: one
// warp per (query, head) row; lane 0 reads both log-sum-exps, the lanes scale and add the
// row's values, and lane 0 writes the new log-sum-exp after the whole row is read (so that
// O and lse may overwrite either input).
__global__ void __launch_bounds__(128) combine2_kernel(const float4 *Oa, const float *la,
                                                      const float4 *Ob, const float *lb,
                                                      int64_t n_rows, int dv4, float4 *O,
                                                      float *lse) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (r >= n_rows) return;
    float a = -INFINITY, b = -INFINITY;
    if (lane == 0) {
        a = la[r];
        b = lb[r];
    }
    a = __shfl_sync(0xFFFFFFFFu, a, 0);
    b = __shfl_sync(0xFFFFFFFFu, b, 0);
    const float M = fmaxf(a, b);
    const float wa = M == -INFINITY ? 0.f : expf(a - M);
    const float wb = M == -INFINITY ? 0.f : expf(b - M);
    const float inv = wa + wb > 0.f ? 1.f / (wa + wb) : 0.f;
    for (int d = lane; d < dv4; d += 32) {
        const float4 x = Oa[r * dv4 + d], y = Ob[r * dv4 + d];
        O[r * dv4 + d] = make_float4((wa * x.x + wb * y.x) * inv, (wa * x.y + wb * y.y) * inv,
                                     (wa * x.z + wb * y.z) * inv, (wa * x.w + wb * y.w) * inv);
    }
    __syncwarp();
    if (lane == 0) lse[r] = M == -INFINITY ? -INFINITY : M + logf(wa + wb);
}

// ------------------------------------------------------------------------------ host side
struct SplitPlan {
    int n_split, split_tokens;
};

// Few (query, KV head) items -> split each list so that the CTAs fill one wave (one CTA per
// SM: each streams a long run of tiles, so its fixed start-up cost is amortised); many items
// -> one CTA per item.
SplitPlan plan_split(int n_q, int h_kv, int64_t n_kv_max, int per_sm = 2, int tile = kT) {
    const int64_t items = (int64_t)n_q * h_kv;
    const int64_t tiles = (n_kv_max + tile - 1) / tile;
    const int64_t target = (int64_t)per_sm * device_sm_count();
    int64_t ns = target / items;
    if (ns > tiles) ns = tiles;
    if (ns < 1) ns = 1;
    const int64_t per = (tiles + ns - 1) / ns;
    SplitPlan sp;
    sp.split_tokens = (int)(per * tile);
    sp.n_split = (int)((tiles + per - 1) / per);
    if (sp.n_split < 1) sp.n_split = 1;
    return sp;
}

// SFA_ATTEND_KERNEL=tcgen05 in the environment (read at each call) picks the tcgen05 kernel.
bool want_tcgen05() {
    const char *e = getenv("SFA_ATTEND_KERNEL");
    return e && strcmp(e, "tcgen05") == 0;
}
// SFA_ATTEND_KERNEL=ws picks the warp-specialised bulk-copy kernel (attend_ws.cu) for bf16.
bool want_ws() {
    const char *e = getenv("SFA_ATTEND_KERNEL");
    return e && strcmp(e, "ws") == 0;
}

bool shape_supported(int dkq, int dv) {
    return (dkq == 576 && dv == 512) || (dkq == 512 && dv == 512) || (dkq == 128 && dv == 128) ||
           (dkq == 64 && dv == 64);
}

// SFA_ATTEND_TT=16 in the environment (read at each call) makes the warp-level kernel stream
// 16-token tiles through up to six stages instead of 32-token tiles through two (measured on
// GB300: no faster in decode, slower in prefill, where the extra barriers per byte cost more
// than the deeper prefetch gains).
int mma_tile() {
    const char *e = getenv("SFA_ATTEND_TT");
    return e && strcmp(e, "16") == 0 ? 16 : 32;
}

// The warp-level MMA attention kernel of a shape: bf16 K/V, or q8_0 K/V rows (Q8).
template <int DKQ, int DV, bool VK, bool Q8, int TT>
constexpr auto mma_kernel() {
    if constexpr (Q8) return attend_q8_kernel<DKQ, DV, VK, TT>;
    else return attend_bf16_kernel<DKQ, DV, VK, TT>;
}

// The ring of a CTA of that kernel for a block list of blk_list entries: two CTAs per SM when
// two stages fit in half the shared memory (more warps to hide the latency of each tile's
// dependent steps), else one; and as many stages (2 .. 6) as then fit.
struct MmaRing {
    int per_sm, stages;
    size_t smem;
};
template <int DKQ, int DV, bool VK, bool Q8, int TT>
MmaRing mma_ring(int blk_list) {
    MmaRing r;
    r.per_sm = mma_smem_bytes<DKQ, DV, VK, Q8, TT>(2, blk_list) <= 113 * 1024 ? 2 : 1;
    const size_t cap = r.per_sm == 2 ? 113 * 1024 : 227 * 1024;
    r.stages = 2;
    while (r.stages < 6 && mma_smem_bytes<DKQ, DV, VK, Q8, TT>(r.stages + 1, blk_list) <= cap)
        ++r.stages;
    r.smem = mma_smem_bytes<DKQ, DV, VK, Q8, TT>(r.stages, blk_list);
    return r;
}

// Whether clusters of ns CTAs of the kernel (its shared memory for blk_list entries) can be
// resident at all; asked once per (device, kernel, ns, list size).
template <int DKQ, int DV, bool VK, bool Q8, int TT>
bool mma_clusters_fit_shape(int ns, int blk_list) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, bool> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    {
        std::lock_guard<std::mutex> lock(mu);
        auto f = cache.find({dev, ns, blk_list});
        if (f != cache.end()) return f->second;
    }
    const MmaRing ring = mma_ring<DKQ, DV, VK, Q8, TT>(blk_list);
    bool ok = ensure_max_dynamic_smem(mma_kernel<DKQ, DV, VK, Q8, TT>());
    if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(ns, 1, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = ring.smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)ns;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        ok = cudaOccupancyMaxActiveClusters(&n, mma_kernel<DKQ, DV, VK, Q8, TT>(), &cfg) ==
                 cudaSuccess && n > 0;
        cudaGetLastError();
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[{dev, ns, blk_list}] = ok;
    return ok;
}

template <int DKQ, int DV, bool VK, bool Q8, int TT>
int launch_mma_shape(const AttnParams &p, dim3 grid, cudaStream_t st, int blk_list) {
    const MmaRing ring = mma_ring<DKQ, DV, VK, Q8, TT>(blk_list);
    if (ring.smem > 227 * 1024) return SFA_ERR_UNSUPPORTED;
    AttnParams q = p;
    q.stages = ring.stages;
    auto kernel = mma_kernel<DKQ, DV, VK, Q8, TT>();
    if constexpr (!Q8 && VK && TT == 32) {
        if (q.tail_fold) kernel = attend_bf16_fold_kernel<DKQ, DV>;
    }
    if (q.tail_fold && kernel == mma_kernel<DKQ, DV, VK, Q8, TT>()) return SFA_ERR_UNSUPPORTED;
    if (!ensure_max_dynamic_smem(kernel)) return SFA_ERR_CUDA;
    const cudaError_t e =
        q.cluster_merge ? launch_pdl_cluster(kernel, grid, dim3(kThreads), ring.smem, st,
                                             q.n_split, q)
                        : launch_pdl(kernel, grid, dim3(kThreads), ring.smem, st, q);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

// Tensor map of a bf16 cache [n_seq][n_tok_cap][h_kv][d] as 3-D {d, h_kv, n_seq * n_tok_cap}
// with 4-row x 64-element boxes in the 128-byte swizzle.
bool encode_cache_map(CUtensorMap *map, const void *base, int d, int h_kv, int64_t rows) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)h_kv, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)h_kv * d * 2};
    const cuuint32_t box[3] = {64, 1, 4}, es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DKQ, int DV, bool VK>
int launch_tc(const AttnParams &p, dim3 grid, cudaStream_t st, int blk_list) {
    const size_t smem = TcLayout<DKQ, DV, VK>::bytes(blk_list);
    if (smem > 227 * 1024) return SFA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)p.n_seq * p.n_tok_cap;
    if (rows > 0x7FFFFFFF) return SFA_ERR_UNSUPPORTED;   // TMA row coordinates are 32-bit
    CUtensorMap kmap, vmap;
    if (!encode_cache_map(&kmap, p.K, DKQ, p.h_kv, rows)) return SFA_ERR_CUDA;
    if (VK) vmap = kmap;
    else if (!encode_cache_map(&vmap, p.V, DV, p.h_kv, rows)) return SFA_ERR_CUDA;
    if (!ensure_max_dynamic_smem(attend_tc_kernel<DKQ, DV, VK>)) return SFA_ERR_CUDA;
    if (launch_pdl(attend_tc_kernel<DKQ, DV, VK>, grid, dim3(tc::kThreads), smem, st, kmap, vmap,
                   p) != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

// The launch plan of one attention call: the kernel, the split of each list over CTAs and
// whether the splits merge inside a cluster (else through combine_kernel).
struct AttendPlan {
    SplitPlan sp;
    int cluster_ns;   // > 1: clusters of this many CTAs merge their splits in place
    bool use_tc;
    bool use_ws;      // the warp-specialised bulk-copy kernel (attend_ws.cu)
    WsPlan wp;
    int tt;           // tokens per tile of the warp-level kernel
};

// The per-shape dispatch of the warp-level MMA kernel's helpers (dkq in {576, 512, 128, 64};
// 576 only with V = K), for tiles of TT tokens.
template <bool Q8, int TT>
int mma_per_sm_tt(int dkq, bool has_v, int bl) {
    if (dkq == 576) return mma_ring<576, 512, true, Q8, TT>(bl).per_sm;
    if (dkq == 512) return has_v ? mma_ring<512, 512, false, Q8, TT>(bl).per_sm : mma_ring<512, 512, true, Q8, TT>(bl).per_sm;
    if (dkq == 128) return has_v ? mma_ring<128, 128, false, Q8, TT>(bl).per_sm : mma_ring<128, 128, true, Q8, TT>(bl).per_sm;
    return has_v ? mma_ring<64, 64, false, Q8, TT>(bl).per_sm : mma_ring<64, 64, true, Q8, TT>(bl).per_sm;
}
template <bool Q8>
int mma_per_sm(int dkq, bool has_v, int bl, int tt) {
    return tt == 32 ? mma_per_sm_tt<Q8, 32>(dkq, has_v, bl) : mma_per_sm_tt<Q8, 16>(dkq, has_v, bl);
}
template <bool Q8, int TT>
bool mma_clusters_fit_tt(int dkq, bool has_v, int ns, int bl) {
    if (dkq == 576) return mma_clusters_fit_shape<576, 512, true, Q8, TT>(ns, bl);
    if (dkq == 512) return has_v ? mma_clusters_fit_shape<512, 512, false, Q8, TT>(ns, bl) : mma_clusters_fit_shape<512, 512, true, Q8, TT>(ns, bl);
    if (dkq == 128) return has_v ? mma_clusters_fit_shape<128, 128, false, Q8, TT>(ns, bl) : mma_clusters_fit_shape<128, 128, true, Q8, TT>(ns, bl);
    return has_v ? mma_clusters_fit_shape<64, 64, false, Q8, TT>(ns, bl) : mma_clusters_fit_shape<64, 64, true, Q8, TT>(ns, bl);
}
template <bool Q8>
bool mma_clusters_fit(int dkq, bool has_v, int ns, int bl, int tt) {
    return tt == 32 ? mma_clusters_fit_tt<Q8, 32>(dkq, has_v, ns, bl) : mma_clusters_fit_tt<Q8, 16>(dkq, has_v, ns, bl);
}
template <bool Q8, int TT>
int mma_launch_tt(int dkq, bool has_v, const AttnParams &p, dim3 grid, cudaStream_t st, int bl) {
    if (dkq == 576) return has_v ? SFA_ERR_UNSUPPORTED : launch_mma_shape<576, 512, true, Q8, TT>(p, grid, st, bl);
    if (dkq == 512) return has_v ? launch_mma_shape<512, 512, false, Q8, TT>(p, grid, st, bl) : launch_mma_shape<512, 512, true, Q8, TT>(p, grid, st, bl);
    if (dkq == 128) return has_v ? launch_mma_shape<128, 128, false, Q8, TT>(p, grid, st, bl) : launch_mma_shape<128, 128, true, Q8, TT>(p, grid, st, bl);
    return has_v ? launch_mma_shape<64, 64, false, Q8, TT>(p, grid, st, bl) : launch_mma_shape<64, 64, true, Q8, TT>(p, grid, st, bl);
}
template <bool Q8>
int mma_launch(int dkq, bool has_v, const AttnParams &p, dim3 grid, cudaStream_t st, int bl, int tt) {
    return tt == 32 ? mma_launch_tt<Q8, 32>(dkq, has_v, p, grid, st, bl) : mma_launch_tt<Q8, 16>(dkq, has_v, p, grid, st, bl);
}

AttendPlan make_attend_plan(int dtype, int n_q, int h_kv, int dkq, bool has_v, int64_t n_kv_max,
                            int cr, int dense, bool paged = false) {
    // bf16 inputs take the warp-level mma.sync kernel, which is the faster one on the decode
    // and prefill shapes measured; SFA_ATTEND_KERNEL=tcgen05 selects the tcgen05 kernel for the
    // 512-wide heads instead (same results within the same tolerances).  fp32 inputs take the
    // SIMT kernel.  The paged layout always takes the mma.sync kernel: the tcgen05 kernel's
    // producers copy runs of four consecutive rows as one TMA box.  q8_0 caches take the
    // mma.sync kernel's quantized-cache variant.
    const int tc_tile = tc::kTT;
    AttendPlan ap{};
    const bool use_tc = dtype == SFA_BF16 && (dkq == 576 || dkq == 512) && !paged && want_tcgen05();
    ap.use_tc = use_tc;
    if (dtype == SFA_BF16 && !use_tc && want_ws() &&
        ws_make_plan(n_q, h_kv, dkq, dkq == 576 ? 512 : dkq, has_v, n_kv_max, cr, dense, &ap.wp)) {
        ap.use_ws = true;
        ap.sp.n_split = ap.wp.n_split;
        ap.sp.split_tokens = ap.wp.split_tokens;
        ap.cluster_ns = ap.wp.cluster;
        return ap;
    }
    const bool q8 = dtype == SFA_Q8_0;
    const bool mma = (dtype == SFA_BF16 && !use_tc) || q8;
    const int tt = mma ? mma_tile() : (use_tc ? tc_tile : kT);
    ap.tt = tt;
    // resident CTAs per SM of the kernel this shape takes (the split plan fills them once)
    int per_sm = 1;
    if (mma) {
        const int bl_max = dense ? 0 : (int)(n_kv_max / cr + 2);
        per_sm = q8 ? mma_per_sm<true>(dkq, has_v, bl_max, tt)
                    : mma_per_sm<false>(dkq, has_v, bl_max, tt);
    }
    SplitPlan sp = plan_split(n_q, h_kv, n_kv_max, per_sm, tt);
    // bf16 decode-like plans of a few splits merge them inside a cluster (2, 4 or 8 CTAs)
    // instead of through a second kernel
    int cluster_ns = 0;
    if (mma && sp.n_split >= 2 && sp.n_split <= 12) {
        const int ns = sp.n_split >= 6 ? 8 : (sp.n_split >= 3 ? 4 : 2);
        const int64_t tiles = (n_kv_max + tt - 1) / tt;
        const int64_t per = (tiles + ns - 1) / ns;
        const int bl = dense ? 0 : (int)(per * tt / cr + 2);
        bool fit = (int64_t)((tiles + per - 1) / per) == ns && bl <= kMaxBlkList;
        if (fit) fit = q8 ? mma_clusters_fit<true>(dkq, has_v, ns, bl, tt)
                          : mma_clusters_fit<false>(dkq, has_v, ns, bl, tt);
        if (fit) {
            cluster_ns = ns;
            sp.n_split = ns;
            sp.split_tokens = (int)(per * tt);
        }
    }
    ap.sp = sp;
    ap.cluster_ns = cluster_ns;
    return ap;
}

int run_attend(const void *Q, const void *K, const void *V, int dtype, int n_seq,
               int64_t n_tok_cap, int n_q, int h_q, int h_kv, int dkq, int dv, float scale,
               const int32_t *q_seq, const int32_t *q_pos, const int32_t *blk_idx,
               const int32_t *n_sel, int top_k, int cr, int dense, int64_t n_kv_max, float *O,
               float *lse, void *ws, size_t ws_bytes, int32_t *status, cudaStream_t st,
               const int32_t *cell_of = nullptr, int64_t n_cells = 0, int64_t window = 0,
               int part = SFA_PART_ALL) {
    if (!Q || !K || !q_seq || !q_pos || !O) return SFA_ERR_INVALID_ARG;
    if (dtype != SFA_BF16 && dtype != SFA_F32 && dtype != SFA_Q8_0) return SFA_ERR_INVALID_ARG;
    if (n_seq < 1 || n_tok_cap < 1 || n_q < 0 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0)
        return SFA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return SFA_ERR_INVALID_ARG;
    if (!dense && (!blk_idx || !n_sel || cr < 1 || top_k < 1)) return SFA_ERR_INVALID_ARG;
    if (!dense && top_k > 2048) return SFA_ERR_UNSUPPORTED;
    if (n_kv_max < 1) return SFA_ERR_INVALID_ARG;
    if (cell_of && (n_cells < 1 || n_cells > 0x7FFFFFFF)) return SFA_ERR_INVALID_ARG;
    if (dv > dkq && !V) return SFA_ERR_INVALID_ARG;
    if (!shape_supported(dkq, dv) || h_q / h_kv > 16) return SFA_ERR_UNSUPPORTED;
    if (!aligned16(Q) || !aligned16(K) || (V && !aligned16(V)) || !aligned16(O))
        return SFA_ERR_INVALID_ARG;
    if (n_q == 0) return SFA_OK;
    if (n_q > 65535 || h_kv > 65535 || n_kv_max > 0x7FFFFFFF) return SFA_ERR_UNSUPPORTED;
    AttendPlan ap = make_attend_plan(dtype, n_q, h_kv, dkq, V != nullptr, n_kv_max, cr, dense,
                                     cell_of != nullptr);
    // The tail folded into the last split: the splits are planned over the kept tokens alone
    // (top_k cr), so that a list of 512 blocks and a 3-token tail takes eight tiles per split
    // instead of nine.  Only where the plan stays an in-cluster merge on the warp-level bf16
    // kernel with V = K, and the tail is a plain suffix (no window) of at most 15 tokens.  (One-
    // split prefill lists measured slower with it: pp2048's attention 905 -> 911 us.)
    int tail_fold = 0;
    if (dtype == SFA_BF16 && !dense && !V && window == 0 && part == SFA_PART_ALL && cr >= 2 &&
        cr <= 16 && ap.cluster_ns > 1 && !ap.use_tc && !ap.use_ws && ap.tt == 32) {
        const int64_t n_kept = (int64_t)top_k * cr < n_kv_max ? (int64_t)top_k * cr : n_kv_max;
        const AttendPlan f = make_attend_plan(dtype, n_q, h_kv, dkq, false, n_kept, cr, dense,
                                              cell_of != nullptr);
        if (n_kept < n_kv_max && f.cluster_ns > 1 && !f.use_tc && !f.use_ws && f.tt == 32) {
            ap = f;
            tail_fold = 1;
        }
    }
    const bool use_tc = ap.use_tc;
    SplitPlan sp = ap.sp;
    const int cluster_ns = ap.cluster_ns;
    const size_t need = sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv_max);
    if (need > 0 && (!ws || ws_bytes < need)) return SFA_ERR_WORKSPACE;

    AttnParams p{};
    p.Q = Q; p.K = K; p.V = V;
    p.q_seq = q_seq; p.q_pos = q_pos; p.blk_idx = blk_idx; p.n_sel = n_sel;
    p.O = O; p.lse = lse; p.status = status;
    // strides in elements of the cache's type: bf16 / fp32 values, or bytes of q8_0 rows
    const int64_t krow = dtype == SFA_Q8_0 ? q8_row_bytes(dkq) : dkq;
    const int64_t vrow = dtype == SFA_Q8_0 ? q8_row_bytes(dv) : dv;
    p.k_tok_stride = (int64_t)h_kv * krow;
    p.k_seq_stride = n_tok_cap * p.k_tok_stride;
    p.v_tok_stride = V ? (int64_t)h_kv * vrow : p.k_tok_stride;
    p.v_seq_stride = V ? n_tok_cap * p.v_tok_stride : p.k_seq_stride;
    p.n_tok_cap = n_tok_cap;
    if (cell_of) {   // rows come from the map: every sequence starts at row 0 of the cell arrays
        p.k_seq_stride = p.v_seq_stride = 0;
        p.cell_of = cell_of;
        p.n_cells = n_cells;
    }
    p.n_seq = n_seq; p.n_q = n_q; p.h_q = h_q; p.h_kv = h_kv; p.G = h_q / h_kv;
    p.top_k = top_k; p.cr = cr; p.dense = dense;
    p.n_split = sp.n_split; p.split_tokens = sp.split_tokens;
    p.cluster_merge = cluster_ns > 1;
    p.n_items = n_q * h_kv * sp.n_split;
    p.n_kv_max = n_kv_max;
    p.window = window;
    p.part = part;
    p.tail_fold = tail_fold;
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
    if (ap.use_ws) {
        rc = ws_launch(p, ap.wp, dkq, dv, V != nullptr, st);
    } else if (use_tc) {
        if (dkq == 576) rc = V ? SFA_ERR_UNSUPPORTED : launch_tc<576, 512, true>(p, grid, st, bl);
        else rc = V ? launch_tc<512, 512, false>(p, grid, st, bl) : launch_tc<512, 512, true>(p, grid, st, bl);
    } else if (dtype == SFA_BF16) {
        rc = mma_launch<false>(dkq, V != nullptr, p, grid, st, bl, ap.tt);
    } else if (dtype == SFA_Q8_0) {
        rc = mma_launch<true>(dkq, V != nullptr, p, grid, st, bl, ap.tt);
    } else {
        const cudaError_t e =
            dkq == 576   ? launch_pdl(attend_f32_kernel<576, 512>, grid, dim3(kThreads), 0, st, p)
            : dkq == 512 ? launch_pdl(attend_f32_kernel<512, 512>, grid, dim3(kThreads), 0, st, p)
            : dkq == 128 ? launch_pdl(attend_f32_kernel<128, 128>, grid, dim3(kThreads), 0, st, p)
                         : launch_pdl(attend_f32_kernel<64, 64>, grid, dim3(kThreads), 0, st, p);
        if (e != cudaSuccess) cudaGetLastError();
        rc = e == cudaSuccess ? SFA_OK : SFA_ERR_CUDA;
    }
    if (rc != SFA_OK) return rc;
    if (sp.n_split > 1 && !p.cluster_merge) {
        if (launch_pdl(combine_kernel, dim3(n_q * h_q), dim3(512),
                       (2 * sp.n_split + 2) * sizeof(float), st, p, dv) != cudaSuccess) {
            cudaGetLastError();
            return SFA_ERR_CUDA;
        }
    }
    return SFA_OK;
}

}  // namespace
}  // namespace sfa

extern "C" int sfa_attend_plan(int dtype, int n_q, int h_kv, int dkq, int has_v,
                               int64_t n_kv_max, int compress_ratio, int dense, int *n_split,
                               int *kernels) {
    using namespace sfa;
    if (!n_split || !kernels || n_q < 1 || h_kv < 1 || n_kv_max < 1 || compress_ratio < 1)
        return SFA_ERR_INVALID_ARG;
    if (dtype != SFA_BF16 && dtype != SFA_F32 && dtype != SFA_Q8_0) return SFA_ERR_INVALID_ARG;
    if (dkq != 576 && dkq != 512 && dkq != 128 && dkq != 64) return SFA_ERR_UNSUPPORTED;
    const AttendPlan ap = make_attend_plan(dtype, n_q, h_kv, dkq, has_v != 0, n_kv_max,
                                           compress_ratio, dense);
    *n_split = ap.sp.n_split;
    *kernels = ap.sp.n_split > 1 && ap.cluster_ns <= 1 ? 2 : 1;
    return SFA_OK;
}

extern "C" size_t sfa_attend_workspace_bytes(int n_q, int h_q, int h_kv, int dv, int64_t n_kv_max) {
    if (n_q <= 0 || h_q <= 0 || h_kv <= 0 || dv <= 0 || n_kv_max <= 0) return 0;
    // the largest split count any kernel's plan takes: the warp-level kernel's (two CTAs per
    // SM, 16-row tiles; 32-row tiles and the tcgen05 kernel split less) and the
    // warp-specialised kernel's (one CTA per SM, pieces of at least 64 rows)
    const sfa::SplitPlan sp = sfa::plan_split(n_q, h_kv, n_kv_max, 2, 16);
    int64_t ns_ws = sfa::device_sm_count() / ((int64_t)n_q * h_kv);
    const int64_t ws_cap = ((n_kv_max + 15) / 16 + 3) / 4;
    if (ns_ws > ws_cap) ns_ws = ws_cap;
    const int ns = sp.n_split > ns_ws ? sp.n_split : (int)ns_ws;
    if (ns <= 1) return 0;
    return (size_t)n_q * h_q * ns * ((size_t)dv + 2) * sizeof(float);
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

extern "C" int64_t sfa_window_kv_max(int top_k, int compress_ratio, int64_t window, int part) {
    if (top_k < 1 || compress_ratio < 1 || window < 0) return 0;
    const int64_t kept = (int64_t)top_k * compress_ratio;
    // the suffix s0 .. p holds at most max(window, cr - 1) positions
    const int64_t suffix = window > compress_ratio - 1 ? window : compress_ratio - 1;
    if (part == SFA_PART_SELECTED) return kept;
    if (part == SFA_PART_WINDOW) return suffix > 0 ? suffix : 1;
    return kept + suffix;
}

extern "C" int sfa_gather_attend_window(const void *Q, const void *K, const void *V, int dtype,
                                        int n_seq, int64_t n_tok_cap, int n_q, int h_q, int h_kv,
                                        int dkq, int dv, float scale, const int32_t *q_seq,
                                        const int32_t *q_pos, const int32_t *blk_idx,
                                        const int32_t *n_sel, int top_k, int compress_ratio,
                                        int64_t window, int part, float *O, float *lse,
                                        void *workspace, size_t workspace_bytes,
                                        int32_t *dev_status, sfa_stream_t stream) {
    if (compress_ratio < 1 || top_k < 1 || window < 0) return SFA_ERR_INVALID_ARG;
    if (part != SFA_PART_ALL && part != SFA_PART_SELECTED && part != SFA_PART_WINDOW)
        return SFA_ERR_INVALID_ARG;
    const int64_t n_kv_max = sfa_window_kv_max(top_k, compress_ratio, window, part);
    return sfa::run_attend(Q, K, V, dtype, n_seq, n_tok_cap, n_q, h_q, h_kv, dkq, dv, scale,
                           q_seq, q_pos, blk_idx, n_sel, top_k, compress_ratio, 0, n_kv_max, O,
                           lse, workspace, workspace_bytes, dev_status, (cudaStream_t)stream,
                           nullptr, 0, window, part);
}

extern "C" int sfa_gather_kv_bandwidth(const void *K, const void *V, int n_seq, int64_t n_tok_cap,
                                       int n_q, int h_kv, int dkq, int dv,
                                       const int32_t *q_seq, const int32_t *q_pos,
                                       const int32_t *blk_idx, const int32_t *n_sel, int top_k,
                                       int compress_ratio, uint32_t *checksum,
                                       int32_t *dev_status, sfa_stream_t stream) {
    using namespace sfa;
    if (!K || !q_seq || !q_pos || !blk_idx || !n_sel || !checksum) return SFA_ERR_INVALID_ARG;
    if (n_seq < 1 || n_tok_cap < 1 || n_q < 0 || h_kv < 1 || compress_ratio < 1 || top_k < 1)
        return SFA_ERR_INVALID_ARG;
    if (top_k > 2048) return SFA_ERR_UNSUPPORTED;
    if (!((dkq == 576 && dv == 512 && !V) || (dkq == 512 && dv == 512)))
        return SFA_ERR_UNSUPPORTED;
    if (!aligned16(K) || (V && !aligned16(V))) return SFA_ERR_INVALID_ARG;
    if (n_q == 0) return SFA_OK;
    if (n_q > 65535 || h_kv > 65535) return SFA_ERR_UNSUPPORTED;
    const int64_t n_kv_max = (int64_t)top_k * compress_ratio + compress_ratio - 1;
    WsPlan wp{};
    if (!ws_make_plan(n_q, h_kv, dkq, dv, V != nullptr, n_kv_max, compress_ratio, 0, &wp))
        return SFA_ERR_UNSUPPORTED;
    AttnParams p{};
    p.K = K; p.V = V;
    p.q_seq = q_seq; p.q_pos = q_pos; p.blk_idx = blk_idx; p.n_sel = n_sel;
    p.status = dev_status;
    p.k_tok_stride = (int64_t)h_kv * dkq;
    p.k_seq_stride = n_tok_cap * p.k_tok_stride;
    p.v_tok_stride = V ? (int64_t)h_kv * dv : p.k_tok_stride;
    p.v_seq_stride = V ? n_tok_cap * p.v_tok_stride : p.k_seq_stride;
    p.n_tok_cap = n_tok_cap;
    p.n_seq = n_seq; p.n_q = n_q; p.h_q = h_kv; p.h_kv = h_kv; p.G = 1;
    p.top_k = top_k; p.cr = compress_ratio; p.dense = 0;
    p.n_split = wp.n_split; p.split_tokens = wp.split_tokens;
    p.n_items = n_q * h_kv * wp.n_split;
    p.n_kv_max = n_kv_max;
    if (wp.split_tokens / compress_ratio + 2 > kMaxBlkList) return SFA_ERR_UNSUPPORTED;
    return ws_gather_launch(p, wp, dkq, dv, V != nullptr, checksum, (cudaStream_t)stream);
}

extern "C" int sfa_combine_attention(const float *O_a, const float *lse_a, const float *O_b,
                                     const float *lse_b, int64_t n_rows, int dv, float *O,
                                     float *lse, sfa_stream_t stream) {
    using namespace sfa;
    if (!O_a || !lse_a || !O_b || !lse_b || !O || !lse || n_rows < 0 || dv < 4 || dv % 4)
        return SFA_ERR_INVALID_ARG;
    if (!aligned16(O_a) || !aligned16(O_b) || !aligned16(O)) return SFA_ERR_INVALID_ARG;
    if (n_rows == 0) return SFA_OK;
    if ((n_rows + 3) / 4 > 0x7FFFFFFF) return SFA_ERR_UNSUPPORTED;
    if (launch_pdl(combine2_kernel, dim3((unsigned)((n_rows + 3) / 4)), dim3(128), 0,
                   (cudaStream_t)stream, reinterpret_cast<const float4 *>(O_a), lse_a,
                   reinterpret_cast<const float4 *>(O_b), lse_b, n_rows, dv / 4,
                   reinterpret_cast<float4 *>(O), lse) != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
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

extern "C" int sfa_gather_attend_paged(const void *Q, const void *K, const void *V, int dtype,
                                       int64_t n_cells, const int32_t *cell_of, int n_seq,
                                       int64_t n_pos_cap, int n_q, int h_q, int h_kv, int dkq,
                                       int dv, float scale, const int32_t *q_seq,
                                       const int32_t *q_pos, const int32_t *blk_idx,
                                       const int32_t *n_sel, int top_k, int compress_ratio,
                                       float *O, float *lse, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status,
                                       sfa_stream_t stream) {
    if (!cell_of || compress_ratio < 1 || top_k < 1) return SFA_ERR_INVALID_ARG;
    const int64_t n_kv_max = (int64_t)top_k * compress_ratio + compress_ratio - 1;
    return sfa::run_attend(Q, K, V, dtype, n_seq, n_pos_cap, n_q, h_q, h_kv, dkq, dv, scale,
                           q_seq, q_pos, blk_idx, n_sel, top_k, compress_ratio, 0, n_kv_max, O,
                           lse, workspace, workspace_bytes, dev_status, (cudaStream_t)stream,
                           cell_of, n_cells);
}

extern "C" int sfa_dense_attend_paged(const void *Q, const void *K, const void *V, int dtype,
                                      int64_t n_cells, const int32_t *cell_of, int n_seq,
                                      int64_t n_pos_cap, int n_q, int h_q, int h_kv, int dkq,
                                      int dv, float scale, const int32_t *q_seq,
                                      const int32_t *q_pos, int64_t n_kv_max, float *O,
                                      float *lse, void *workspace, size_t workspace_bytes,
                                      int32_t *dev_status, sfa_stream_t stream) {
    if (!cell_of) return SFA_ERR_INVALID_ARG;
    return sfa::run_attend(Q, K, V, dtype, n_seq, n_pos_cap, n_q, h_q, h_kv, dkq, dv, scale,
                           q_seq, q_pos, nullptr, nullptr, 0, 1, 1, n_kv_max, O, lse, workspace,
                           workspace_bytes, dev_status, (cudaStream_t)stream, cell_of, n_cells);
}

// ---------------------------------------------------------------------------------------
// sfa_gather_attend_noalloc: the split-KV scratch lives in this file-scope device array, so
// the call allocates nothing.  Host code may not use the array's name as a device address:
// the address is looked up once per device with cudaGetSymbolAddress and cached.
namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[SFA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
struct NoallocSlot {
    void *ctx;    // the context the address was looked up in
    void *ptr;    // device address of g_noalloc_scratch in that context
};
NoallocSlot g_noalloc_slot[64] = {};

// Device address of g_noalloc_scratch on the current device (nullptr on failure).  The address
// is looked up once per device and context: a new context on the device (after
// cudaDeviceReset, or another context made current) looks it up again.
void *noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    void *ctx = sfa::current_context();
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocSlot &s = g_noalloc_slot[dev];
    if (!s.ptr || s.ctx != ctx || !ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            s.ptr = nullptr;
            return nullptr;
        }
        s.ptr = p;
        s.ctx = ctx;
    }
    return s.ptr;
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
