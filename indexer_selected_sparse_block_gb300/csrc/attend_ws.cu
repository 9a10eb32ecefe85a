// attend_ws.cu -- gathered flash attention over the kept cells, warp-specialised, for bf16
// caches: the default kernel of sfa_gather_attend / sfa_dense_attend and their paged twins.
//
// What it computes is fixed by llama.cpp PR #27970 "CUDA + ggml: add sparse-fa for DSV4/GLM"
// (flash attention over only the selected K/V cells; V the first 512 dims of K for the MLA
// heads, separate V for 512/512; no ALiBi, no softcap) and by the QSA paragraphs of llama.cpp
// commit "model: add Qwen3.8-Flash-Next (qwen4exp)" (the kept blocks plus the tail).  The
// design is this library's own:
//
//   * one CTA per SM, 9 warps.  Warp 8 is the producer: for each work item (query, KV head,
//     piece of its list) it reads the item's list metadata and kept block ids, copies the
//     item's Q rows, then streams the list in tiles of 16 token rows through a ring of shared
//     memory stages.  Each row is one 1-D bulk copy (cp.async.bulk, its bytes counted on the
//     stage's mbarrier) into a row padded by 16 bytes, so that ldmatrix reads of 8 rows at the
//     same column hit 8 different bank groups.  Rows outside the list are zeroed and masked.
//   * warps 0-3 and 4-7 are two consumer warpgroups that take alternate tiles (ping-pong), so
//     that one group's softmax overlaps the other's tensor-core work.  Per tile a group runs
//       S = Q K^T   (mma.sync m16n8k16: M = the 16 query heads of the KV head; the head dim
//                   split over its 4 warps, partial sums reduced in shared memory),
//       online softmax in base 2 over the 16 tokens,
//       O += P V    (the value dims split over its 4 warps).
//     P V runs on binary16 operands when P16 (P rounded to binary16, the bf16 V fragments
//     converted to binary16 after ldmatrix: exact for |v| in [2^-14, 65504], absolute error at
//     most 2^-25 below; a non-finite result raises SFA_DEV_FP16_RANGE), else on bf16 with P
//     carried as two bf16 halves (hi + lo).
//   * at the end of an item the two groups merge their (m, l, O) through shared memory, each
//     finishing half of the rows; the result is written as the final output, as a partial for
//     combine_kernel, or (cluster plans) kept in shared memory and merged over distributed
//     shared memory by the CTAs of the item's cluster.
//
// Plans (ws_make_plan): few (query, KV head) items -> each list is cut into n_split pieces,
// one per CTA, merged in a cluster of 2, 4 or 8 CTAs when one fits, else by combine_kernel;
// many items -> one piece per item and a persistent grid of one CTA per SM, whose producer
// runs ahead into the next item while the consumers finish the current one.
//
// Every mbarrier wait is bounded (SFA_DEV_TIMEOUT); after a timeout the kernel keeps the same
// control flow with no further waiting, so every named barrier is still met, and the producer
// waits (bounded) for its own copies before it leaves.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <map>
#include <mutex>
#include <tuple>

#include <cooperative_groups.h>

#include "attend_common.cuh"

namespace sfa {
namespace ws {

namespace cg = cooperative_groups;

constexpr int kTT = 32;            // token rows per tile
constexpr int kSlots = 8;          // a tile is 8 slots of kSlotRows consecutive list positions
constexpr int kSlotRows = 4;
constexpr int kThreads = 288;      // eight consumer warps + the producer warp
constexpr int kProdWarp = 8;
constexpr int kSpPitch = 24;       // fp32 S-partial row pitch (16 tokens + 8)
constexpr int kPPitch = kTT + 8;   // 16-bit P row pitch (elements)
constexpr int kMaxStages = 8;
constexpr int kMinSplitTiles = 2;  // a piece of a list holds at least 2 tiles (64 rows)

// Shared-memory layout of one CTA (byte offsets); ns stages, bl block-list entries.  A stage
// holds one tile: K (and separate V) as 8 slots of 4 rows at the cache's row size, slot j at
// j * (4 rows + 16 bytes), so that row r of slot j -- the tile's token n = 8 r + j in MMA order
// -- starts in 16-byte bank group (j + r * rows/16) mod 8 = j mod 8: the 8 rows any ldmatrix
// reads (8 consecutive n) lie in 8 different bank groups.
template <int DKQ, int DV, bool V_IS_K>
struct Layout {
    static constexpr int KR = DKQ * 2, VR = DV * 2;          // bytes of one K / V row
    static constexpr int KSLOT = kSlotRows * KR + 16, VSLOT = kSlotRows * VR + 16;
    static constexpr int KTILE = kSlots * KSLOT, VTILE = V_IS_K ? 0 : kSlots * VSLOT;
    static constexpr int STAGE = KTILE + VTILE;
    static constexpr int QP = KR + 16;                       // padded Q row pitch
    static constexpr int SP_BYTES = 8 * 16 * kSpPitch * 4;   // S partials of the 8 warps
    static constexpr int P_BYTES = 2 * 16 * kPPitch * 2;     // P (or P hi, P lo)
    int ns, bl;
    __host__ __device__ int off_q() const { return ns * STAGE; }
    __host__ __device__ int off_sp() const { return off_q() + 16 * QP; }
    __host__ __device__ int off_p() const { return off_sp() + SP_BYTES; }
    __host__ __device__ int off_stat() const { return off_p() + P_BYTES; }   // alpha, m, l [16]
    __host__ __device__ int off_tok() const { return off_stat() + 3 * 16 * 4; }
    __host__ __device__ int off_item() const { return off_tok() + ns * kTT * 4; }
    __host__ __device__ int off_bar() const { return off_item() + 48; }
    __host__ __device__ int n_bars() const { return 2 * ns + 2; }
    __host__ __device__ int off_abort() const { return off_bar() + n_bars() * 8; }
    __host__ __device__ int off_blk() const { return off_abort() + 16; }
    __host__ __device__ int bytes() const { return off_blk() + bl * 4 + 16; }
};
static_assert(Layout<576, 512, true>::STAGE % 16 == 0, "16-byte aligned stages");
static_assert((Layout<576, 512, true>::KSLOT / 16) % 8 == 1, "slot bases rotate the bank groups");

// Address offset (bytes) of the tile's token n (MMA order) in a K or V tile with slots of
// `slot` bytes and rows of `row` bytes.
__device__ __forceinline__ int tok_off(int n, int slot, int row) {
    return (n & (kSlots - 1)) * slot + (n >> 3) * row;
}

// mbarrier wait that gives up at `deadline` (raising SFA_DEV_TIMEOUT and the CTA's abort flag)
// or at once when another thread of the CTA already gave up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, uint64_t deadline,
                                              volatile int *abort_flag, int32_t *status) {
    const uint32_t a = smem_u32(bar);
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 63u) == 63u) {
            if (*abort_flag) return false;
            if (global_timer_ns() > deadline) {
                *abort_flag = 1;
                set_status(status, SFA_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

// Two bf16 values -> two binary16 values (round to nearest even; exact in binary16's normal
// range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack_f16(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// Work item -> (query, KV head, piece of its list).
struct Item {
    int i, g, split;
};
__device__ __forceinline__ Item decompose(const AttnParams &p, int item) {
    Item it;
    it.split = item % p.n_split;
    const int ig = item / p.n_split;
    it.g = ig % p.h_kv;
    it.i = ig / p.h_kv;
    return it;
}

// The merge of the n_split CTAs of one item's cluster (flash-decoding without a second
// kernel): each CTA holds its unnormalised rows sPart[G][DV] and their (m, l) in sM, sL
// (base 2); CTA r writes the value dims [r DV/ns, (r+1) DV/ns) of every row as
// sum_c w_c O_c / sum_c w_c l_c with w_c = 2^(m_c - M).  sW (ns * 16 floats) is scratch.  Run by
// the 256 consumer threads; the producer warp meets the two cluster barriers on its own.
template <int DV>
__device__ void cluster_merge(const AttnParams &p, float *sPart, const float *sL,
                              const float *sM, float *sW, int i, int g, int ctid) {
    cg::cluster_group cl = cg::this_cluster();
    const int G = p.G, ns = p.n_split;
    cl.sync();   // every CTA's partial rows and statistics are in its shared memory
    const int r = (int)cl.block_rank();
    if (ctid < G) {
        float M = -INFINITY;
        for (int c = 0; c < ns; ++c) M = fmaxf(M, cl.map_shared_rank(sM, c)[ctid]);
        float Lsum = 0.f;
        for (int c = 0; c < ns; ++c) {
            const float m = cl.map_shared_rank(sM, c)[ctid];
            const float w = m == -INFINITY ? 0.f : exp2f(m - M);
            sW[c * 16 + ctid] = w;
            Lsum += w * cl.map_shared_rank(sL, c)[ctid];
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        for (int c = 0; c < ns; ++c) sW[c * 16 + ctid] *= inv;
        if (r == 0 && p.lse)
            p.lse[(int64_t)i * p.h_q + g * G + ctid] =
                Lsum > 0.f ? (M + log2f(Lsum)) / kLog2e : -INFINITY;
    }
    named_barrier(1, 256);
    const int dq = DV / ns / 4;   // float4 per row in this CTA's slice
    const int d0 = r * (DV / ns);
    for (int e = ctid; e < G * dq; e += 256) {
        const int row = e / dq, d = d0 + 4 * (e % dq);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < ns; ++c) {
            const float w = sW[c * 16 + row];
            if (w == 0.f) continue;   // an empty piece: its rows are not written
            const float4 v =
                *reinterpret_cast<const float4 *>(cl.map_shared_rank(sPart, c) + row * DV + d);
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        *reinterpret_cast<float4 *>(p.O + ((int64_t)i * p.h_q + g * G + row) * DV + d) = acc;
    }
    cl.sync();   // no CTA leaves while another may still read its shared memory
}

template <int DKQ, int DV, bool V_IS_K, bool P16>
__global__ void __launch_bounds__(kThreads, 1)
    attend_ws_kernel(const AttnParams p, const int ns, const int bl_cap) {
    using Lay = Layout<DKQ, DV, V_IS_K>;
    constexpr int KR = Lay::KR, VR = Lay::VR, KSLOT = Lay::KSLOT, VSLOT = Lay::VSLOT;
    constexpr int STAGE = Lay::STAGE, QP = Lay::QP;
    constexpr int KS = DKQ / 64;        // k16 steps of S per warp (the head dim over 4 warps)
    constexpr int NTV = DV / 64;        // n8 tiles of O per warp (the value dims over 8 warps)
    static_assert(KS >= 1 && NTV >= 1 && (NTV == 1 || NTV % 2 == 0), "head sizes");
    const Lay lay{ns, bl_cap};

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sRing = smem;
    uint8_t *sQ = smem + lay.off_q();
    float *sSP = reinterpret_cast<float *>(smem + lay.off_sp());      // [8][16][kSpPitch]
    uint16_t *sP = reinterpret_cast<uint16_t *>(smem + lay.off_p());  // [2][16][kPPitch]
    float *sAlpha = reinterpret_cast<float *>(smem + lay.off_stat()); // [16]
    float *sM = sAlpha + 16, *sL = sM + 16;                           // final (m, l) [16]
    int *sTok = reinterpret_cast<int *>(smem + lay.off_tok());        // [ns][kTT], MMA order
    int *sItem = reinterpret_cast<int *>(smem + lay.off_item());      // [2][4] + [4]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.off_bar());
    uint64_t *full = bars, *empty = bars + ns, *qfull = bars + 2 * ns, *qempty = qfull + 1;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + lay.off_abort());
    int *sBlk = reinterpret_cast<int *>(smem + lay.off_blk());

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.G;
    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 1);    // the producer's expect-tx arrival
            mbar_init(&empty[s], 8);   // the eight consumer warps
        }
        mbar_init(qfull, 1);
        mbar_init(qempty, 8);          // every consumer warp holds Q in registers
        *abort_flag = 0;
        fence_mbar_init();
    }
    // Q rows >= G stay zero for the whole kernel: the Q copies only write rows < G.
    for (int e = tid; e < (16 - G) * (QP / 16); e += kThreads) {
        const int r = G + e / (QP / 16), c = e % (QP / 16);
        *reinterpret_cast<uint4 *>(sQ + r * QP + c * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    pdl_wait();   // global memory from here on
    const uint64_t deadline = global_timer_ns() + kWaitLimitNs;

    if (warp == kProdWarp) {
        // ------------------------------------------------------------------- producer
        // Lane j < 8 fills slot j of every tile: the 4 consecutive list positions
        // 32 t + 4 j .. + 3.  When their rows are consecutive in the cache (a kept block of
        // cr >= 4 rows, a run of the tail, the dense case: rows of one KV head back to back)
        // the slot is one bulk copy of 4 rows; otherwise (the ragged end of a list, a KV
        // head's rows interleaved with other heads', blocks of fewer than 4 tokens, paged
        // cells out of order) each valid row is copied on its own and missing rows are zeroed.
        const __nv_bfloat16 *Kb = reinterpret_cast<const __nv_bfloat16 *>(p.K);
        const __nv_bfloat16 *Vb = reinterpret_cast<const __nv_bfloat16 *>(p.V);
        const __nv_bfloat16 *Qb = reinterpret_cast<const __nv_bfloat16 *>(p.Q);
        const bool k_dense = p.k_tok_stride == DKQ, v_dense = p.v_tok_stride == DV;
        int gt = 0, k = 0;
        for (int item = blockIdx.x; item < p.n_items; item += gridDim.x, ++k) {
            const Item it = decompose(p, item);
            const ListInfo L = list_info(p, it.i, lane == 0 && it.split == 0 && it.g == 0);
            const int j0 = it.split * p.split_tokens;
            const int j1 = L.ok ? min(L.len, j0 + p.split_tokens) : 0;
            const int n_tiles = j0 < j1 ? (j1 - j0 + kTT - 1) / kTT : 0;
            // Q of this item, once every consumer warp holds the previous item's Q
            wait_or_abort(qempty, (k & 1) ^ 1, deadline, abort_flag, p.status);
            const bool live = n_tiles > 0 && !*abort_flag;
            if (live && lane < G)
                bulk_load(sQ + lane * QP,
                          Qb + ((int64_t)it.i * p.h_q + (int64_t)it.g * G + lane) * DKQ, KR, qfull);
            if (lane == 0) sItem[(k & 1) * 4] = n_tiles;
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(qfull, live ? (uint32_t)(G * KR) : 0u);
            int jb0 = 0;
            if (n_tiles > 0) jb0 = load_block_list(p, it.i, L, j0, j1, sBlk, it.g == 0, lane, 32);
            __syncwarp();

            const __nv_bfloat16 *Kseq =
                L.ok ? Kb + (int64_t)L.seq * p.k_seq_stride + (int64_t)it.g * DKQ : Kb;
            const __nv_bfloat16 *Vseq =
                V_IS_K ? Kseq
                       : (L.ok ? Vb + (int64_t)L.seq * p.v_seq_stride + (int64_t)it.g * DV : Vb);
            for (int t = 0; t < n_tiles; ++t, ++gt) {
                const int st = gt % ns;
                const uint32_t fill = (uint32_t)(gt / ns);
                // the rows of this lane's slot (lanes >= 8 hold none)
                int tok[kSlotRows];
                int64_t row[kSlotRows];
#pragma unroll
                for (int r = 0; r < kSlotRows; ++r) {
                    tok[r] = lane < kSlots
                                 ? token_at(p, L, j0 + t * kTT + lane * kSlotRows + r, j1, sBlk, jb0)
                                 : -1;
                    row[r] = tok[r] < 0 ? -1
                                        : (p.cell_of ? checked_cell(p, __ldg(p.cell_of + (int64_t)L.seq * p.n_tok_cap + tok[r]))
                                                     : (int64_t)tok[r]);
                }
                wait_or_abort(&empty[st], (fill & 1u) ^ 1u, deadline, abort_flag, p.status);
                const bool ab = *abort_flag;
                uint8_t *kdst = sRing + (size_t)st * STAGE + lane * KSLOT;
                uint8_t *vdst = sRing + (size_t)st * STAGE + Lay::KTILE + lane * VSLOT;
                int n_valid = 0;
                if (lane < kSlots) {
                    bool run = !ab;
                    bool zero_any = false;
#pragma unroll
                    for (int r = 0; r < kSlotRows; ++r) {
                        sTok[st * kTT + r * kSlots + lane] = row[r] >= 0 ? tok[r] : -1;
                        n_valid += row[r] >= 0;
                        run &= row[r] >= 0 && row[r] == row[0] + r;
                    }
                    if (run && k_dense && (V_IS_K || v_dense)) {
                        bulk_load(kdst, Kseq + row[0] * p.k_tok_stride, kSlotRows * KR, &full[st]);
                        if constexpr (!V_IS_K)
                            bulk_load(vdst, Vseq + row[0] * p.v_tok_stride, kSlotRows * VR,
                                      &full[st]);
                    } else {
#pragma unroll
                        for (int r = 0; r < kSlotRows; ++r) {
                            if (row[r] >= 0 && !ab) {
                                bulk_load(kdst + r * KR, Kseq + row[r] * p.k_tok_stride, KR,
                                          &full[st]);
                                if constexpr (!V_IS_K)
                                    bulk_load(vdst + r * VR, Vseq + row[r] * p.v_tok_stride, VR,
                                              &full[st]);
                            } else {
                                for (int c = 0; c < KR / 16; ++c)
                                    *reinterpret_cast<uint4 *>(kdst + r * KR + c * 16) =
                                        make_uint4(0u, 0u, 0u, 0u);
                                if constexpr (!V_IS_K)
                                    for (int c = 0; c < VR / 16; ++c)
                                        *reinterpret_cast<uint4 *>(vdst + r * VR + c * 16) =
                                            make_uint4(0u, 0u, 0u, 0u);
                                zero_any = true;
                            }
                        }
                        if (zero_any) fence_proxy_async_smem();
                    }
                    if (ab) n_valid = 0;
                }
                // bytes of this tile: every valid row, once the copies of all slots are issued
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) n_valid += __shfl_xor_sync(0xFFFFFFFFu, n_valid, o);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[st], (uint32_t)n_valid * (uint32_t)(KR + (V_IS_K ? 0 : VR)));
            }
        }
        // no copy of this warp is in flight when it leaves: the last fills have landed
        for (int d = gt > ns ? gt - ns : 0; d < gt; ++d)
            wait_or_abort(&full[d % ns], (uint32_t)(d / ns) & 1u, deadline, abort_flag, p.status);
        if (p.cluster_merge) {   // the cluster merge's two cluster barriers
            cg::cluster_group cl = cg::this_cluster();
            cl.sync();
            cl.sync();
        }
        return;
    }

    // ----------------------------------------------------------------------- consumers
    // S: warp w scores tokens 16 (w / 4) .. + 15 of each tile over head dims
    // (w % 4) DKQ/4 .. (a k-slice); P V: warp w owns value dims w DV/8 .. over all 32 tokens.
    const int sh = warp >> 2, wq = warp & 3;
    const int gq = lane >> 2, tq = lane & 3;
    const uint32_t q_base = smem_u32(sQ);
    const uint32_t p_base = smem_u32(sP);
    const int dv0 = warp * (DV / 8);

    int gt = 0, k = 0;
    Item cur{0, 0, 0};
    for (int item = blockIdx.x; item < p.n_items; item += gridDim.x, ++k) {
        cur = decompose(p, item);
        wait_or_abort(qfull, k & 1, deadline, abort_flag, p.status);
        // one thread reads the item's tile count and every consumer takes it from there, so
        // that all consumer loops (and their barriers) agree even after a timeout
        if (tid == 0) sItem[8] = sItem[(k & 1) * 4];
        named_barrier(1, 256);
        const int n_tiles = sItem[8];
        // Q fragments of this warp's head-dim slice (A operand, kept in registers)
        uint32_t qa[KS][4];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int kg = wq * KS + ks;
            const int r = lane & 15, c = kg * 2 + (lane >> 4);
            ldsm_x4(q_base + r * QP + c * 16, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(qempty);

        float o[NTV][4];
#pragma unroll
        for (int n = 0; n < NTV; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;   // of row tid / 16, kept by its 16 threads

        for (int t = 0; t < n_tiles; ++t) {
            const int g2 = gt + t;
            const int st = g2 % ns;
            wait_or_abort(&full[st], (uint32_t)(g2 / ns) & 1u, deadline, abort_flag, p.status);
            const uint32_t kbase = smem_u32(sRing + (size_t)st * STAGE);
            const uint32_t vbase = V_IS_K ? kbase : kbase + Lay::KTILE;

            // ---- S partial: 16 heads x 16 tokens (n = 16 sh ..) over this warp's k-slice
            {
                float acc[2][4];
#pragma unroll
                for (int n = 0; n < 2; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
                const int mi = lane >> 3, r8 = lane & 7;
                const int n = sh * 16 + (mi >> 1) * 8 + r8;
                const uint32_t rowaddr = kbase + tok_off(n, KSLOT, KR);
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int c = (wq * KS + ks) * 2 + (mi & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(rowaddr + c * 16, b0, b1, b2, b3);
                    mma_bf16_16816(acc[0], qa[ks], b0, b1);
                    mma_bf16_16816(acc[1], qa[ks], b2, b3);
                }
                float *sp = sSP + warp * 16 * kSpPitch;
#pragma unroll
                for (int n2 = 0; n2 < 2; ++n2) {
                    *reinterpret_cast<float2 *>(sp + gq * kSpPitch + n2 * 8 + 2 * tq) =
                        make_float2(acc[n2][0], acc[n2][1]);
                    *reinterpret_cast<float2 *>(sp + (gq + 8) * kSpPitch + n2 * 8 + 2 * tq) =
                        make_float2(acc[n2][2], acc[n2][3]);
                }
            }
            named_barrier(1, 256);

            // ---- online softmax: thread -> row tid / 16, tokens 2 (tid % 16), +1
            {
                const int row = tid >> 4, c0 = (tid & 15) * 2;
                const int h2 = c0 >> 4, cc = c0 & 15;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int w4 = 0; w4 < 4; ++w4) {
                    const float2 v = *reinterpret_cast<const float2 *>(
                        sSP + ((h2 * 4 + w4) * 16 + row) * kSpPitch + cc);
                    s0 += v.x;
                    s1 += v.y;
                }
                s0 = sTok[st * kTT + c0] >= 0 ? s0 * p.scale_log2 : -INFINITY;
                s1 = sTok[st * kTT + c0 + 1] >= 0 ? s1 * p.scale_log2 : -INFINITY;
                float mx = fmaxf(s0, s1);
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
                const float m_new = fmaxf(m_run, mx);
                const bool none = m_new == -INFINITY;
                const float alpha = none ? 1.f : exp2f(m_run - m_new);
                const float p0 = none ? 0.f : exp2f(s0 - m_new);
                const float p1 = none ? 0.f : exp2f(s1 - m_new);
                if constexpr (P16) {
                    *reinterpret_cast<uint32_t *>(sP + row * kPPitch + c0) = pack_f16(p0, p1);
                } else {
                    const float h0 = __bfloat162float(__float2bfloat16_rn(p0));
                    const float h1 = __bfloat162float(__float2bfloat16_rn(p1));
                    *reinterpret_cast<uint32_t *>(sP + row * kPPitch + c0) = pack_bf16(h0, h1);
                    *reinterpret_cast<uint32_t *>(sP + (16 + row) * kPPitch + c0) =
                        pack_bf16(p0 - h0, p1 - h1);
                }
                float rs = p0 + p1;
                rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 1);
                rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 2);
                rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 4);
                rs += __shfl_xor_sync(0xFFFFFFFFu, rs, 8);
                l_run = l_run * alpha + rs;
                m_run = m_new;
                if ((tid & 15) == 0) sAlpha[row] = alpha;
            }
            named_barrier(1, 256);

            // ---- O = O * alpha + P V over this warp's value dims
            {
                const float a0 = sAlpha[gq], a1 = sAlpha[gq + 8];
#pragma unroll
                for (int n = 0; n < NTV; ++n) {
                    o[n][0] *= a0;
                    o[n][1] *= a0;
                    o[n][2] *= a1;
                    o[n][3] *= a1;
                }
#pragma unroll
                for (int ks = 0; ks < kTT / 16; ++ks) {
                    uint32_t pa[4], pb[4];
                    {
                        const uint32_t a =
                            p_base + (lane & 15) * (kPPitch * 2) + ks * 32 + (lane >> 4) * 16;
                        ldsm_x4(a, pa[0], pa[1], pa[2], pa[3]);
                        if constexpr (!P16)
                            ldsm_x4(a + 16 * kPPitch * 2, pb[0], pb[1], pb[2], pb[3]);
                    }
                    if constexpr (NTV == 1) {
                        const int kk = ks * 16 + (lane & 15);
                        uint32_t b0, b1;
                        ldsm_x2_t(vbase + tok_off(kk, V_IS_K ? KSLOT : VSLOT, V_IS_K ? KR : VR) +
                                      (dv0 / 8) * 16,
                                  b0, b1);
                        if constexpr (P16) {
                            mma_f16_16816(o[0], pa, bf16x2_to_f16x2(b0), bf16x2_to_f16x2(b1));
                        } else {
                            mma_bf16_16816(o[0], pa, b0, b1);
                            mma_bf16_16816(o[0], pb, b0, b1);
                        }
                    } else {
                        const int mi = lane >> 3, r8 = lane & 7;
                        const int kk = ks * 16 + (mi & 1) * 8 + r8;
                        const uint32_t rowaddr =
                            vbase + tok_off(kk, V_IS_K ? KSLOT : VSLOT, V_IS_K ? KR : VR);
#pragma unroll
                        for (int np = 0; np < NTV / 2; ++np) {
                            const int c = dv0 / 8 + np * 2 + (mi >> 1);
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4_t(rowaddr + c * 16, b0, b1, b2, b3);
                            if constexpr (P16) {
                                mma_f16_16816(o[2 * np], pa, bf16x2_to_f16x2(b0),
                                              bf16x2_to_f16x2(b1));
                                mma_f16_16816(o[2 * np + 1], pa, bf16x2_to_f16x2(b2),
                                              bf16x2_to_f16x2(b3));
                            } else {
                                mma_bf16_16816(o[2 * np], pa, b0, b1);
                                mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
                                mma_bf16_16816(o[2 * np], pb, b0, b1);
                                mma_bf16_16816(o[2 * np + 1], pb, b2, b3);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        gt += n_tiles;

        // ---- the item's output: final rows, a partial for combine_kernel, or (cluster
        // plans) the unnormalised rows kept here for the cluster merge
        if ((tid & 15) == 0) {
            sM[tid >> 4] = m_run;
            sL[tid >> 4] = l_run;
        }
        named_barrier(1, 256);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int row = gq + 8 * half;
            if (row >= G) continue;
            const float M = sM[row], l = sL[row];
            bool finite = true;
#pragma unroll
            for (int n = 0; n < NTV; ++n)
                finite &= isfinite(o[n][2 * half]) && isfinite(o[n][2 * half + 1]);
            if (P16 && !finite) set_status(p.status, SFA_DEV_FP16_RANGE);
            const int h = cur.g * G + row;
            if (p.cluster_merge) {
                float *sPart = reinterpret_cast<float *>(sRing);
#pragma unroll
                for (int n = 0; n < NTV; ++n)
                    *reinterpret_cast<float2 *>(sPart + row * DV + dv0 + n * 8 + 2 * tq) =
                        make_float2(o[n][2 * half], o[n][2 * half + 1]);
            } else if (p.n_split == 1) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                float *dst = p.O + ((int64_t)cur.i * p.h_q + h) * DV + dv0;
#pragma unroll
                for (int n = 0; n < NTV; ++n)
                    *reinterpret_cast<float2 *>(dst + n * 8 + 2 * tq) =
                        make_float2(o[n][2 * half] * inv, o[n][2 * half + 1] * inv);
                if (p.lse && warp == 0 && tq == 0)
                    p.lse[(int64_t)cur.i * p.h_q + h] = l > 0.f ? (M + log2f(l)) / kLog2e : -INFINITY;
            } else {
                const int64_t base =
                    (((int64_t)cur.i * p.h_kv + cur.g) * p.n_split + cur.split) * G + row;
                float *dst = p.part_o + base * DV + dv0;
#pragma unroll
                for (int n = 0; n < NTV; ++n)
                    *reinterpret_cast<float2 *>(dst + n * 8 + 2 * tq) =
                        make_float2(o[n][2 * half], o[n][2 * half + 1]);
                if (warp == 0 && tq == 0) {
                    p.part_ml[base * 2] = M;
                    p.part_ml[base * 2 + 1] = l;
                }
            }
        }
        named_barrier(1, 256);   // sM, sL and sItem are free for the next item
    }
    if (p.cluster_merge)   // one item per CTA in cluster plans
        cluster_merge<DV>(p, reinterpret_cast<float *>(sRing), sL, sM,
                          reinterpret_cast<float *>(sRing) + 16 * DV, cur.i, cur.g, tid);
}

// ---------------------------------------------------------------------------------------
// gather_rows_kernel -- the data movement of the attention and nothing else: the K (and V)
// rows of every query's attended list copied into a ring of shared-memory tiles of the layout
// above, each run of 4 consecutive rows (a kept block of cr >= 4, a run of the tail) as one bulk
// copy, issued by four producer warps (two slots of each tile each); a fifth warp waits for
// every tile, reads the first word of each attended row and releases the stage.  The sum of
// those words goes to *checksum, so that the copies cannot be dropped.  Its time is the data-movement ceiling of
// the attention on the same lists.
constexpr int kGatherThreads = 160;

template <int DKQ, int DV, bool V_IS_K>
__global__ void __launch_bounds__(kGatherThreads, 1)
    gather_rows_kernel(const AttnParams p, const int ns, const int bl_cap, uint32_t *checksum) {
    using Lay = Layout<DKQ, DV, V_IS_K>;
    constexpr int KR = Lay::KR, VR = Lay::VR, KSLOT = Lay::KSLOT, VSLOT = Lay::VSLOT;
    constexpr int STAGE = Lay::STAGE;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *sRing = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)ns * STAGE);
    uint64_t *full = bars, *empty = bars + ns;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * ns);
    int *sTok = const_cast<int *>(abort_flag) + 8;                   // [ns][kTT], MMA order
    int *sBlk = sTok + ns * kTT;                                     // [bl_cap]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 4);    // one expect-tx arrival per producer warp
            mbar_init(&empty[s], 1);   // the reading warp
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    const uint64_t deadline = global_timer_ns() + kWaitLimitNs;
    const bool k_dense = p.k_tok_stride == DKQ, v_dense = p.v_tok_stride == DV;
    const __nv_bfloat16 *Kb = reinterpret_cast<const __nv_bfloat16 *>(p.K);
    const __nv_bfloat16 *Vb = reinterpret_cast<const __nv_bfloat16 *>(p.V);
    uint32_t sum = 0;
    int gt = 0;
    for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
        const Item it = decompose(p, item);
        const ListInfo L = list_info(p, it.i, false);
        const int j0 = it.split * p.split_tokens;
        const int j1 = L.ok ? min(L.len, j0 + p.split_tokens) : 0;
        const int n_tiles = j0 < j1 ? (j1 - j0 + kTT - 1) / kTT : 0;
        int jb0 = 0;
        if (warp < 4) {
            if (n_tiles > 0) jb0 = load_block_list(p, it.i, L, j0, j1, sBlk, false, tid, 128);
            named_barrier(1, 128);   // the producers' block list
            const __nv_bfloat16 *Kseq =
                L.ok ? Kb + (int64_t)L.seq * p.k_seq_stride + (int64_t)it.g * DKQ : Kb;
            const __nv_bfloat16 *Vseq =
                V_IS_K ? Kseq
                       : (L.ok ? Vb + (int64_t)L.seq * p.v_seq_stride + (int64_t)it.g * DV : Vb);
            for (int t = 0; t < n_tiles; ++t) {
                const int g2 = gt + t, st = g2 % ns;
                wait_or_abort(&empty[st], ((uint32_t)(g2 / ns) & 1u) ^ 1u, deadline, abort_flag,
                              p.status);
                const int slot = warp * 2 + lane;   // lanes 0, 1: slots 2 warp, 2 warp + 1
                int n_valid = 0;
                if (lane < 2) {
                    int tok[kSlotRows];
                    int64_t row[kSlotRows];
                    bool run = !*abort_flag;
#pragma unroll
                    for (int r = 0; r < kSlotRows; ++r) {
                        tok[r] = token_at(p, L, j0 + t * kTT + slot * kSlotRows + r, j1, sBlk, jb0);
                        row[r] = tok[r];
                        n_valid += row[r] >= 0;
                        run &= row[r] >= 0 && row[r] == row[0] + r;
                        sTok[st * kTT + r * kSlots + slot] = tok[r];
                    }
                    uint8_t *kdst = sRing + (size_t)st * STAGE + slot * KSLOT;
                    uint8_t *vdst = sRing + (size_t)st * STAGE + Lay::KTILE + slot * VSLOT;
                    if (run && k_dense && (V_IS_K || v_dense)) {
                        bulk_load(kdst, Kseq + row[0] * p.k_tok_stride, kSlotRows * KR, &full[st]);
                        if constexpr (!V_IS_K)
                            bulk_load(vdst, Vseq + row[0] * p.v_tok_stride, kSlotRows * VR,
                                      &full[st]);
                    } else {
                        n_valid = 0;
#pragma unroll
                        for (int r = 0; r < kSlotRows; ++r)
                            if (row[r] >= 0 && !*abort_flag) {
                                ++n_valid;
                                bulk_load(kdst + r * KR, Kseq + row[r] * p.k_tok_stride, KR,
                                          &full[st]);
                                if constexpr (!V_IS_K)
                                    bulk_load(vdst + r * VR, Vseq + row[r] * p.v_tok_stride, VR,
                                              &full[st]);
                            }
                    }
                    if (*abort_flag) n_valid = 0;
                }
                n_valid += __shfl_xor_sync(0xFFFFFFFFu, n_valid, 1);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[st],
                                          (uint32_t)n_valid * (uint32_t)(KR + (V_IS_K ? 0 : VR)));
            }
            named_barrier(1, 128);   // every producer is done with the block list
        } else {   // the reading warp
            for (int t = 0; t < n_tiles; ++t) {
                const int g2 = gt + t, st = g2 % ns;
                wait_or_abort(&full[st], (uint32_t)(g2 / ns) & 1u, deadline, abort_flag, p.status);
                if (sTok[st * kTT + lane] >= 0)
                    sum += *reinterpret_cast<const uint32_t *>(sRing + (size_t)st * STAGE +
                                                               tok_off(lane, KSLOT, KR));
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
        }
        gt += n_tiles;
    }
    // no copy is in flight when the CTA leaves: the reading warp waited for every fill
    if (warp == 4) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
        if (lane == 0 && checksum) atomicAdd(checksum, sum);
    }
}

// ------------------------------------------------------------------------------ host side
// SFA_ATTEND_PV=bf16x2 in the environment (read at each call) makes P V run on bf16 operands
// with P as two bf16 halves instead of binary16 operands.
bool want_p16() {
    const char *e = getenv("SFA_ATTEND_PV");
    return !(e && strcmp(e, "bf16x2") == 0);
}

template <int DKQ, int DV, bool VK, bool P16>
constexpr auto kernel_of() {
    return attend_ws_kernel<DKQ, DV, VK, P16>;
}

// The most stages (up to kMaxStages, at least 3) that fit next to a block list of bl entries.
template <int DKQ, int DV, bool VK>
int stages_for(int bl) {
    for (int ns = kMaxStages; ns >= 3; --ns)
        if (Layout<DKQ, DV, VK>{ns, bl}.bytes() <= 227 * 1024) return ns;
    return 0;
}

// How many clusters of c CTAs of the kernel can be resident at once (0: none); asked once per
// (device, kernel, c, shared memory).
template <int DKQ, int DV, bool VK, bool P16>
int max_active_clusters(int c, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    {
        std::lock_guard<std::mutex> lock(mu);
        auto f = cache.find({dev, c, smem});
        if (f != cache.end()) return f->second;
    }
    auto fn = kernel_of<DKQ, DV, VK, P16>();
    int n = 0;
    if (ensure_max_dynamic_smem(fn)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c, 1, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
        cudaGetLastError();
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[{dev, c, smem}] = n;
    return n;
}

template <int DKQ, int DV, bool VK>
bool make_plan_shape(int n_q, int h_kv, int64_t n_kv_max, int cr, int dense, WsPlan *out) {
    const int64_t items = (int64_t)n_q * h_kv;
    const int64_t sms = device_sm_count();
    const int64_t tiles = (n_kv_max + kTT - 1) / kTT;
    int64_t ns = sms / items;
    const int64_t ns_cap = (tiles + kMinSplitTiles - 1) / kMinSplitTiles;
    if (ns > ns_cap) ns = ns_cap;
    if (ns < 1) ns = 1;
    auto fill = [&](int64_t n_split) {
        const int64_t per = (tiles + n_split - 1) / n_split;
        out->split_tokens = (int)(per * kTT);
        out->n_split = (int)((tiles + per - 1) / per);
    };
    auto bl_of = [&]() { return dense ? 0 : out->split_tokens / cr + 2; };
    out->cluster = 0;
    if (ns >= 2 && ns <= 16) {
        // a cluster of 2, 4 or 8 CTAs per item merges in place, when the item count fits
        const bool p16 = want_p16();
        for (int c = 8; c >= 2; c /= 2) {
            if (c > ns) continue;
            fill(c);
            if (out->n_split != c) continue;
            const int bl = bl_of();
            if (bl > kMaxBlkList) continue;
            const int st = stages_for<DKQ, DV, VK>(bl);
            if (!st) continue;
            const size_t smem = Layout<DKQ, DV, VK>{st, bl}.bytes();
            const int fit = p16 ? max_active_clusters<DKQ, DV, VK, true>(c, smem)
                                : max_active_clusters<DKQ, DV, VK, false>(c, smem);
            if (fit >= items) {
                out->cluster = c;
                out->grid = (int)(items * c);
                return true;
            }
        }
    }
    fill(ns);
    if (bl_of() > kMaxBlkList || !stages_for<DKQ, DV, VK>(bl_of())) return false;
    const int64_t n_items = items * out->n_split;
    out->grid = (int)(n_items < sms ? n_items : sms);
    return true;
}

template <int DKQ, int DV, bool VK>
int launch_shape(const AttnParams &p, const WsPlan &plan, cudaStream_t st) {
    const int bl = p.dense ? 0 : plan.split_tokens / p.cr + 2;
    const int ns = stages_for<DKQ, DV, VK>(bl);
    if (!ns) return SFA_ERR_UNSUPPORTED;
    const size_t smem = Layout<DKQ, DV, VK>{ns, bl}.bytes();
    auto fn = want_p16() ? kernel_of<DKQ, DV, VK, true>() : kernel_of<DKQ, DV, VK, false>();
    if (!ensure_max_dynamic_smem(fn)) return SFA_ERR_CUDA;
    const cudaError_t e =
        plan.cluster > 1
            ? launch_pdl_cluster(fn, dim3(plan.grid), dim3(kThreads), smem, st, plan.cluster, p,
                                 ns, bl)
            : launch_pdl(fn, dim3(plan.grid), dim3(kThreads), smem, st, p, ns, bl);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

template <int DKQ, int DV, bool VK>
int launch_gather(const AttnParams &p, const WsPlan &plan, uint32_t *checksum,
                  cudaStream_t st) {
    using Lay = Layout<DKQ, DV, VK>;
    const int bl = p.dense ? 0 : plan.split_tokens / p.cr + 2;
    int ns = 6;
    auto bytes = [&](int n) {
        return (size_t)n * Lay::STAGE + (size_t)(2 * n) * 8 + 32 + (size_t)n * kTT * 4 +
               (size_t)bl * 4 + 16;
    };
    while (ns > 2 && bytes(ns) > 227 * 1024) --ns;
    if (bytes(ns) > 227 * 1024) return SFA_ERR_UNSUPPORTED;
    auto fn = gather_rows_kernel<DKQ, DV, VK>;
    if (!ensure_max_dynamic_smem(fn)) return SFA_ERR_CUDA;
    AttnParams q = p;
    q.cluster_merge = 0;
    const int grid = q.n_items < device_sm_count() ? q.n_items : device_sm_count();
    if (launch_pdl(fn, dim3(grid), dim3(kGatherThreads), bytes(ns), st, q, ns, bl, checksum) !=
        cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

}  // namespace ws

int ws_gather_launch(const AttnParams &p, const WsPlan &plan, int dkq, int dv, bool has_v,
                     uint32_t *checksum, cudaStream_t st) {
    using namespace ws;
    if (dkq == 576 && dv == 512 && !has_v) return launch_gather<576, 512, true>(p, plan, checksum, st);
    if (dkq == 512 && dv == 512)
        return has_v ? launch_gather<512, 512, false>(p, plan, checksum, st)
                     : launch_gather<512, 512, true>(p, plan, checksum, st);
    return SFA_ERR_UNSUPPORTED;
}

bool ws_make_plan(int n_q, int h_kv, int dkq, int dv, bool has_v, int64_t n_kv_max, int cr,
                  int dense, WsPlan *out) {
    using namespace ws;
    if (dkq == 576 && dv == 512 && !has_v)
        return make_plan_shape<576, 512, true>(n_q, h_kv, n_kv_max, cr, dense, out);
    if (dkq == 512 && dv == 512)
        return has_v ? make_plan_shape<512, 512, false>(n_q, h_kv, n_kv_max, cr, dense, out)
                     : make_plan_shape<512, 512, true>(n_q, h_kv, n_kv_max, cr, dense, out);
    if (dkq == 128 && dv == 128)
        return has_v ? make_plan_shape<128, 128, false>(n_q, h_kv, n_kv_max, cr, dense, out)
                     : make_plan_shape<128, 128, true>(n_q, h_kv, n_kv_max, cr, dense, out);
    if (dkq == 64 && dv == 64)
        return has_v ? make_plan_shape<64, 64, false>(n_q, h_kv, n_kv_max, cr, dense, out)
                     : make_plan_shape<64, 64, true>(n_q, h_kv, n_kv_max, cr, dense, out);
    return false;
}

int ws_launch(const AttnParams &p, const WsPlan &plan, int dkq, int dv, bool has_v,
              cudaStream_t st) {
    using namespace ws;
    if (dkq == 576 && dv == 512 && !has_v) return launch_shape<576, 512, true>(p, plan, st);
    if (dkq == 512 && dv == 512)
        return has_v ? launch_shape<512, 512, false>(p, plan, st)
                     : launch_shape<512, 512, true>(p, plan, st);
    if (dkq == 128 && dv == 128)
        return has_v ? launch_shape<128, 128, false>(p, plan, st)
                     : launch_shape<128, 128, true>(p, plan, st);
    if (dkq == 64 && dv == 64)
        return has_v ? launch_shape<64, 64, false>(p, plan, st)
                     : launch_shape<64, 64, true>(p, plan, st);
    return SFA_ERR_UNSUPPORTED;
}

}  // namespace sfa
