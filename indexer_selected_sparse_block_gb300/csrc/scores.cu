// scores.cu -- the indexer score of every visible block (sfa_index_scores).
//
//   s_ib = sum_j w_ij * max(0, qidx_ij . kbar_b)
// (each head's dot product is rectified before the sum over heads, and a query meets only
// the blocks of its own sequence: llama.cpp commit "model: add Qwen3.8-Flash-Next (qwen4exp)",
// QSA paragraphs.)
//
// Design (sm_103a): the q.kbar contraction is a GEMM D[blocks x (queries*heads)] on the
// tcgen05 tensor cores with the fp32 accumulator in tensor memory.  The pooled key is stored
// as two bf16 halves (hi, lo) per row, so one bf16 MMA chain over K' = 2*d_idx against the
// duplicated query [q | q] yields q.(hi + lo) in fp32: selection-grade accuracy at bf16
// tensor-core rates.  The ReLU, the head weights and the head sum are applied while the
// accumulator is read back from tensor memory, so only the final score is written.
//
// One CTA = one tile of q_tile queries of one sequence x a run of 128-block tiles.
//   warp 0      TMA producer: one pipeline stage = one 128-row x 128-byte slab of Kbar
//               (16 KB, 128-byte swizzle); a tile is 2 (d_idx 64) or 4 (d_idx 128) slabs
//   warp 1      tensor-memory owner and single-thread MMA issuer (M = 128, N = q_tile*H pad 16)
//   warps 2..5  epilogue (2..13 for wide tiles): tcgen05.ld (lane = block), ReLU . w, head
//               sum, coalesced stores
// Two accumulator buffers in tensor memory let the epilogue of tile t overlap the MMAs of
// tile t + 1; for narrow tiles the producer fills the pipeline before the rest of the set-up.
// Every wait is bounded (SFA_DEV_TIMEOUT) and tensor memory is always released.
#include <mutex>

#include "sfa_common.cuh"

namespace sfa {
namespace {

constexpr int kBM = 128;               // blocks per tile (MMA M)
// Warps: the TMA producer, the MMA issuer and the epilogue warps -- four for narrow tiles
// (decode, four CTAs per SM), twelve for wide ones (prefill, one CTA per SM: three epilogue
// warps per scheduler hide each other's tensor-memory and arithmetic latency; pp2048's scores
// took 430 us with four, 281 with eight, 248 with twelve and 262 with sixteen).
template <bool WIDE>
struct Warps {
    static constexpr int kEpi = WIDE ? 12 : 4;
    static constexpr int kThreads = 64 + 32 * kEpi;
};
constexpr int kSlabBytes = kBM * 128;  // one pipeline stage
// The bounded mode's error bound per score: |s - a| <= e = kMargin * C_q * r_b (+ kAbs), with
// C_q = sum_j |w_j| |q_j|_2 and r_b = |lo_b|_2 + 2^-14 |hi_b|_2 from the pooling pass.  The
// exact difference of the two scores is at most C_q |lo_b|_2 (ReLU is 1-Lipschitz, the head
// sum is weighted by w, Cauchy-Schwarz per head); the fp32 rounding of the two MMA chains and
// of the head sums is below 2^-15 C_q |hi_b|_2, which the second term of r_b covers twice;
// kMargin covers the rounding of C_q and of e itself.
constexpr float kMargin = 1.0f + 9.765625e-4f;
constexpr float kAbs = 1e-30f;

struct ScoreParams {
    const __nv_bfloat16 *q_idx;
    const float *w;
    const int32_t *q_seq;
    const int32_t *q_pos;
    float *scores;       // exact mode: the scores; bounded mode: their lower bounds
    float *bounds;       // bounded mode: the upper bounds (else null)
    const float *kbar_r; // bounded mode: the per-block bound factors r_b
    int64_t kr_seq_stride;
    int32_t *status;
    int64_t score_stride;
    int64_t blk_cap;
    int64_t n_blk_max;
    int n_q, q_tile, n_seq, cr, N, stages, tiles_per_cta, tmem_cols;
};

template <int KP>
struct Layout {
    static constexpr int kSlabs = KP / 64;
};

// HI = false: K' = 2 d_idx over [hi | lo] against [q | q] (the exact score).  HI = true (the
// bounded mode): K' = d_idx over hi only against q; the score from hi, less and plus its error
// bound (from the norm of the hi row), gives the lower and upper bounds of the exact score
// (see sfa_index_scores_bounded).  WIDE: tiles of more than 32 columns (prefill), one CTA per
// SM with twelve epilogue warps and a five-stage ring; narrow tiles (decode) run four CTAs
// per SM with four epilogue warps each.
template <int KP, int H, bool HI, bool WIDE>
__global__ void __launch_bounds__(Warps<WIDE>::kThreads, WIDE ? 1 : 4)
    index_score_kernel(const __grid_constant__ CUtensorMap kbar_map, const ScoreParams p) {
    using L = Layout<HI ? KP / 2 : KP>;   // KP: the stored row (2 d_idx); L: the slabs read
    constexpr int kThreads = Warps<WIDE>::kThreads, kEpi = Warps<WIDE>::kEpi;
    constexpr int D = KP / 2;
    // The B operand holds each query row once (d_idx wide): the exact mode's chain over
    // [hi | lo] meets the same q rows for both halves, so its lo slabs reuse the hi slabs' B.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const int S = p.stages, N = p.N;
    uint8_t *sA = smem;                                    // S x kSlabBytes
    uint8_t *sB = sA + (size_t)S * kSlabBytes;             // N x D bf16, swizzled
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + (size_t)N * D * 2);
    uint64_t *full = bars, *empty = bars + S, *acc_full = bars + 2 * S,
             *acc_empty = bars + 2 * S + 2, *drain = bars + 2 * S + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_nblk = reinterpret_cast<int *>(tmem_slot + 2);  // [q_tile] visible blocks, -1 skip
    float *s_w = reinterpret_cast<float *>(s_nblk + 256);  // [q_tile * H]
    float *s_cq = s_w + p.q_tile * H;                       // [q_tile] sum_j |w_j| |q_j|_2

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = blockIdx.y * p.q_tile;
    const int nq_tile = min(p.q_tile, p.n_q - q0);

    // ---------------------------------------------------------------- set-up (all warps)
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], kEpi);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) prefetch_tensormap(&kbar_map);
    if (warp == 1) {
        tmem_alloc(tmem_slot, (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    pdl_wait();   // global memory from here on
    const int seq0 = p.q_seq[q0];
    const uint64_t deadline = global_timer_ns() + kWaitLimitNs;
    // For narrow tiles the producer fills the pipeline before the rest of the set-up: its tile
    // range needs only the visible block counts of the tile's queries (the rule of s_nblk).
    int primed = 0;
    if (warp == 0 && N <= 32) {   // narrow (decode) tiles stream; wide ones measured no gain
        int nbw = 0;
        for (int qq = lane; qq < nq_tile; qq += 32) {
            const int s = p.q_seq[q0 + qq], pos = p.q_pos[q0 + qq];
            if (s == seq0 && s >= 0 && s < p.n_seq && pos >= 0)
                nbw = max(nbw, (int)min(min((int64_t)(pos + 1) / p.cr, p.n_blk_max), p.blk_cap));
        }
        nbw = __reduce_max_sync(0xFFFFFFFFu, nbw);
        const int tb = blockIdx.x * p.tiles_per_cta;
        const int mine = max(0, min(p.tiles_per_cta, (nbw + kBM - 1) / kBM - tb));
        if (lane == 0) {
            const int n_loads = mine * L::kSlabs;
            const int64_t r0 = (int64_t)seq0 * p.blk_cap;
            for (; primed < S && primed < n_loads; ++primed) {
                mbar_arrive_expect_tx(&full[primed], kSlabBytes);
                const int tile = primed / L::kSlabs, sl = primed % L::kSlabs;
                tma_load_2d(sA + (size_t)primed * kSlabBytes, &kbar_map, sl * 64,
                            (int32_t)(r0 + (int64_t)(tb + tile) * kBM), &full[primed]);
            }
        }
    }
    for (int qq = threadIdx.x; qq < p.q_tile; qq += kThreads) {
        int nb = -1;
        if (qq < nq_tile) {
            const int qi = q0 + qq;
            const int s = p.q_seq[qi], pos = p.q_pos[qi];
            if (s != seq0 || s < 0 || s >= p.n_seq || pos < 0) {
                set_status(p.status, SFA_DEV_BAD_QUERY);
            } else {
                const int64_t b = min((int64_t)(pos + 1) / p.cr, p.n_blk_max);
                nb = (int)min(b, p.blk_cap);
            }
        }
        s_nblk[qq] = nb;
    }
    for (int e = threadIdx.x; e < p.q_tile * H; e += kThreads) {
        const int qq = e / H;
        s_w[e] = qq < nq_tile ? p.w[(int64_t)(q0 + qq) * H + (e % H)] : 0.f;
    }
    // B operand: row n = (query qq, head j), its d_idx dims in slabs of 64; 16-byte chunks,
    // 128-byte swizzle.
    for (int e = threadIdx.x; e < N * (D / 8); e += kThreads) {
        const int n = e / (D / 8), c = e % (D / 8);
        const int qq = n / H, j = n % H;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (qq < nq_tile && n < p.q_tile * H)
            v = *reinterpret_cast<const uint4 *>(p.q_idx + ((int64_t)(q0 + qq) * H + j) * D + c * 8);
        const int slab = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4 *>(sB + (size_t)slab * N * 128 + n * 128 + ((cc ^ (n & 7)) << 4)) =
            v;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int max_nb = 0;
    for (int qq = 0; qq < nq_tile; ++qq) max_nb = max(max_nb, s_nblk[qq]);
    const int n_tiles_q = (max_nb + kBM - 1) / kBM;
    const int t_begin = blockIdx.x * p.tiles_per_cta;
    const int my_tiles = max(0, min(p.tiles_per_cta, n_tiles_q - t_begin));
    const int64_t row0 = (int64_t)seq0 * p.blk_cap;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && my_tiles > 0) {
            int issued = primed;
            const int n_loads = my_tiles * L::kSlabs;
            for (int it = primed; it < n_loads && !*abort_flag; ++it) {
                const int st = it % S;
                if (!mbar_wait(&empty[st], ((it / S) & 1) ^ 1, deadline)) {
                    set_status(p.status, SFA_DEV_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[st], kSlabBytes);
                const int tile = it / L::kSlabs, sl = it % L::kSlabs;
                const int32_t y = (int32_t)(row0 + (int64_t)(t_begin + tile) * kBM);
                tma_load_2d(sA + (size_t)st * kSlabBytes, &kbar_map, sl * 64, y, &full[st]);
                ++issued;
            }
            // never leave a copy in flight: wait (bounded) for the last load of each stage
            for (int it = max(0, issued - S); it < issued; ++it)
                mbar_wait(&full[it % S], (it / S) & 1, deadline + kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && my_tiles > 0) {
            const uint32_t idesc = idesc_bf16_f32(kBM, N);
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
            int issued = 0, ld = 0;
            bool ok = true;
            for (int it = 0; it < my_tiles && ok && !*abort_flag; ++it) {
                const int acc = it & 1;
                if (!mbar_wait(&acc_empty[acc], ((it >> 1) & 1) ^ 1, deadline)) {
                    ok = false;
                    break;
                }
                const uint32_t d = tmem_base + (uint32_t)(acc * N);
                for (int sl = 0; sl < L::kSlabs; ++sl, ++ld) {
                    const int st = ld % S;
                    if (!mbar_wait(&full[st], (ld / S) & 1, deadline)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_st = a0 + st * kSlabBytes;
                    const uint32_t b_sl = b0 + (sl % (D / 64)) * (N * 128);   // hi and lo: the same q
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16(d, sw128_kmajor_desc(a_st + kk * 32),
                                    sw128_kmajor_desc(b_sl + kk * 32), idesc,
                                    (sl > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&empty[st]);
                }
                if (!ok) break;
                tc_commit(&acc_full[acc]);
                ++issued;
            }
            if (!ok) {
                set_status(p.status, SFA_DEV_TIMEOUT);
                *abort_flag = 1;
                tc_commit(drain);  // arrives once every MMA issued so far is done
                mbar_wait(drain, 0, deadline + kWaitLimitNs);
            } else if (issued > 0) {  // tensor memory may only be released once the MMAs are done
                const int last = issued - 1;
                mbar_wait(&acc_full[last & 1], (last >> 1) & 1, deadline + kWaitLimitNs);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue warps
        // Warp w reads tensor-memory lanes 32 (w % 4) .. + 31 (its quarter of the tile's
        // blocks); the kEpi / 4 warps of a quarter take its column batches in turn.
        const int ew = warp - 2;
        const int quarter = warp & 3;
        constexpr int kParts = kEpi / 4;
        const int part = ew >> 2;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const int ncols = nq_tile * H;
        if (HI) {
            // C_q = sum_j |w_j| |q_j|_2, from the query rows of the B operand in shared memory
            // (the sum of squares of a row covers all its 16-byte chunks, so the swizzle does
            // not matter): no global round trip before the epilogue's first tile.  (Computed
            // from global memory in the set-up, it held every warp for 3.5 us per launch.)
            constexpr int kCpr = D / 8;         // 16-byte chunks per B row
            constexpr int kHpp = 32 / kCpr;     // heads per warp pass
            for (int qq = ew; qq < nq_tile; qq += kEpi) {
                float c = 0.f;
#pragma unroll
                for (int j0 = 0; j0 < H; j0 += kHpp) {
                    const int j = j0 + lane / kCpr, cc = lane % kCpr;
                    float ss = 0.f;
                    if (j < H) {
                        const int n = qq * H + j;
                        const uint4 v = *reinterpret_cast<const uint4 *>(
                            sB + (size_t)(cc >> 3) * N * 128 + n * 128 +
                            (((cc & 7) ^ (n & 7)) << 4));
                        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float e0 = __uint_as_float(u[k] << 16);
                            const float e1 = __uint_as_float(u[k] & 0xFFFF0000u);
                            ss = fmaf(e0, e0, fmaf(e1, e1, ss));
                        }
                    }
#pragma unroll
                    for (int o = 1; o < kCpr; o <<= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
                    if (cc == 0 && j < H) c = fmaf(fabsf(s_w[qq * H + j]), sqrtf(ss), c);
                }
#pragma unroll
                for (int o = kCpr; o < 32; o <<= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
                if (lane == 0) s_cq[qq] = c;
            }
            named_barrier(1, 32 * kEpi);   // the epilogue warps
        }
        // bounded mode: this thread's block's bound factor, loaded one tile ahead so that its
        // latency overlaps the tile before
        const float *kr = HI ? p.kbar_r + (int64_t)seq0 * p.kr_seq_stride + quarter * 32 + lane
                             : nullptr;
        auto load_rb = [&](int it) {
            const int64_t b = (int64_t)(t_begin + it) * kBM + quarter * 32 + lane;
            return (HI && it < my_tiles && b < p.n_blk_max)
                       ? __ldg(kr + (int64_t)(t_begin + it) * kBM)
                       : 0.f;
        };
        float rb_next = load_rb(0);
        for (int it = 0; it < my_tiles; ++it) {
            const int acc = it & 1;
            if (*abort_flag) break;
            const int64_t b = (int64_t)(t_begin + it) * kBM + quarter * 32 + lane;
            const float rb = rb_next;
            rb_next = load_rb(it + 1);
            if (!mbar_wait(&acc_full[acc], (it >> 1) & 1, deadline)) {
                set_status(p.status, SFA_DEV_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            // 16 columns per wait on tensor memory (batches of 32 or 64 measured slower).  The
            // queries of a batch are summed with no branch between them (a query past the tile
            // reads the last query's weights and stores nothing), so their head sums interleave.
            constexpr int kCB = 16;
            constexpr int kQB = kCB / H;   // queries per batch
            static_assert(kCB % H == 0 && H % 4 == 0, "whole queries per column batch");
            for (int c0 = part * kCB; c0 < ncols; c0 += kParts * kCB) {
                uint32_t r[kCB / 16][16];
#pragma unroll
                for (int u = 0; u < kCB / 16; ++u)
                    if (c0 + 16 * u < ncols)
                        tmem_ld16(tmem_base + lane_addr + (uint32_t)(acc * N + c0 + 16 * u), r[u]);
                tmem_ld_wait();
                float sq[kQB];
#pragma unroll
                for (int g = 0; g < kQB; ++g) {
                    const int qq = min(c0 / H + g, nq_tile - 1);
                    const float4 *w4 = reinterpret_cast<const float4 *>(s_w + qq * H);
                    float s = 0.f;
#pragma unroll
                    for (int j4 = 0; j4 < H / 4; ++j4) {
                        const float4 v = w4[j4];
                        const float wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int col = g * H + 4 * j4 + k;
                            s = fmaf(wv[k], fmaxf(__uint_as_float(r[col / 16][col % 16]), 0.f), s);
                        }
                    }
                    sq[g] = s;
                }
#pragma unroll
                for (int g = 0; g < kQB; ++g) {
                    const int qq = c0 / H + g;
                    if (qq < nq_tile && b < s_nblk[qq]) {
                        const int64_t o = (int64_t)(q0 + qq) * p.score_stride + b;
                        if (HI) {
                            const float e = fmaf(kMargin * s_cq[qq], rb, kAbs);
                            p.scores[o] = sq[g] - e;   // the hi + lo score lies in [s - e, s + e]
                            p.bounds[o] = sq[g] + e;
                        } else {
                            p.scores[o] = sq[g];
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
    }
}

int pow2_at_least(int v) {
    int r = 32;
    while (r < v) r <<= 1;
    return r;
}

template <int KP, int H, bool HI, bool WIDE>
int launch_shape(const CUtensorMap &map, ScoreParams p, int n_qtiles, int n_blk_tiles,
                 cudaStream_t stream) {
    const size_t b_bytes = (size_t)p.N * (KP / 2) * 2;   // each query row once
    // Narrow B tiles (decode) are HBM-bound streams: four CTAs per SM, three stages each,
    // overlap four producer -> MMA -> epilogue chains (measured 6% faster than two CTAs of six
    // stages, 10% faster than one of thirteen); wide ones (prefill) are tensor-bound: one CTA
    // per SM with a deep pipeline.
    const int per_sm = WIDE ? 1 : 4;
    const size_t budget = per_sm == 4 ? 55 * 1024 : 220 * 1024;
    const size_t misc = 1024 + 8 * (2 * 16 + 5) + 8 + 256 * 4 + (size_t)p.q_tile * (H + 1) * 4;
    if (budget < b_bytes + misc + kSlabBytes) return SFA_ERR_UNSUPPORTED;
    int stages = (int)((budget - b_bytes - misc) / kSlabBytes);
    if (stages > 16) stages = 16;
    // Wide tiles: five stages (a tile and a slab) measured faster than nine (297 against
    // 318 us on pp2048's scores); three starve the tensor cores.
    if (WIDE && stages > 5) stages = 5;
    p.stages = stages;
    const size_t smem = 1024 + (size_t)stages * kSlabBytes + b_bytes + 8 * (2 * stages + 5) + 8 +
                        256 * 4 + (size_t)p.q_tile * (H + 1) * 4;
    if (!ensure_max_dynamic_smem(index_score_kernel<KP, H, HI, WIDE>)) return SFA_ERR_CUDA;
    // One wave: the block tiles of each query tile are split over as many CTAs as the
    // resident slots allow.
    const int slots = per_sm * device_sm_count();
    int cta_per_qtile = slots / n_qtiles;
    if (cta_per_qtile > n_blk_tiles) cta_per_qtile = n_blk_tiles;
    if (cta_per_qtile < 1) cta_per_qtile = 1;
    p.tiles_per_cta = (n_blk_tiles + cta_per_qtile - 1) / cta_per_qtile;
    const int grid_x = (n_blk_tiles + p.tiles_per_cta - 1) / p.tiles_per_cta;
    if (launch_pdl(index_score_kernel<KP, H, HI, WIDE>, dim3(grid_x, n_qtiles),
                   dim3(Warps<WIDE>::kThreads), smem, stream, map, p) != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}
template <int KP, int H, bool HI>
int launch(const CUtensorMap &map, ScoreParams p, int n_qtiles, int n_blk_tiles,
           cudaStream_t stream) {
    return p.N <= 32 ? launch_shape<KP, H, HI, false>(map, p, n_qtiles, n_blk_tiles, stream)
                     : launch_shape<KP, H, HI, true>(map, p, n_qtiles, n_blk_tiles, stream);
}

}  // namespace
}  // namespace sfa

namespace sfa {
namespace {

int run_scores(const void *q_idx, const float *w, const int32_t *q_seq, const int32_t *q_pos,
               int n_q, int q_group, int h_idx, int d_idx, int compress_ratio, const void *Kbar,
               int64_t kbar_seq_stride, const float *kbar_r, int64_t kr_seq_stride, int n_seq,
               int64_t n_blk_max, float *scores, float *bounds, int64_t score_stride,
               int32_t *dev_status, cudaStream_t st) {
    const bool hi = bounds != nullptr;
    if (hi && (!kbar_r || kr_seq_stride < n_blk_max)) return SFA_ERR_INVALID_ARG;
    if (!q_idx || !w || !q_seq || !q_pos || !Kbar || !scores) return SFA_ERR_INVALID_ARG;
    if (n_q < 0 || q_group < 1 || n_seq < 1 || compress_ratio < 1 || n_blk_max < 0)
        return SFA_ERR_INVALID_ARG;
    if (d_idx != 64 && d_idx != 128) return SFA_ERR_UNSUPPORTED;
    if (h_idx != 4 && h_idx != 8 && h_idx != 16) return SFA_ERR_UNSUPPORTED;
    const int KP = 2 * d_idx;
    if (kbar_seq_stride % KP != 0 || kbar_seq_stride <= 0) return SFA_ERR_INVALID_ARG;
    const int64_t blk_cap = kbar_seq_stride / KP;
    if (n_blk_max > blk_cap || n_blk_max > score_stride) return SFA_ERR_INVALID_ARG;
    if (!aligned16(q_idx) || !aligned16(Kbar) || !aligned16(scores)) return SFA_ERR_INVALID_ARG;
    if (n_q == 0 || n_blk_max == 0) return SFA_OK;
    if ((int64_t)n_seq * blk_cap > 0x7FFFFFFFll) return SFA_ERR_UNSUPPORTED;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return SFA_ERR_CUDA;

    // Queries per tile: the largest power of two that divides q_group and fits N <= 256 (the
    // B tile then takes 64 KB of the 220 KB budget at d_idx = 128, leaving nine pooled-key
    // stages; pp2048's scores ran 453 us with N capped at 128 there, 429 us at 256).
    const int n_cap = 256;
    int q_tile = 1;
    while (q_tile * 2 * h_idx <= n_cap && q_group % (q_tile * 2) == 0) q_tile *= 2;
    ScoreParams p{};
    p.q_idx = reinterpret_cast<const __nv_bfloat16 *>(q_idx);
    p.w = w;
    p.q_seq = q_seq;
    p.q_pos = q_pos;
    p.scores = scores;
    p.bounds = bounds;
    p.kbar_r = kbar_r;
    p.kr_seq_stride = kr_seq_stride;
    p.status = dev_status;
    p.score_stride = score_stride;
    p.blk_cap = blk_cap;
    p.n_blk_max = n_blk_max;
    p.n_q = n_q;
    p.q_tile = q_tile;
    p.n_seq = n_seq;
    p.cr = compress_ratio;
    p.N = ((q_tile * h_idx + 15) / 16) * 16;
    p.tmem_cols = pow2_at_least(2 * p.N);

    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)KP, (cuuint64_t)(n_seq * blk_cap)};
    const cuuint64_t gstride[1] = {(cuuint64_t)KP * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estride[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(Kbar), gdim, gstride,
            box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SFA_ERR_INVALID_ARG;

    const int n_qtiles = (n_q + q_tile - 1) / q_tile;
    if (n_qtiles > 65535) return SFA_ERR_UNSUPPORTED;
    const int n_blk_tiles = (int)((n_blk_max + kBM - 1) / kBM);
#define SFA_SCORES_LAUNCH(KP_, H_)                                                            \
    return hi ? launch<KP_, H_, true>(map, p, n_qtiles, n_blk_tiles, st)                      \
              : launch<KP_, H_, false>(map, p, n_qtiles, n_blk_tiles, st)
    if (d_idx == 64 && h_idx == 4) SFA_SCORES_LAUNCH(128, 4);
    if (d_idx == 64 && h_idx == 8) SFA_SCORES_LAUNCH(128, 8);
    if (d_idx == 64 && h_idx == 16) SFA_SCORES_LAUNCH(128, 16);
    if (d_idx == 128 && h_idx == 4) SFA_SCORES_LAUNCH(256, 4);
    if (d_idx == 128 && h_idx == 8) SFA_SCORES_LAUNCH(256, 8);
    SFA_SCORES_LAUNCH(256, 16);
#undef SFA_SCORES_LAUNCH
}

}  // namespace
}  // namespace sfa

extern "C" int sfa_index_scores(const void *q_idx, const float *w, const int32_t *q_seq,
                                const int32_t *q_pos, int n_q, int q_group, int h_idx,
                                int d_idx, int compress_ratio, const void *Kbar,
                                int64_t kbar_seq_stride, int n_seq, int64_t n_blk_max,
                                float *scores, int64_t score_stride, int32_t *dev_status,
                                sfa_stream_t stream) {
    return sfa::run_scores(q_idx, w, q_seq, q_pos, n_q, q_group, h_idx, d_idx, compress_ratio,
                           Kbar, kbar_seq_stride, nullptr, 0, n_seq, n_blk_max, scores, nullptr,
                           score_stride, dev_status, (cudaStream_t)stream);
}

extern "C" int sfa_index_scores_bounded(const void *q_idx, const float *w, const int32_t *q_seq,
                                        const int32_t *q_pos, int n_q, int q_group, int h_idx,
                                        int d_idx, int compress_ratio, const void *Kbar,
                                        int64_t kbar_seq_stride, const float *Kbar_r,
                                        int64_t kr_seq_stride, int n_seq, int64_t n_blk_max,
                                        float *lower, float *upper, int64_t score_stride,
                                        int32_t *dev_status, sfa_stream_t stream) {
    if (!upper || !sfa::aligned16(upper)) return SFA_ERR_INVALID_ARG;
    return sfa::run_scores(q_idx, w, q_seq, q_pos, n_q, q_group, h_idx, d_idx, compress_ratio,
                           Kbar, kbar_seq_stride, Kbar_r, kr_seq_stride, n_seq, n_blk_max, lower,
                           upper, score_stride, dev_status, (cudaStream_t)stream);
}
