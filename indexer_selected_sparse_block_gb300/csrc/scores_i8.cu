// scores_i8.cu -- the bound pass of the bounded selection on 8-bit copies of the pooled keys
// (sfa_quantize_pooled_keys_i8, sfa_index_scores_bounded_i8).
//
// The bounded selection needs, for every visible block, an interval that holds the exact
// score s_ib = sum_j w_ij max(0, q_ij . m_b), m_b = hi_b + lo_b (the value the exact scores
// use; llama.cpp commit "model: add Qwen3.8-Flash-Next (qwen4exp)", QSA paragraphs).  Here
// the interval comes from a third copy of the pooled key, 8-bit codes with one fp32 scale per
// row,
//   sc_b = max_i |m_bi| / 127,   c_bi = round(m_bi / sc_b) in [-127, 127]  (stored as c + 128),
//   r_b  = (|m_b - sc_b c_b|_2 + 2^-14 sc_b |c_b|_2) (1 + 2^-16),
// so that the pass reads d_idx bytes per block (the hi-only pass reads 2 d_idx):
//   q~_ij = binary16(q_ij)     (clamped to +-65504)
//   a_bj = q~_ij . c_b         (binary16 x small integers on the tensor cores: exact products,
//                               fp32 sums)
//   s~_b = sc_b sum_j w_ij max(0, a_bj)
//   |s_ib - s~_b| <= C_i r_b + D_i 127 sqrt(d_idx) sc_b,
//   C_i = sum_j |w_ij| |q_ij|_2,  D_i = sum_j |w_ij| |q_ij - q~_ij|_2
// (ReLU is 1-Lipschitz and sc_b >= 0; per head |q.m - q~.sc c| <= |q|_2 |m - sc c|_2 +
// |q - q~|_2 sc |c|_2 by Cauchy-Schwarz, with |c|_2 <= 127 sqrt(d_idx); the fp32 rounding of
// this chain, of the scale products and of the exact hi + lo chain together stays below
// 2^-15 C_i sc_b |c_b|_2, which the second term of r_b covers twice).  lower = s~ - e,
// upper = s~ + e with e = (1 + 2^-10) (C_i r_b + D_i 127 sqrt(d_idx) sc_b) + 1e-30 then bracket
// the exact score like the hi-only bounds, and sfa_topk_blocks_refine takes them unchanged.
// The codes are looser than the hi halves (about twice as many blocks survive the bounds),
// and the pass reads half the bytes.
//
// The score kernel streams 128-row tiles of codes with 2-D TMA into a ring of shared-memory
// stages filled by one producer warp; four warps each take 32 rows through mma.sync m16n8k16
// (codes widened to binary16 in registers, exactly, with one byte permute and one paired
// subtraction per pair), with the k order permuted so that each thread's A elements of a
// k-step are four consecutive bytes and its B elements four consecutive query elements.
// Widening to bf16 instead (fp32 arithmetic and a pack per pair) ran 20% slower: the pass is
// bound by its instruction issue as much as by its bytes.  Every wait is bounded
// (SFA_DEV_TIMEOUT).
#include <mutex>

#include "sfa_common.cuh"

namespace sfa {
namespace {

constexpr float kMarginI8 = 1.0f + 9.765625e-4f;   // 1 + 2^-10
constexpr float kAbsI8 = 1e-30f;

// ---------------------------------------------------------------------------------- codes
// One warp per pooled row; lane l holds elements [E l, E l + E) (E = d_idx / 32).
template <int D>
__global__ void __launch_bounds__(256)
    quantize_pooled_i8_kernel(const __nv_bfloat16 *__restrict__ Kbar, int64_t kbar_seq_stride,
                              int64_t blk_begin, int64_t n_rows, int8_t *__restrict__ K8,
                              int64_t k8_seq_stride, float *__restrict__ sr,
                              int64_t sr_seq_stride) {
    constexpr int E = D / 32;
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= n_rows) return;
    const int64_t seq = blockIdx.y, b = blk_begin + row;
    const __nv_bfloat16 *hi = Kbar + seq * kbar_seq_stride + b * (2 * D) + E * lane;
    float m[E];
    float mx = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        // hi + lo is exact in fp32: two bf16 values whose significands span at most 17 bits
        m[e] = __bfloat162float(hi[e]) + __bfloat162float(hi[D + e]);
        mx = fmaxf(mx, fabsf(m[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    const float sc = mx / 127.f;
    float res2 = 0.f, c2 = 0.f;
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        float c = sc > 0.f ? rintf(m[e] / sc) : 0.f;
        c = fminf(fmaxf(c, -127.f), 127.f);
        const float rr = fmaf(-sc, c, m[e]);   // the residual with one rounding
        res2 = fmaf(rr, rr, res2);
        c2 = fmaf(c, c, c2);
        packed |= (uint32_t)((int)c + 128) << (8 * e);   // offset binary: c + 128
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        res2 += __shfl_xor_sync(0xFFFFFFFFu, res2, o);
        c2 += __shfl_xor_sync(0xFFFFFFFFu, c2, o);
    }
    int8_t *dst = K8 + seq * k8_seq_stride + b * D + E * lane;
    if constexpr (E == 4)
        *reinterpret_cast<uint32_t *>(dst) = packed;
    else
        *reinterpret_cast<uint16_t *>(dst) = (uint16_t)packed;
    if (lane == 0) {
        float *o = sr + seq * sr_seq_stride + 2 * b;
        o[0] = sc;
        o[1] = (sqrtf(res2) + 6.103515625e-05f * sc * sqrtf(c2)) * (1.0f + 1.52587890625e-05f);
    }
}

}  // namespace
}  // namespace sfa

namespace sfa {
namespace {

// ---------------------------------------------------------------------------------- scores
constexpr int kI8Rows = 128;                       // blocks per tile
constexpr int kI8Warps = 4;                        // compute warps, 32 rows each
constexpr int kI8Threads = (kI8Warps + 1) * 32;    // + one producer warp

struct I8Params {
    const __nv_bfloat16 *q_idx;   // [n_q][H][D]
    const float *w;               // [n_q][H]
    const int32_t *q_seq, *q_pos;
    const float *sr;              // [n_seq][sr_seq_stride]: (scale, bound factor) per block
    int64_t sr_seq_stride;
    float *lower, *upper;
    int64_t score_stride;
    int32_t *status;
    int64_t blk_cap, n_blk_max;
    int n_q, n_seq, cr, stages, tiles_per_cta;
};

// Where linear byte `lin` of a tile lands in shared memory.  d_idx = 128: TMA writes the
// tile with the 128-byte swizzle (tile base 1024-byte aligned; the 16-byte chunk index is
// XORed with the row index mod 8), so that the eight threads of a quarter-warp, which read
// chunks 2t + h of rows g and g + 1, hit distinct banks.  d_idx = 64: no swizzle (chunk t of
// rows g and g + 1 already spans all banks).
template <int D>
__device__ __forceinline__ uint32_t tile_off(uint32_t lin) {
    if constexpr (D == 128) return lin ^ (((lin >> 7) & 7u) << 4);
    return lin;
}

// Two 8-bit codes (bytes e, e + 1 of u, each code + 128) as a binary16 pair, exactly: a byte
// placed under the binary16 exponent of 1024 reads as 1024 + (code + 128), and one paired
// subtraction of 1152 leaves the code.
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t u, uint32_t e) {
    const uint32_t x = __byte_perm(u, 0x64646464u, e == 0 ? 0x5140u : 0x7362u);
    const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&x), __float2half2_rn(1152.f));
    return *reinterpret_cast<const uint32_t *>(&r);
}

template <int D, int H>
__global__ void __launch_bounds__(kI8Threads)
    index_score_i8_kernel(const __grid_constant__ CUtensorMap k8_map, const I8Params p) {
    constexpr int NT = (H + 7) / 8;   // n8 tiles of heads
    constexpr int KS = D / 16;        // k-steps
    constexpr int BPT = D / 4;        // bytes of a row per thread (its A elements)
    constexpr int TB = kI8Rows * D;   // bytes per tile
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sA = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const int S = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(sA + (size_t)S * TB), *empty = full + S;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + S);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.y;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kI8Warps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kI8Warps && lane == 0) prefetch_tensormap(&k8_map);
    __syncthreads();
    pdl_wait();   // global memory from here on
    const int seq = p.q_seq[i], pos = p.q_pos[i];
    int nb = 0;
    if (seq < 0 || seq >= p.n_seq || pos < 0) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_status(p.status, SFA_DEV_BAD_QUERY);
    } else {
        nb = (int)min(min((int64_t)(pos + 1) / p.cr, p.n_blk_max), p.blk_cap);
    }
    const int n_tiles = (nb + kI8Rows - 1) / kI8Rows;
    const int t_begin = blockIdx.x * p.tiles_per_cta;
    const int my = max(0, min(p.tiles_per_cta, n_tiles - t_begin));
    const uint64_t deadline = global_timer_ns() + kWaitLimitNs;

    if (warp == kI8Warps) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && my > 0) {
            int issued = 0;
            const int32_t row0 = (int32_t)((int64_t)seq * p.blk_cap + (int64_t)t_begin * kI8Rows);
            for (int it = 0; it < my && !*abort_flag; ++it) {
                const int st = it % S;
                if (it >= S && !mbar_wait(&empty[st], ((it / S) - 1) & 1, deadline)) {
                    set_status(p.status, SFA_DEV_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[st], TB);
                tma_load_2d(sA + (size_t)st * TB, &k8_map, 0, row0 + it * kI8Rows, &full[st]);
                ++issued;
            }
            // never leave a copy in flight: wait (bounded) for the last load of each stage
            for (int it = max(0, issued - S); it < issued; ++it)
                mbar_wait(&full[it % S], (it / S) & 1, deadline + kWaitLimitNs);
        }
        return;
    }

    // ------------------------------------------------------------ compute warps
    const int g = lane >> 2, t = lane & 3;
    // B fragments: the query of head n = 8 nt + g in binary16 (q~ = fp16(q), clamped to
    // +-65504); in k-step ks, b0 holds query elements BPT t + 4 ks + {0, 1} and b1 elements
    // BPT t + 4 ks + {2, 3} -- the same bytes the A fragments take from a row (the k order of
    // both operands permuted alike).  The codes widen to binary16 exactly with two
    // instructions per pair (below), and binary16 x codes products are exact in the fp32 sums.
    // Per query: C_q = sum_n |w_n| |q_n|_2 and Dq = sum_n |w_n| |q_n - q~_n|_2 (the rounding of
    // q to binary16, below 2^-11 |q_n| in range).
    uint32_t bq[NT][KS][2];
    float wv[NT][2];
    float cq = 0.f, dq = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int n = 8 * nt + g;
        const __nv_bfloat16 *qr = p.q_idx + ((int64_t)i * H + (n < H ? n : 0)) * D + BPT * t;
        float ss = 0.f, d2 = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint2 v = make_uint2(0u, 0u);
            if (n < H) v = *reinterpret_cast<const uint2 *>(qr + 4 * ks);
            const uint32_t u[2] = {v.x, v.y};
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float e0 = __uint_as_float(u[k] << 16);
                const float e1 = __uint_as_float(u[k] & 0xFFFF0000u);
                ss = fmaf(e0, e0, fmaf(e1, e1, ss));
                const float h0 = fminf(fmaxf(e0, -65504.f), 65504.f);
                const float h1 = fminf(fmaxf(e1, -65504.f), 65504.f);
                const uint32_t hh = pack_f16(h0, h1);
                const __half2 hv = *reinterpret_cast<const __half2 *>(&hh);
                const float r0 = e0 - __low2float(hv), r1 = e1 - __high2float(hv);
                d2 = fmaf(r0, r0, fmaf(r1, r1, d2));
                bq[nt][ks][k] = hh;
            }
        }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {   // over t: the whole head in the quad
            ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
            d2 += __shfl_xor_sync(0xFFFFFFFFu, d2, o);
        }
        const float wn = (t == 0 && n < H) ? fabsf(p.w[(int64_t)i * H + n]) : 0.f;
        float c = wn * sqrtf(ss), d = wn * sqrtf(d2);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
            d += __shfl_xor_sync(0xFFFFFFFFu, d, o);
        }
        cq += c;
        dq += d;
        const int h0 = 8 * nt + 2 * t;   // this thread's accumulator columns
        wv[nt][0] = h0 < H ? p.w[(int64_t)i * H + h0] : 0.f;
        wv[nt][1] = h0 + 1 < H ? p.w[(int64_t)i * H + h0 + 1] : 0.f;
    }
    // |q . m - q~ . sc c| <= |q|_2 |m - sc c|_2 + |q - q~|_2 sc |c|_2, sc |c|_2 <= 127 sqrt(D) sc
    const float dq_row = dq * (D == 128 ? 1437.0f : 1016.0f);

    // (scale, bound factor) of this thread's four rows of a tile, loaded one tile ahead
    const float *srs = p.sr + (int64_t)(nb > 0 ? seq : 0) * p.sr_seq_stride;
    auto load_sr = [&](int it, float2 (&o)[2][2]) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int blk = (t_begin + it) * kI8Rows + 32 * warp + 16 * mt + g + 8 * h;
                o[mt][h] = (it < my && blk < nb)
                               ? __ldg(reinterpret_cast<const float2 *>(srs + 2 * (int64_t)blk))
                               : make_float2(0.f, 0.f);
            }
    };
    float2 srn[2][2];
    load_sr(0, srn);
    float *lo_row = p.lower + (int64_t)i * p.score_stride;
    float *up_row = p.upper + (int64_t)i * p.score_stride;
    for (int it = 0; it < my; ++it) {
        if (*abort_flag) break;
        const int st = it % S;
        float2 src[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) src[mt][0] = srn[mt][0], src[mt][1] = srn[mt][1];
        load_sr(it + 1, srn);
        if (!mbar_wait(&full[st], (it / S) & 1, deadline)) {
            set_status(p.status, SFA_DEV_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        const uint8_t *tile = sA + (size_t)st * TB;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const int ra = 32 * warp + 16 * mt + g;   // rows ra and ra + 8 of the tile
            uint32_t wa[BPT / 4], wb[BPT / 4];
#pragma unroll
            for (int c = 0; c < BPT / 16; ++c) {
                const uint32_t la = ra * D + BPT * t + 16 * c;   // linear byte of row ra
                const uint4 va = *reinterpret_cast<const uint4 *>(tile + tile_off<D>(la));
                const uint4 vb = *reinterpret_cast<const uint4 *>(tile + tile_off<D>(la + 8 * D));
                wa[4 * c] = va.x, wa[4 * c + 1] = va.y, wa[4 * c + 2] = va.z, wa[4 * c + 3] = va.w;
                wb[4 * c] = vb.x, wb[4 * c + 1] = vb.y, wb[4 * c + 2] = vb.z, wb[4 * c + 3] = vb.w;
            }
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint32_t ua = wa[ks], ub = wb[ks];
                const uint32_t a[4] = {codes_to_f16x2(ua, 0), codes_to_f16x2(ub, 0),
                                       codes_to_f16x2(ua, 2), codes_to_f16x2(ub, 2)};
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_f16_16816(acc[nt], a, bq[nt][ks][0], bq[nt][ks][1]);
            }
            // sum_j w_j max(0, a_j) of rows ra (columns 0, 1) and ra + 8 (columns 2, 3)
            float pa = 0.f, pb = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                pa = fmaf(wv[nt][0], fmaxf(acc[nt][0], 0.f), pa);
                pa = fmaf(wv[nt][1], fmaxf(acc[nt][1], 0.f), pa);
                pb = fmaf(wv[nt][0], fmaxf(acc[nt][2], 0.f), pb);
                pb = fmaf(wv[nt][1], fmaxf(acc[nt][3], 0.f), pb);
            }
            pa += __shfl_xor_sync(0xFFFFFFFFu, pa, 1);
            pa += __shfl_xor_sync(0xFFFFFFFFu, pa, 2);
            pb += __shfl_xor_sync(0xFFFFFFFFu, pb, 1);
            pb += __shfl_xor_sync(0xFFFFFFFFu, pb, 2);
            const int blk = (t_begin + it) * kI8Rows + ra;
            if (t < 2) {   // lane t == 0 writes row ra, t == 1 row ra + 8
                const int b = blk + 8 * t;
                const float2 f = t ? src[mt][1] : src[mt][0];
                if (b < nb) {
                    const float sv = f.x * (t ? pb : pa);
                    const float e = fmaf(kMarginI8, fmaf(cq, f.y, dq_row * f.x), kAbsI8);
                    lo_row[b] = sv - e;   // the hi + lo score lies in [sv - e, sv + e]
                    up_row[b] = sv + e;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
}

}  // namespace
}  // namespace sfa

namespace sfa {
namespace {

template <int D, int H>
int launch_i8(const CUtensorMap &map, I8Params p, int n_blk_tiles, cudaStream_t st) {
    constexpr int TB = kI8Rows * D;
    // four CTAs per SM, each a ring of as many tiles as 55 KB holds (3 of 16 KB at d_idx 128):
    // twelve tiles in flight per SM
    const int per_sm = 4;
    const size_t budget = 55 * 1024, misc = 1024 + 16 * 16 + 16;
    int stages = (int)((budget - misc) / TB);
    stages = stages < 2 ? 2 : (stages > 16 ? 16 : stages);
    p.stages = stages;
    const size_t smem = 1024 + (size_t)stages * TB + 16 * (size_t)stages + 16;
    auto fn = index_score_i8_kernel<D, H>;
    if (!ensure_max_dynamic_smem(fn)) return SFA_ERR_CUDA;
    // one wave: the block tiles of each query are split over as many CTAs as the slots allow
    const int slots = per_sm * device_sm_count();
    int cta_per_q = slots / p.n_q;
    if (cta_per_q > n_blk_tiles) cta_per_q = n_blk_tiles;
    if (cta_per_q < 1) cta_per_q = 1;
    p.tiles_per_cta = (n_blk_tiles + cta_per_q - 1) / cta_per_q;
    const int grid_x = (n_blk_tiles + p.tiles_per_cta - 1) / p.tiles_per_cta;
    if (launch_pdl(fn, dim3(grid_x, p.n_q), dim3(kI8Threads), smem, st, map, p) != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

}  // namespace
}  // namespace sfa

extern "C" int sfa_quantize_pooled_keys_i8(const void *Kbar, int64_t kbar_seq_stride, int n_seq,
                                           int d_idx, int64_t blk_begin, int64_t blk_end,
                                           void *K8, int64_t k8_seq_stride, float *K8_sr,
                                           int64_t sr_seq_stride, sfa_stream_t stream) {
    using namespace sfa;
    if (!Kbar || !K8 || !K8_sr || n_seq < 1) return SFA_ERR_INVALID_ARG;
    if (d_idx != 64 && d_idx != 128) return SFA_ERR_UNSUPPORTED;
    if (blk_begin < 0 || blk_end < blk_begin) return SFA_ERR_INVALID_ARG;
    if (kbar_seq_stride < blk_end * 2 * d_idx || k8_seq_stride < blk_end * d_idx ||
        sr_seq_stride < 2 * blk_end)
        return SFA_ERR_INVALID_ARG;
    if (!aligned16(Kbar) || !aligned16(K8) || (reinterpret_cast<uintptr_t>(K8_sr) & 7u) ||
        kbar_seq_stride % 8 != 0 || k8_seq_stride % 16 != 0 || sr_seq_stride % 2 != 0)
        return SFA_ERR_INVALID_ARG;
    const int64_t n_rows = blk_end - blk_begin;
    if (n_rows == 0) return SFA_OK;
    if (n_seq > 65535) return SFA_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)((n_rows + 7) / 8), (unsigned)n_seq);
    const auto *kb = reinterpret_cast<const __nv_bfloat16 *>(Kbar);
    auto *k8 = reinterpret_cast<int8_t *>(K8);
    const cudaError_t e =
        d_idx == 128 ? launch_pdl(quantize_pooled_i8_kernel<128>, grid, dim3(256), 0,
                                  (cudaStream_t)stream, kb, kbar_seq_stride, blk_begin, n_rows, k8,
                                  k8_seq_stride, K8_sr, sr_seq_stride)
                     : launch_pdl(quantize_pooled_i8_kernel<64>, grid, dim3(256), 0,
                                  (cudaStream_t)stream, kb, kbar_seq_stride, blk_begin, n_rows, k8,
                                  k8_seq_stride, K8_sr, sr_seq_stride);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    return SFA_OK;
}

extern "C" int sfa_index_scores_bounded_i8(const void *q_idx, const float *w, const int32_t *q_seq,
                                           const int32_t *q_pos, int n_q, int h_idx, int d_idx,
                                           int compress_ratio, const void *K8,
                                           int64_t k8_seq_stride, const float *K8_sr,
                                           int64_t sr_seq_stride, int n_seq, int64_t n_blk_max,
                                           float *lower, float *upper, int64_t score_stride,
                                           int32_t *dev_status, sfa_stream_t stream) {
    using namespace sfa;
    if (!q_idx || !w || !q_seq || !q_pos || !K8 || !K8_sr || !lower || !upper)
        return SFA_ERR_INVALID_ARG;
    if (n_q < 0 || n_seq < 1 || compress_ratio < 1 || n_blk_max < 0) return SFA_ERR_INVALID_ARG;
    if (d_idx != 64 && d_idx != 128) return SFA_ERR_UNSUPPORTED;
    if (h_idx != 4 && h_idx != 8 && h_idx != 16) return SFA_ERR_UNSUPPORTED;
    if (k8_seq_stride <= 0 || k8_seq_stride % d_idx != 0) return SFA_ERR_INVALID_ARG;
    const int64_t blk_cap = k8_seq_stride / d_idx;   // sequences are contiguous runs of rows
    if (n_blk_max > blk_cap || n_blk_max > score_stride || sr_seq_stride < 2 * n_blk_max ||
        sr_seq_stride % 2 != 0)
        return SFA_ERR_INVALID_ARG;
    if (!aligned16(q_idx) || !aligned16(K8) || (reinterpret_cast<uintptr_t>(K8_sr) & 7u))
        return SFA_ERR_INVALID_ARG;
    if (n_q == 0 || n_blk_max == 0) return SFA_OK;
    if (n_q > 65535 || (int64_t)n_seq * blk_cap > 0x7FFFFFFFll) return SFA_ERR_UNSUPPORTED;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return SFA_ERR_CUDA;
    CUtensorMap map;
    const cuuint64_t gdim[2] = {(cuuint64_t)d_idx, (cuuint64_t)(n_seq * blk_cap)};
    const cuuint64_t gstride[1] = {(cuuint64_t)d_idx};
    const cuuint32_t box[2] = {(cuuint32_t)d_idx, (cuuint32_t)kI8Rows};
    const cuuint32_t estride[2] = {1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(K8), gdim, gstride, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
            d_idx == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SFA_ERR_INVALID_ARG;
    I8Params p{};
    p.q_idx = reinterpret_cast<const __nv_bfloat16 *>(q_idx);
    p.w = w;
    p.q_seq = q_seq;
    p.q_pos = q_pos;
    p.sr = K8_sr;
    p.sr_seq_stride = sr_seq_stride;
    p.lower = lower;
    p.upper = upper;
    p.score_stride = score_stride;
    p.status = dev_status;
    p.blk_cap = blk_cap;
    p.n_blk_max = n_blk_max;
    p.n_q = n_q;
    p.n_seq = n_seq;
    p.cr = compress_ratio;
    const int n_blk_tiles = (int)((n_blk_max + kI8Rows - 1) / kI8Rows);
    const cudaStream_t st = (cudaStream_t)stream;
    if (d_idx == 64) {
        if (h_idx == 4) return launch_i8<64, 4>(map, p, n_blk_tiles, st);
        if (h_idx == 8) return launch_i8<64, 8>(map, p, n_blk_tiles, st);
        return launch_i8<64, 16>(map, p, n_blk_tiles, st);
    }
    if (h_idx == 4) return launch_i8<128, 4>(map, p, n_blk_tiles, st);
    if (h_idx == 8) return launch_i8<128, 8>(map, p, n_blk_tiles, st);
    return launch_i8<128, 16>(map, p, n_blk_tiles, st);
}
