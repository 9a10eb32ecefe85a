/*
 * sfa.h -- C ABI of libsfa: indexer-selected block-sparse attention on one GB300 (sm_103a).
 *
 * The method (llama.cpp commit "model: add Qwen3.8-Flash-Next (qwen4exp)", the QSA indexer
 * paragraphs; llama.cpp PR #27970 "CUDA + ggml: add sparse-fa for DSV4/GLM"): for each query
 * token i of sequence s_i at position p_i, an indexer scores one mean-pooled key per block of
 * compress_ratio (cr) cached tokens, as the weighted sum over index heads of the rectified dot
 * product; the best indexer_top_k blocks plus the tail of tokens that do not form a complete
 * block are kept; softmax attention then runs over those cells only.
 *
 *   B_i    = floor((p_i + 1) / cr)                complete blocks visible to query i
 *   tail_i = [B_i*cr, p_i]                        always attended
 *   kbar_b = (1/cr) sum_{t in block b} X[s_i][t]  raw index keys, pooled   (sfa_pool_index_keys)
 *   s_ib   = sum_j w_ij * max(0, qidx_ij . kbar_b),  b < B_i                (sfa_index_scores)
 *   Sel_i  = all b < B_i if B_i <= top_k, else the top_k best by (score desc, block asc)
 *                                                                           (sfa_topk_blocks)
 *   O_ih   = softmax_t(scale * Q_ih . K[s_i][t][g]) V[s_i][t][g] over t in Sel_i-blocks + tail,
 *            g = h / (h_q / h_kv)                                           (sfa_gather_attend)
 *   below the budget (every B_i <= top_k) this is dense causal attention    (sfa_dense_attend)
 *
 * Conventions shared by every entry point:
 *  - Returns an sfa status (SFA_OK = 0).  Never aborts, never synchronises the stream, never
 *    allocates device memory.  Invalid arguments are rejected on the host before anything is
 *    enqueued.  A CUDA launch error returns SFA_ERR_CUDA.
 *  - All data pointers are caller-owned DEVICE pointers, with two exceptions: the attention
 *    outputs O and lse may also point to page-locked host memory that the device addresses
 *    directly (cudaHostAlloc, or cudaHostRegister'd, with unified addressing) -- the kernels
 *    then write the results over the host link and the caller reads them once the stream has
 *    passed the call -- and sfa_copy_cache_rows takes either kind.  Work is enqueued on
 *    `stream` (a cudaStream_t; NULL is the legacy default stream).  The library keeps no
 *    state between calls except a per-device cache of the SM count and of the CUDA driver's
 *    tensor-map encoder.
 *  - Strides are in elements of the buffer's own type.  Buffers must be 16-byte aligned.
 *  - `dev_status` (nullable) is a device int32 the kernels OR bits into (SFA_DEV_*) when they
 *    meet data they cannot use (a block id outside [0, B_i), a non-ascending list, n_sel out
 *    of range, a query outside the caches, a bounded wait that ran out).  The offending entry
 *    is skipped; nothing traps.  The caller clears it and reads it when it wishes
 *    (sfa_read_device_status).
 */
#ifndef SFA_H
#define SFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *sfa_stream_t; /* identical to cudaStream_t */

enum sfa_status {
    SFA_OK = 0,
    SFA_ERR_INVALID_ARG = 1, /* a pointer, size, stride or alignment the call cannot accept */
    SFA_ERR_UNSUPPORTED = 2, /* a valid shape the library has no kernel for               */
    SFA_ERR_CUDA = 3,        /* the CUDA runtime reported an error while enqueuing         */
    SFA_ERR_WORKSPACE = 4    /* the workspace is NULL or smaller than the size query says  */
};

/* SFA_Q8_0: K and V are q8_0 cache rows (sfa_quantize_kv_q8_0) and Q is bf16; the attention
 * then runs its tensor-core products on binary16 operands.                                 */
enum sfa_dtype { SFA_BF16 = 0, SFA_F32 = 1, SFA_Q8_0 = 2 };

/* bits of the device status word */
#define SFA_DEV_BAD_BLOCK 0x1 /* a selected block id outside [0, B_i) or not ascending      */
#define SFA_DEV_BAD_NSEL 0x2  /* n_sel[i] < 0 or > top_k (clamped)                         */
#define SFA_DEV_BAD_QUERY 0x4 /* q_seq/q_pos outside the caches, or a query group that
                                 spans sequences (that query is skipped), or a dense query
                                 with q_pos + 1 > n_kv_max (its first n_kv_max keys only) */
#define SFA_DEV_TIMEOUT 0x8   /* a bounded wait inside a kernel ran out; the kernel
                                 released its resources and returned early                */
#define SFA_DEV_BAD_CELL 0x10 /* a paged cell map entry outside [0, n_cells): that position
                                 reads as a zero row (pool) or is left out (attention)    */
#define SFA_DEV_FP16_RANGE 0x20 /* a binary16 operand path: a value beyond binary16's range
                                 (a q8_0 scale, a query element or a dequantized K/V value;
                                 with SFA_ATTEND_KERNEL=ws, a bf16 V element at or above
                                 65520 in magnitude); the results involving it are not
                                 finite                                                  */

/*
 * sfa_pool_index_keys -- one mean-pooled index key per block of compress_ratio tokens, taken
 * over the RAW index keys, since the model pools before it normalises and rotates them (QSA
 * commit, indexer key cache paragraph; block pooling: QSA commit, budget paragraph).  Blocks
 * are cut on positions: block b holds tokens [b*cr, b*cr + cr).
 *
 *   X      [n_seq][x_seq_stride / d_idx][d_idx], x_dtype SFA_BF16 or SFA_F32 (raw keys)
 *   Kbar   [n_seq][kbar_seq_stride / (2*d_idx)][2*d_idx] bf16 (uint16 storage): row b of
 *          sequence s holds the pooled key split in two bf16 halves,
 *            m      = fl32(sum_t X[s][t]) / cr   (fp32 sum in token order, IEEE division)
 *            hi     = bf16_rn(m),  lo = bf16_rn(m - hi)
 *            row b  = (hi[0..d_idx), lo[0..d_idx))
 *          so that hi + lo carries m to about 2^-17 relative while the tensor cores read it
 *          as plain bf16.
 *   Kbar_r [n_seq][kr_seq_stride] fp32, or NULL: the error-bound factor of each pooled row
 *          for sfa_index_scores_bounded, from the stored halves,
 *            r_b = (|lo|_2 + 2^-14 |hi|_2) * (1 + 2^-16)   (fp32 norms)
 * Writes rows [blk_begin, blk_end) of every sequence; reads tokens [blk_begin*cr, blk_end*cr).
 * Limits: 1 <= cr <= 64, d_idx in {32, 64, 96, 128} (Kbar_r: not 96), 0 <= blk_begin <=
 * blk_end; kr_seq_stride >= blk_end when Kbar_r is given.
 */
int sfa_pool_index_keys(const void *X, int x_dtype, int64_t x_seq_stride, int n_seq, int d_idx,
                        int compress_ratio, int64_t blk_begin, int64_t blk_end, void *Kbar,
                        int64_t kbar_seq_stride, float *Kbar_r, int64_t kr_seq_stride,
                        sfa_stream_t stream);

/*
 * sfa_pool_index_keys_transformed -- sfa_pool_index_keys with the norm and the rotation the
 * model applies to the pooled index key before scoring (QSA commit: the index-key cache holds
 * raw keys because pooling precedes the norm and the rotation; the indexer ropes with the main
 * attention's rotary width).  The pages name neither the norm nor the rotary pairing nor the
 * position of a pooled block, so the caller chooses:
 *   norm 0: none; 1: RMS norm, y = m / sqrt(mean(m^2) + eps) * gamma;
 *        2: layer norm, y = (m - mean(m)) / sqrt(var(m) + eps) * gamma + beta
 *        (over the d_idx dims of the pooled row m; gamma, beta: [d_idx] fp32 device arrays)
 *   n_rot dims (even, <= d_idx; 0: no rotation) turned pairwise at position
 *        p_b = b * compress_ratio + pos_offset, pair j by p_b * rope_base^(-2j / n_rot);
 *        rope_neox 1: pairs (j, j + n_rot/2) (n_rot a multiple of 16); 0: pairs (2j, 2j + 1)
 * The transformed key is what is split into hi + lo and what Kbar_r bounds.  Norm statistics
 * are fp32; angles, sines and cosines double.
 * Limits: those of sfa_pool_index_keys; d_idx in {32, 64, 128} when a transform is given.
 */
int sfa_pool_index_keys_transformed(const void *X, int x_dtype, int64_t x_seq_stride, int n_seq,
                                    int d_idx, int compress_ratio, int64_t blk_begin,
                                    int64_t blk_end, int norm, const float *gamma,
                                    const float *beta, float eps, int n_rot, float rope_base,
                                    int rope_neox, int64_t pos_offset, void *Kbar,
                                    int64_t kbar_seq_stride, float *Kbar_r, int64_t kr_seq_stride,
                                    sfa_stream_t stream);

/*
 * sfa_index_scores -- the indexer score of every complete block visible to each query: each
 * index head's dot product passes through a ReLU before the weighted sum over heads (QSA
 * commit, index comparison paragraph); a query is scored only against the blocks of its own
 * sequence (QSA commit, multi-stream scoring).
 *
 *   q_idx   [n_q][h_idx][d_idx] bf16 index queries;   w [n_q][h_idx] fp32 head weights
 *   q_seq, q_pos [n_q] int32: sequence and position of each query
 *   Kbar    pooled keys as written by sfa_pool_index_keys (rows >= B_i are not read for i)
 *   scores  [n_q][score_stride] fp32: scores[i][b] = s_ib for b < min(B_i, n_blk_max);
 *           entries at b >= B_i are left untouched.
 *   q_group: the caller's promise that queries [k*q_group, (k+1)*q_group) share one sequence
 *           (1 for decode batches of independent sequences; n_q for one prefill ubatch).
 *           Tiles of queries that share a sequence share every pooled-key load.  A query that
 *           breaks the promise is skipped and SFA_DEV_BAD_QUERY is set.
 *   n_blk_max: host bound on max_i B_i (<= blk_cap = kbar_seq_stride / (2*d_idx), and
 *           <= score_stride).
 * The q.kbar contraction runs on tcgen05 tensor cores (bf16 x (hi, lo) into an fp32 TMEM
 * accumulator); the ReLU, weights and head sum run in the TMEM read-back.
 * Limits: d_idx in {64, 128}; h_idx in {4, 8, 16}; n_seq * blk_cap < 2^31.
 */
int sfa_index_scores(const void *q_idx, const float *w, const int32_t *q_seq,
                     const int32_t *q_pos, int n_q, int q_group, int h_idx, int d_idx,
                     int compress_ratio, const void *Kbar, int64_t kbar_seq_stride, int n_seq,
                     int64_t n_blk_max, float *scores, int64_t score_stride,
                     int32_t *dev_status, sfa_stream_t stream);

/*
 * sfa_topk_blocks -- the budget rule: the indexer_top_k best blocks are kept, and the tail of
 * tokens that do not yet fill a block is always attended; when a query sees no more blocks
 * than the budget, every block is kept and the result is dense (QSA commit, budget
 * paragraph).  The budget is whole blocks, so the cut falls on a block boundary (QSA commit,
 * expansion paragraph).  Ties at the cut go to the lower block index (the pages do not order
 * equal scores; this is the stated reading).  -0.0 counts as +0.0; a NaN score ranks lowest.
 *
 *   scores  as written by sfa_index_scores; row i is read at [0, B_i)
 *   blk_idx [n_q][top_k] int32: the kept block ids of query i, ascending, padded with -1
 *           (the padding convention of PR #27970's sparse index rows)
 *   n_sel   [n_q] int32: min(top_k, B_i)
 *   workspace: sfa_topk_workspace_bytes(n_q, n_blk_max, top_k) bytes of device memory.
 * The tail is not listed: it is implied by q_pos and cr and always attended.
 * Limits: 1 <= top_k <= 2048; n_blk_max <= 2^21.
 */
size_t sfa_topk_workspace_bytes(int n_q, int64_t n_blk_max, int top_k);
int sfa_topk_blocks(const float *scores, int64_t score_stride, const int32_t *q_pos, int n_q,
                    int compress_ratio, int top_k, int64_t n_blk_max, int32_t *blk_idx,
                    int32_t *n_sel, void *workspace, size_t workspace_bytes,
                    int32_t *dev_status, sfa_stream_t stream);

/*
 * sfa_index_scores_bounded / sfa_topk_blocks_refine -- the same kept sets as
 * sfa_index_scores + sfa_topk_blocks from half the pooled-key bytes (a library addition: the
 * pages score and select in one pass each).
 *
 * sfa_index_scores_bounded: arguments as sfa_index_scores plus Kbar_r, kr_seq_stride (the
 * bound factors written by sfa_pool_index_keys with the same Kbar); it reads only the hi
 * halves of the pooled keys and writes lower and upper bounds of the hi + lo score s_ib:
 *   lower, upper [n_q][score_stride] fp32: lower = a - e <= s_ib <= a + e = upper, with
 *           a_ib = sum_j w_ij * max(0, qidx_ij . hi_b) and
 *           e_ib = (1 + 2^-10) * (sum_j |w_ij| |qidx_ij|_2) * r_b.  The exact difference is at
 *           most (sum_j |w_ij| |qidx_ij|_2) |lo_b|_2 (ReLU is 1-Lipschitz; Cauchy-Schwarz per
 *           head); r_b's second term covers the fp32 rounding of both scores (< 2^-15 of
 *           sum_j |w_ij| |qidx_ij|_2 |hi_b|_2).
 * Both arrays share score_stride; entries at b >= B_i are left untouched.
 *
 * sfa_topk_blocks_refine: per query, L = a lower bound of the k-th largest lower bound: the
 * row is split over the CTAs of a cluster; each CTA takes the maxima of the lower bounds of
 * its groups of four consecutive blocks and a quota k_r of them (proportional to its share of
 * the row's groups, the quotas summing to at least k), finds a floor X_r under its k_r
 * largest (a histogram bin), and L = min_r X_r; every block
 * with upper >= L is a candidate (every block of the top k by s is one, and so is every block
 * whose s ties the k-th); the candidates are rescored from hi + lo (bf16 products, fp32 sums)
 * and the top indexer_top_k of them by (score desc, block asc) are written as sfa_topk_blocks
 * writes them.  One kernel launch; each query's row is split over a cluster of four CTAs
 * (eight past 36864 blocks).
 *   lower, upper: as written by sfa_index_scores_bounded (or sfa_index_scores_bounded_i8) for
 *           the same queries and Kbar
 *   q_idx, w, q_seq, q_pos, Kbar, kbar_seq_stride, n_seq: as given to it; Kbar 16-byte
 *           aligned with kbar_seq_stride a multiple of 8, q_idx 4-byte aligned
 *   blk_idx, n_sel: as sfa_topk_blocks
 *   workspace: sfa_topk_refine_workspace_bytes(n_q, n_blk_max) bytes of device memory (used
 *           for candidate lists longer than 4096)
 * Limits: n_blk_max <= 131072 (each CTA of a row's cluster takes 3 rounds of 4096 blocks
 * up to 36864 blocks per row, 8 beyond); 1 <= top_k <= 2048; d_idx in {64, 128};
 * 1 <= h_idx <= 16.
 * Errors as the other entry points (host checks before any launch, SFA_DEV_* flags); a
 * candidate id outside its row (which only inconsistent lower/upper arrays could produce) is
 * not read and raises SFA_DEV_BAD_BLOCK.
 */
int sfa_index_scores_bounded(const void *q_idx, const float *w, const int32_t *q_seq,
                             const int32_t *q_pos, int n_q, int q_group, int h_idx, int d_idx,
                             int compress_ratio, const void *Kbar, int64_t kbar_seq_stride,
                             const float *Kbar_r, int64_t kr_seq_stride, int n_seq,
                             int64_t n_blk_max, float *lower, float *upper, int64_t score_stride,
                             int32_t *dev_status, sfa_stream_t stream);
size_t sfa_topk_refine_workspace_bytes(int n_q, int64_t n_blk_max);
int sfa_topk_blocks_refine(const float *lower, const float *upper, int64_t score_stride,
                           const void *q_idx, const float *w, const int32_t *q_seq,
                           const int32_t *q_pos, int n_q, int h_idx, int d_idx,
                           const void *Kbar, int64_t kbar_seq_stride, int n_seq,
                           int compress_ratio, int top_k, int64_t n_blk_max, int32_t *blk_idx,
                           int32_t *n_sel, void *workspace, size_t workspace_bytes,
                           int32_t *dev_status, sfa_stream_t stream);

/*
 * sfa_quantize_pooled_keys_i8 / sfa_index_scores_bounded_i8 -- the same lower and upper bounds
 * from 8-bit copies of the pooled keys: the bound pass then reads d_idx bytes per block instead
 * of the 2*d_idx bytes of the hi halves (the bounds are looser: about twice as many
 * candidates reach the rescoring).
 *
 * sfa_quantize_pooled_keys_i8 writes, for rows [blk_begin, blk_end) of every sequence, from the
 * pooled keys m = hi + lo of Kbar (as written by any sfa_pool_index_keys* call):
 *   K8    [n_seq][k8_seq_stride / d_idx][d_idx] bytes: c_bi + 128 (offset binary), with
 *         c_bi = round(m_bi / sc_b) clamped to [-127, 127] and sc_b = max_i |m_bi| / 127 (0 for
 *         a zero row: c = 0)
 *   K8_sr [n_seq][sr_seq_stride] fp32, pairs per block: (sc_b, r_b),
 *         r_b = (|m_b - sc_b c_b|_2 + 2^-14 sc_b |c_b|_2) (1 + 2^-16)   (fp32 norms)
 * Call it for the rows each pool call wrote.  Limits: d_idx in {64, 128}; Kbar and K8 16-byte
 * aligned, K8_sr 8-byte aligned; kbar_seq_stride >= blk_end*2*d_idx (a multiple of 8),
 * k8_seq_stride >= blk_end*d_idx (a multiple of 16), sr_seq_stride >= 2*blk_end (even).
 *
 * sfa_index_scores_bounded_i8 writes lower and upper bounds of the hi + lo score s_ib:
 *   lower = a - e <= s_ib <= a + e = upper,  a_ib = sc_b * sum_j w_ij * max(0, q~_ij . c_b),
 *   q~ = binary16(qidx) (clamped to +-65504),
 *   e_ib = (1 + 2^-10) * (C_i r_b + D_i 127 sqrt(d_idx) sc_b),  C_i = sum_j |w_ij| |qidx_ij|_2,
 *   D_i = sum_j |w_ij| |qidx_ij - q~_ij|_2.  The exact difference is at most
 *   C_i |m_b - sc_b c_b|_2 + D_i sc_b |c_b|_2 (ReLU is 1-Lipschitz, sc_b >= 0, Cauchy-Schwarz
 *   per head, |c_b|_2 <= 127 sqrt(d_idx)); r_b's second term covers the fp32 rounding of both
 *   scores.
 *   K8, K8_sr: as written by sfa_quantize_pooled_keys_i8; the sequences' rows must be
 *          contiguous (blk_cap = k8_seq_stride / d_idx rows per sequence, no gaps)
 *   other arguments as sfa_index_scores_bounded (each query on its own: no query groups).
 * Entries at b >= B_i are left untouched.  Limits: d_idx in {64, 128}, h_idx in {4, 8, 16};
 * q_idx 16-byte aligned.  Errors as the other entry points.
 */
int sfa_quantize_pooled_keys_i8(const void *Kbar, int64_t kbar_seq_stride, int n_seq, int d_idx,
                                int64_t blk_begin, int64_t blk_end, void *K8,
                                int64_t k8_seq_stride, float *K8_sr, int64_t sr_seq_stride,
                                sfa_stream_t stream);
int sfa_index_scores_bounded_i8(const void *q_idx, const float *w, const int32_t *q_seq,
                                const int32_t *q_pos, int n_q, int h_idx, int d_idx,
                                int compress_ratio, const void *K8, int64_t k8_seq_stride,
                                const float *K8_sr, int64_t sr_seq_stride, int n_seq,
                                int64_t n_blk_max, float *lower, float *upper,
                                int64_t score_stride, int32_t *dev_status, sfa_stream_t stream);

/*
 * sfa_gather_attend -- softmax attention of each query over the cells of its kept blocks plus
 * its tail (PR #27970: flash attention whose K/V tile loads are gathered through a per-query
 * index list; V may be a view of the first DV dims of K; no ALiBi, no softcap).
 *
 *   Q    [n_q][h_q][dkq]                       dtype (SFA_BF16 or SFA_F32)
 *   K    [n_seq][n_tok_cap][h_kv][dkq]         dtype
 *   V    [n_seq][n_tok_cap][h_kv][dv] dtype, or NULL: V = K[..., :dv] (MLA layout)
 *   blk_idx, n_sel: as written by sfa_topk_blocks (any ascending subset of [0, B_i) works)
 *   O    [n_q][h_q][dv] fp32;  lse [n_q][h_q] fp32 natural-log sum of exp(logits), nullable
 *   workspace: sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, top_k*cr + cr - 1) bytes
 *           (split-KV partial results; may be NULL when that size is 0).
 * Query head h reads KV head h / (h_q / h_kv).  p_i < n_tok_cap is required.
 * Limits (bf16): (dkq, dv) in {(576, 512), (512, 512), (128, 128), (64, 64)}, h_q/h_kv <= 16;
 *        dv > dkq needs a separate V.  Kernel choice (read from the environment at each call):
 *        default, the warp-level mma.sync kernel with 32-token tiles (SFA_ATTEND_TT=16: 16-token
 *        tiles, deeper prefetch); SFA_ATTEND_KERNEL=tcgen05, the tcgen05 kernel for dkq 576 /
 *        512; SFA_ATTEND_KERNEL=ws, the warp-specialised bulk-copy kernel (P V on binary16
 *        operands, SFA_ATTEND_PV=bf16x2 for bf16 hi + lo).  All meet the same tolerances.
 *        (fp32): the same (dkq, dv) pairs and h_q/h_kv <= 16.
 * Few (query, KV head) lists are split over several CTAs (flash-decoding); with the bf16
 * kernel, 2 to 8 splits merge inside a thread-block cluster, else a second kernel merges them.
 */
size_t sfa_attend_workspace_bytes(int n_q, int h_q, int h_kv, int dv, int64_t n_kv_max);
/*
 * sfa_attend_plan -- the launch plan the attention entry points take on the current device
 * for these sizes: *n_split CTAs per (query, KV head) list and *kernels launched per call
 * (1, or 2 when a merge kernel follows).  n_kv_max as in sfa_attend_workspace_bytes (the
 * dense entry point: n_tok_cap, dense = 1); has_v: a separate V is given; dtype as the entry
 * points (SFA_BF16, SFA_F32 or SFA_Q8_0).  It describes the per-sequence layout; the paged
 * calls take the same plan, except that they never take the tcgen05 kernel.  Host only, no
 * launch.  SFA_ERR_INVALID_ARG / SFA_ERR_UNSUPPORTED as the entry points.
 */
int sfa_attend_plan(int dtype, int n_q, int h_kv, int dkq, int has_v, int64_t n_kv_max,
                    int compress_ratio, int dense, int *n_split, int *kernels);
int sfa_gather_attend(const void *Q, const void *K, const void *V, int dtype, int n_seq,
                      int64_t n_tok_cap, int n_q, int h_q, int h_kv, int dkq, int dv,
                      float scale, const int32_t *q_seq, const int32_t *q_pos,
                      const int32_t *blk_idx, const int32_t *n_sel, int top_k,
                      int compress_ratio, float *O, float *lse, void *workspace,
                      size_t workspace_bytes, int32_t *dev_status, sfa_stream_t stream);

/*
 * sfa_gather_attend_window -- attention over the kept blocks, the tail AND a dense window of
 * the `window` most recent positions p_i - window + 1 .. p_i (clipped at 0): the dense +
 * sparse variant of PR #27970's review discussion (dense attention over the continuous block
 * of keys, sparse attention over the selected keys, the results combined).  Let s0 be the
 * first position of the suffix attended in full: min(B_i*cr, p_i - window + 1) (B_i*cr when
 * window = 0).  `part` chooses what one call attends:
 *   SFA_PART_ALL       the whole set in one pass: the kept tokens before s0, then s0 .. p_i;
 *   SFA_PART_SELECTED  only the kept tokens before s0 (no tail, no window);
 *   SFA_PART_WINDOW    only the suffix s0 .. p_i;
 * the two parts are disjoint and cover the set, so sfa_combine_attention of their (O, lse)
 * gives SFA_PART_ALL's result.  window = 0 with SFA_PART_ALL is sfa_gather_attend.  A part
 * with nothing to attend gives O = 0 and lse = -inf.
 *   workspace: sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv,
 *               sfa_window_kv_max(top_k, compress_ratio, window, part)) bytes.
 * Arguments otherwise, limits and kernels as sfa_gather_attend; window >= 0.
 */
enum sfa_part { SFA_PART_ALL = 0, SFA_PART_SELECTED = 1, SFA_PART_WINDOW = 2 };
int64_t sfa_window_kv_max(int top_k, int compress_ratio, int64_t window, int part);
int sfa_gather_attend_window(const void *Q, const void *K, const void *V, int dtype, int n_seq,
                             int64_t n_tok_cap, int n_q, int h_q, int h_kv, int dkq, int dv,
                             float scale, const int32_t *q_seq, const int32_t *q_pos,
                             const int32_t *blk_idx, const int32_t *n_sel, int top_k,
                             int compress_ratio, int64_t window, int part, float *O,
                             float *lse, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, sfa_stream_t stream);

/*
 * sfa_gather_kv_bandwidth -- a measurement, not part of the method: moves exactly the K (and
 * V) rows that sfa_gather_attend attends for these lists (the kept blocks' rows and the tail's)
 * into shared memory and computes nothing.  Each run of 4 consecutive rows (a kept block of
 * cr >= 4, a run of the tail) is one bulk copy, issued by four warps per CTA, one CTA per SM;
 * the first word of every row is summed into *checksum (device uint32, atomically added) so
 * that no copy can be dropped.  Its time is the data-movement ceiling of the attention on the
 * same lists: with the caches in HBM, that of the gather pattern out of HBM; with them in L2,
 * that of the L2 -> shared-memory gather.  Arguments as sfa_gather_attend (bf16 K/V; (dkq, dv)
 * in {(576, 512) with V = NULL, (512, 512)}).
 */
int sfa_gather_kv_bandwidth(const void *K, const void *V, int n_seq, int64_t n_tok_cap,
                            int n_q, int h_kv, int dkq, int dv, const int32_t *q_seq,
                            const int32_t *q_pos, const int32_t *blk_idx, const int32_t *n_sel,
                            int top_k, int compress_ratio, uint32_t *checksum,
                            int32_t *dev_status, sfa_stream_t stream);

/*
 * sfa_combine_attention -- merges two attentions of the same queries over disjoint key sets
 * into the attention over their union, by their log-sum-exp (the "combining the result" step
 * of the dense + sparse variant; exact: softmax over a disjoint union):
 *   O[r] = (e^lse_a[r] O_a[r] + e^lse_b[r] O_b[r]) / (e^lse_a[r] + e^lse_b[r]),
 *   lse[r] = log(e^lse_a[r] + e^lse_b[r]),
 * for the n_rows rows of dv fp32 values (rows = query x head).  A part with lse = -inf
 * contributes nothing; both -inf gives O = 0, lse = -inf.  O may be O_a or O_b and lse may be
 * lse_a or lse_b (in place); every pointer is device memory, 16-byte aligned; dv a multiple
 * of 4.  One kernel launch.  SFA_ERR_INVALID_ARG for bad arguments.
 */
int sfa_combine_attention(const float *O_a, const float *lse_a, const float *O_b,
                          const float *lse_b, int64_t n_rows, int dv, float *O, float *lse,
                          sfa_stream_t stream);

/*
 * sfa_dense_attend -- causal attention of each query over all of its sequence's tokens
 * 0..p_i: the below-budget case, where the sparse result is exactly dense (QSA commit, budget
 * paragraph); a layer without a compression ratio also attends densely.  n_kv_max must bound p_i + 1 for
 * every query (the role of PR #27970's n_kv_max hint); it sizes the split-KV work.
 * Arguments otherwise as sfa_gather_attend.
 */
int sfa_dense_attend(const void *Q, const void *K, const void *V, int dtype, int n_seq,
                     int64_t n_tok_cap, int n_q, int h_q, int h_kv, int dkq, int dv,
                     float scale, const int32_t *q_seq, const int32_t *q_pos, int64_t n_kv_max,
                     float *O, float *lse, void *workspace, size_t workspace_bytes,
                     int32_t *dev_status, sfa_stream_t stream);

/*
 * Paged (non-contiguous) cell layout.  The cache holds each stream's tokens in cells of a flat
 * array in any order; blocks are still cuts of the position line, so the block of position t
 * is t / cr wherever its cell sits, and a map from positions to cells, kept per stream because
 * a cell index means a different token in each stream, is all the kernels need (qwen4exp
 * commits in llama.cpp: the QSA paragraph that computes every layout-dependent input on the
 * host and cuts blocks on positions, and "support a non-unified KV cache in QSA", where the
 * cell maps gain a stream dimension).  The scores and the selection work on pooled blocks and
 * are unchanged; the pool and the attention read their rows through the map:
 *
 *   cell_of [n_seq][n_pos_cap] int32 (device): cell_of[s][t] = the cell that holds position t
 *           of sequence s.  Only the positions a call reads are looked at (t < blk_end*cr for
 *           the pool, t <= p_i for the attention), so unused entries may hold anything.
 *   X       [n_cells][d_idx] raw index keys (pool);  K [n_cells][h_kv][dkq], V [n_cells][h_kv][dv]
 *           or NULL (attention), each row one cell.
 *
 * Results equal those of the per-sequence calls on the gathered layout X'[s][t] = X[cell_of[s][t]]
 * (K', V' the same) bit for bit under the default kernel choice: the same kernels read the
 * same values in the same order.  An entry outside [0, n_cells) sets SFA_DEV_BAD_CELL
 * (dev_status is nullable for the pool too).  The
 * attention calls never take the tcgen05 kernel (its producers copy runs of four consecutive
 * rows as one TMA box), whatever SFA_ATTEND_KERNEL says; sfa_attend_plan describes them
 * otherwise.  n_pos_cap plays the role of n_tok_cap (p_i < n_pos_cap); n_cells < 2^31.
 * Arguments otherwise as sfa_pool_index_keys, sfa_gather_attend and sfa_dense_attend.
 */
int sfa_pool_index_keys_paged(const void *X, int x_dtype, int64_t n_cells, const int32_t *cell_of,
                              int64_t n_pos_cap, int n_seq, int d_idx, int compress_ratio,
                              int64_t blk_begin, int64_t blk_end, void *Kbar,
                              int64_t kbar_seq_stride, float *Kbar_r, int64_t kr_seq_stride,
                              int32_t *dev_status, sfa_stream_t stream);
int sfa_gather_attend_paged(const void *Q, const void *K, const void *V, int dtype,
                            int64_t n_cells, const int32_t *cell_of, int n_seq, int64_t n_pos_cap,
                            int n_q, int h_q, int h_kv, int dkq, int dv, float scale,
                            const int32_t *q_seq, const int32_t *q_pos, const int32_t *blk_idx,
                            const int32_t *n_sel, int top_k, int compress_ratio, float *O,
                            float *lse, void *workspace, size_t workspace_bytes,
                            int32_t *dev_status, sfa_stream_t stream);
int sfa_dense_attend_paged(const void *Q, const void *K, const void *V, int dtype,
                           int64_t n_cells, const int32_t *cell_of, int n_seq, int64_t n_pos_cap,
                           int n_q, int h_q, int h_kv, int dkq, int dv, float scale,
                           const int32_t *q_seq, const int32_t *q_pos, int64_t n_kv_max, float *O,
                           float *lse, void *workspace, size_t workspace_bytes,
                           int32_t *dev_status, sfa_stream_t stream);

/*
 * Quantized KV cache (q8_0).  The qwen4exp commits let the QSA attention path read a quantized
 * KV cache; q8_0 is the 8-bit block format of the llama.cpp caches they describe.  Each row of
 * d elements (one token and KV head of K, or of V) is cut into blocks of 32; per block
 *   delta = max |x| / 127 (binary32), code_j = x_j / delta rounded half away from zero
 *   (binary32; 0 when delta = 0), scale = delta rounded to binary16 (ties to even),
 * and the element stands for scale * code_j.  A cache row holds the d int8 codes, then the
 * d/32 binary16 scales, then zero bytes up to sfa_q8_0_row_bytes(d) (a multiple of 16):
 * 624 bytes for d = 576, 544 for 512, 144 for 128, 80 for 64.  With V = NULL the values are the
 * first dv elements of K: the first dv codes and dv/32 scales of the K row.
 *
 * sfa_quantize_kv_q8_0 writes such rows: for o < n_outer and i < n_inner, the d elements at
 * X + o*x_outer_stride + i*d (elements of x_dtype) go to the row at
 * Y + o*y_outer_stride + i*sfa_q8_0_row_bytes(d) (bytes), so a slice of new tokens of every
 * sequence is one call.  d in {64, 128, 512, 576}.  A scale beyond binary16 sets
 * SFA_DEV_FP16_RANGE (inputs must be finite).  The codes and scales equal the rule above bit for
 * bit.
 *
 * The attention entry points (gathered, dense, paged) take dtype = SFA_Q8_0: K is
 * [n_seq][n_tok_cap][h_kv][row_bytes(dkq)] (or [n_cells][h_kv][row_bytes(dkq)] paged) and V the
 * same with dv, or NULL; Q is bf16.  The kernel gathers the quantized rows (about half the
 * bytes of bf16 rows), dequantizes each tile in shared memory to binary16, converts Q to
 * binary16, and runs S = Q K^T and O = P V on binary16 tensor-core operands with fp32
 * accumulation (P as binary16 hi + lo halves).  The dequantized values have up to 19
 * significant bits, so binary16 (11) keeps the outputs within the 2e-3 bf16 tolerance where
 * bf16 (8) would not.  A query element or a dequantized value beyond binary16's range sets
 * SFA_DEV_FP16_RANGE.  Limits: those of the bf16 kernel.
 */
size_t sfa_q8_0_row_bytes(int d);
int sfa_quantize_kv_q8_0(const void *X, int x_dtype, int64_t n_outer, int64_t n_inner, int d,
                         int64_t x_outer_stride, void *Y, int64_t y_outer_stride,
                         int32_t *dev_status, sfa_stream_t stream);

/*
 * sfa_gather_attend_noalloc -- sfa_gather_attend for callers that cannot allocate device
 * memory.  (No counterpart in the pages: it is a property of this library's interface.)
 *
 * Some callers have no way to hand the library a workspace at the point of the call: a host
 * application that owns every byte of device memory through its own allocator and exposes
 * none of it, or a latency-critical decode loop that must never call cudaMalloc/cudaFree
 * (cudaFree synchronises the whole device and would stall every other stream).  This entry
 * point computes exactly what sfa_gather_attend computes, with the same kernels, but takes its
 * split-KV scratch from a fixed array compiled into libsfa (SFA_NOALLOC_SCRATCH_BYTES per GPU,
 * held by every GPU that loads the library until the process exits) instead of `workspace`.
 * It calls no cudaMalloc, cudaFree or allocating library routine.
 *
 *  - Arguments and results are those of sfa_gather_attend without the workspace pair; the
 *    caller still owns Q, K, V, the block lists, O and lse.
 *  - If the scratch that this shape needs (sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv,
 *    top_k*cr + cr - 1)) exceeds SFA_NOALLOC_SCRATCH_BYTES the call returns
 *    SFA_ERR_WORKSPACE and enqueues nothing; use sfa_gather_attend with a workspace instead.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call before any stream
 *    capture begins.
 *  - Every call on a device shares the one array and leaves the last call's partial results
 *    in it.  Nothing in it needs to start at zero: every split writes its partial before the
 *    merge reads it.  Calls whose work overlaps on the GPU (for example on two streams at
 *    once) race on the array: order them on one stream or with events.
 */
#define SFA_NOALLOC_SCRATCH_BYTES (16u << 20)
int sfa_gather_attend_noalloc(const void *Q, const void *K, const void *V, int dtype, int n_seq,
                              int64_t n_tok_cap, int n_q, int h_q, int h_kv, int dkq, int dv,
                              float scale, const int32_t *q_seq, const int32_t *q_pos,
                              const int32_t *blk_idx, const int32_t *n_sel, int top_k,
                              int compress_ratio, float *O, float *lse, int32_t *dev_status,
                              sfa_stream_t stream);

/*
 * sfa_copy_cache_rows -- plumbing, not part of the method: places n_rows rows of row_bytes
 * bytes, spaced src_pitch bytes apart at src, into rows spaced dst_pitch bytes apart at dst --
 * typically a step's new cache rows (one per sequence) written into their slots of the K, V
 * or index-key caches, or a step's query inputs (one row).  Either side may be device memory
 * or page-locked host memory that the device addresses (unified addressing); the copy is one
 * kernel on `stream` (SM loads and stores, 16 bytes at a time when the addresses, pitches and
 * row size are multiples of 16).  row_bytes >= 1, pitches >= row_bytes, n_rows >= 0;
 * SFA_ERR_INVALID_ARG otherwise, SFA_ERR_CUDA if the launch fails.
 */
int sfa_copy_cache_rows(void *dst, int64_t dst_pitch, const void *src, int64_t src_pitch,
                        int64_t row_bytes, int64_t n_rows, sfa_stream_t stream);
/*
 * sfa_copy_cache_rows_multi -- n (<= SFA_MAX_ROW_COPIES) such copies in one kernel launch
 * (a step's query inputs and the new rows of each cache at once).  Every entry is checked as
 * sfa_copy_cache_rows checks its arguments before anything is launched; entries with n_rows = 0
 * are skipped.  The copies must not overlap one another.
 */
#define SFA_MAX_ROW_COPIES 8
typedef struct {
    void *dst;
    int64_t dst_pitch;
    const void *src;
    int64_t src_pitch;
    int64_t row_bytes;
    int64_t n_rows;
} sfa_row_copy;
int sfa_copy_cache_rows_multi(int n, const sfa_row_copy *copies, sfa_stream_t stream);

/* Copies *dev_status to *host_out after the work already enqueued on `stream` (this call
 * synchronises the stream). */
int sfa_read_device_status(const int32_t *dev_status, int32_t *host_out, sfa_stream_t stream);

/* A static, human-readable name of a status code. */
const char *sfa_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* SFA_H */
