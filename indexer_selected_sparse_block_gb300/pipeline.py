"""One step of indexer-selected block-sparse attention through the C ABI, with its buffers.

``SfaStep`` owns the intermediate device buffers of the method (pooled keys, block scores,
kept block lists, workspaces, outputs) and runs the stages as the C entry points:

  sfa_pool_index_keys -> sfa_index_scores -> sfa_topk_blocks -> sfa_gather_attend

(decode-like steps -- few queries per sequence, rows of at most 131072 blocks -- take a bound
pass -> sfa_topk_blocks_refine for the middle two: the same kept sets from a quarter of the
pooled-key bytes (sfa_index_scores_bounded_i8 on the 8-bit copy that
sfa_quantize_pooled_keys_i8 writes after each pool call; bound_pass="hi":
sfa_index_scores_bounded on the hi halves, half the bytes) plus the rescoring of the few blocks
the bounds cannot rule out)

or, when every query is below the budget (B_i <= indexer_top_k for all i), the dense case
``sfa_dense_attend``: every block then fits the budget, so the method is exactly dense
attention (llama.cpp commit "model: add Qwen3.8-Flash-Next (qwen4exp)", QSA paragraphs).

With ``window > 0`` the attention also covers the ``window`` most recent positions densely
(the dense + sparse + combine variant of PR #27970's review discussion): in one pass over the
whole set, or (``window_mode="split"``) as the kept part and the window part attended apart and
merged by ``sfa_combine_attention``.

With a position -> cell map (``cell_of``), the caches are flat cell arrays in any order (a
paged serving cache) and the pool and the attention take their ``_paged`` entry points; the
scores and the selection work on pooled blocks, which are cut on positions either way.  K and
V may be q8_0 cache rows (uint8 tensors written by ``sfa_quantize_kv_q8_0``): the attention
entry points then take them as ``SFA_Q8_0``; the index keys stay bf16.
"""
from __future__ import annotations

import torch

from . import _binding as B


# Pooled-key bytes per step of the exact scores (n_q * n_blk_max * 4 * d_idx) from which a
# decode-like step takes the bounded selection by default.
BOUNDED_MIN_BYTES = 96 << 20


class SfaStep:
    def __init__(self, *, n_seq: int, n_tok_cap: int, n_q: int, h_q: int, h_kv: int, dkq: int,
                 dv: int, h_idx: int, d_idx: int, compress_ratio: int, indexer_top_k: int,
                 n_blk_max: int, q_group: int = 1, bounded=None, key_transform=None,
                 cell_of=None, window: int = 0, window_mode: str = "single",
                 bound_pass=None, device="cuda"):
        self.__dict__.update(n_seq=n_seq, n_tok_cap=n_tok_cap, n_q=n_q, h_q=h_q, h_kv=h_kv,
                             dkq=dkq, dv=dv, h_idx=h_idx, d_idx=d_idx, cr=compress_ratio,
                             top_k=indexer_top_k, n_blk_max=n_blk_max, q_group=q_group)
        dev = torch.device(device)
        self.blk_cap = n_tok_cap // compress_ratio
        assert n_blk_max <= self.blk_cap
        self.Kbar = torch.zeros(B.kbar_shape(n_seq, self.blk_cap, d_idx), dtype=torch.bfloat16,
                                device=dev)
        self.dense = n_blk_max <= indexer_top_k
        # the norm and rotation of pooled index keys (keyword arguments of
        # sfa_pool_index_keys_transformed), or None: raw pooled keys
        self.key_transform = dict(key_transform) if key_transform else None
        # paged caches: cell_of [n_seq][n_tok_cap] int32 on the device gives the cell of each
        # position; X, K and V are then [n_cells][...] arrays
        self.cell_of = cell_of
        if cell_of is not None:
            if tuple(cell_of.shape) != (n_seq, n_tok_cap) or cell_of.dtype != torch.int32:
                raise ValueError("cell_of must be an int32 [n_seq][n_tok_cap] tensor")
            if self.key_transform:
                raise ValueError("the paged pool takes raw pooled keys (no key transform)")
        # The bounded selection (cheap bound pass + exact rescoring of the blocks the bounds
        # cannot rule out) cuts the pooled-key bytes of decode-like steps, where each query
        # streams its sequence's pooled keys; prefill tiles share those reads and take the
        # exact scores directly.  Rows of at most 131072 blocks.  Its selection is a latency
        # chain of 22-27 us, which pays only once the exact pass would stream enough bytes:
        # measured on GB300, the exact pair was faster up to 67 MB of pooled keys per step
        # (16 queries x 8192 blocks: 48.1 against 50.2 us; one query x 1024 blocks: 31.2
        # against 35.9 us) and slower from 268 MB (4 x 131072 blocks: 91 against 59 us).
        if bounded is None:
            exact_bytes = n_q * n_blk_max * 4 * d_idx
            bounded = (q_group <= 4 and n_blk_max <= B.SFA_REFINE_MAX_BLOCKS
                       and exact_bytes >= BOUNDED_MIN_BYTES)
        self.bounded = bool(bounded) and not self.dense
        if self.bounded and n_blk_max > B.SFA_REFINE_MAX_BLOCKS:
            raise ValueError(f"bounded selection takes rows of at most "
                             f"{B.SFA_REFINE_MAX_BLOCKS} blocks, got n_blk_max={n_blk_max}")
        # bounded: the bound pass reads the 8-bit copy of the pooled keys ("i8": codes, a
        # scale and a bound factor per row, written after each pool call) or the hi halves
        # ("hi": the pooling pass also writes each pooled row's bound factor)
        # Default: the 8-bit pass up to a budget of 1024 blocks.  Its bounds leave about three
        # times the budget as candidates, which the selection resolves in shared memory up to
        # 4096; past that (token-level budgets of 2048) the hi-only pass, whose bounds leave
        # fewer, measured faster.
        if bound_pass is None:
            bound_pass = "i8" if indexer_top_k <= 1024 else "hi"
        if bound_pass not in ("i8", "hi"):
            raise ValueError("bound_pass must be 'i8' or 'hi'")
        self.bound_pass = bound_pass if self.bounded else None
        cap = max(self.blk_cap, 1)
        self.Kbar_r = (torch.zeros((n_seq, cap), dtype=torch.float32, device=dev)
                       if self.bound_pass == "hi" else None)
        if self.bound_pass == "i8":
            k8, sr = B.k8_shapes(n_seq, cap, d_idx)
            self.K8 = torch.zeros(k8, dtype=torch.int8, device=dev)
            self.K8_sr = torch.zeros(sr, dtype=torch.float32, device=dev)
        self.scores = torch.empty((n_q, max(n_blk_max, 1)), dtype=torch.float32, device=dev)
        # bounded: scores holds the lower bounds and upper the upper bounds
        self.upper = (torch.empty_like(self.scores) if self.bounded else None)
        nr = B.sfa_topk_refine_workspace_bytes(n_q, max(n_blk_max, 1)) if self.bounded else 0
        self.refine_ws = torch.empty(max(nr, 16), dtype=torch.uint8, device=dev)
        self.blk_idx = torch.empty((n_q, indexer_top_k), dtype=torch.int32, device=dev)
        self.n_sel = torch.empty(n_q, dtype=torch.int32, device=dev)
        nt = B.sfa_topk_workspace_bytes(n_q, max(n_blk_max, 1), indexer_top_k)
        self.topk_ws = torch.empty(max(nt, 16), dtype=torch.uint8, device=dev)
        # the dense window of recent keys beside the kept blocks (window > 0): one pass over
        # the whole set ("single"), or the kept part and the window part attended apart and
        # combined by their log-sum-exp ("split")
        if window < 0 or window_mode not in ("single", "split"):
            raise ValueError("window must be >= 0 and window_mode 'single' or 'split'")
        if window and cell_of is not None:
            raise ValueError("the windowed attention takes the per-sequence layout")
        self.window, self.window_mode = int(window), window_mode
        self.n_kv_dense = n_tok_cap
        n_kv = (n_tok_cap if self.dense else
                B.sfa_window_kv_max(indexer_top_k, compress_ratio, self.window, 0))
        na = B.sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv)
        self.attn_ws = torch.empty(max(na, 16), dtype=torch.uint8, device=dev)
        self.O = torch.empty((n_q, h_q, dv), dtype=torch.float32, device=dev)
        self.lse = torch.empty((n_q, h_q), dtype=torch.float32, device=dev)
        if self.window and window_mode == "split" and not self.dense:
            self.O_sel, self.O_win = torch.empty_like(self.O), torch.empty_like(self.O)
            self.lse_sel, self.lse_win = torch.empty_like(self.lse), torch.empty_like(self.lse)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def set_output(self, O):
        """Makes O the buffer the attention writes: a [n_q][h_q][dv] fp32 tensor on the device,
        or in page-locked host memory, which the attention kernels then write directly (no
        separate read-back).  The split window mode keeps its partial parts on the device and
        only the merged result goes to O.  Returns the buffer it replaces."""
        if tuple(O.shape) != tuple(self.O.shape) or O.dtype != torch.float32:
            raise ValueError(f"O must be a float32 tensor of shape {tuple(self.O.shape)}")
        if not O.is_contiguous() or not (O.is_cuda or O.is_pinned()):
            raise ValueError("O must be contiguous, on the device or in page-locked host memory")
        old, self.O = self.O, O
        return old

    def pool(self, X, blk_begin: int, blk_end: int, stream=None):
        if blk_end > blk_begin:
            if self.cell_of is not None:
                B.sfa_pool_index_keys_paged(X, self.cell_of, self.cr, blk_begin, blk_end,
                                            self.Kbar, self.Kbar_r, dev_status=self.status,
                                            stream=stream)
            elif self.key_transform:
                B.sfa_pool_index_keys_transformed(X, self.cr, blk_begin, blk_end, self.Kbar,
                                                  self.Kbar_r, stream=stream, **self.key_transform)
            else:
                B.sfa_pool_index_keys(X, self.cr, blk_begin, blk_end, self.Kbar, self.Kbar_r,
                                      stream=stream)
            if self.bound_pass == "i8":
                B.sfa_quantize_pooled_keys_i8(self.Kbar, blk_begin, blk_end, self.K8, self.K8_sr,
                                              stream=stream)

    def score(self, q_idx, w, q_seq, q_pos, stream=None):
        if self.bound_pass == "i8":
            B.sfa_index_scores_bounded_i8(q_idx, w, q_seq, q_pos, self.K8, self.K8_sr, self.cr,
                                          self.n_blk_max, self.scores, self.upper,
                                          dev_status=self.status, stream=stream)
        elif self.bounded:
            B.sfa_index_scores_bounded(q_idx, w, q_seq, q_pos, self.Kbar, self.Kbar_r, self.cr,
                                       self.n_blk_max, self.scores, self.upper,
                                       q_group=self.q_group, dev_status=self.status,
                                       stream=stream)
        else:
            B.sfa_index_scores(q_idx, w, q_seq, q_pos, self.Kbar, self.cr, self.n_blk_max,
                               self.scores, q_group=self.q_group, dev_status=self.status,
                               stream=stream)

    def topk(self, q_idx, w, q_seq, q_pos, stream=None):
        if self.bounded:
            B.sfa_topk_blocks_refine(self.scores, self.upper, q_idx, w, q_seq, q_pos, self.Kbar,
                                     self.cr, self.top_k, self.n_blk_max, self.blk_idx,
                                     self.n_sel, workspace=self.refine_ws,
                                     dev_status=self.status, stream=stream)
        else:
            B.sfa_topk_blocks(self.scores, q_pos, self.cr, self.top_k, self.n_blk_max,
                              self.blk_idx, self.n_sel, workspace=self.topk_ws,
                              dev_status=self.status, stream=stream)

    def select(self, q_idx, w, q_seq, q_pos, stream=None):
        self.score(q_idx, w, q_seq, q_pos, stream=stream)
        self.topk(q_idx, w, q_seq, q_pos, stream=stream)

    def attend(self, Q, K, V, q_seq, q_pos, scale: float, stream=None):
        if self.cell_of is not None:
            if self.dense:
                B.sfa_dense_attend_paged(Q, K, V, self.cell_of, q_seq, q_pos, self.n_kv_dense,
                                         scale, self.O, lse=self.lse, workspace=self.attn_ws,
                                         dev_status=self.status, stream=stream)
            else:
                B.sfa_gather_attend_paged(Q, K, V, self.cell_of, q_seq, q_pos, self.blk_idx,
                                          self.n_sel, self.top_k, self.cr, scale, self.O,
                                          lse=self.lse, workspace=self.attn_ws,
                                          dev_status=self.status, stream=stream)
        elif self.dense:
            B.sfa_dense_attend(Q, K, V, q_seq, q_pos, self.n_kv_dense, scale, self.O,
                               lse=self.lse, workspace=self.attn_ws, dev_status=self.status,
                               stream=stream)
        elif self.window and self.window_mode == "single":
            B.sfa_gather_attend_window(Q, K, V, q_seq, q_pos, self.blk_idx, self.n_sel,
                                       self.top_k, self.cr, self.window, scale, self.O,
                                       lse=self.lse, part=B.SFA_PART_ALL, workspace=self.attn_ws,
                                       dev_status=self.status, stream=stream)
        elif self.window:
            for part, O, lse in ((B.SFA_PART_SELECTED, self.O_sel, self.lse_sel),
                                 (B.SFA_PART_WINDOW, self.O_win, self.lse_win)):
                B.sfa_gather_attend_window(Q, K, V, q_seq, q_pos, self.blk_idx, self.n_sel,
                                           self.top_k, self.cr, self.window, scale, O, lse=lse,
                                           part=part, workspace=self.attn_ws,
                                           dev_status=self.status, stream=stream)
            B.sfa_combine_attention(self.O_sel, self.lse_sel, self.O_win, self.lse_win, self.O,
                                    self.lse, stream=stream)
        else:
            B.sfa_gather_attend(Q, K, V, q_seq, q_pos, self.blk_idx, self.n_sel, self.top_k,
                                self.cr, scale, self.O, lse=self.lse, workspace=self.attn_ws,
                                dev_status=self.status, stream=stream)

    @staticmethod
    def graphed(fn, warmup: int = 2):
        """fn() captured into a CUDA graph, after `warmup` runs on a side stream.  The entry
        points launch on the current stream and never synchronise or allocate, so a step of
        them -- with the caller's input copies and output read-back -- replays as one graph
        launch (torch.cuda.CUDAGraph.replay()), free of per-call host overhead."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def run(self, X, K, V, Q, q_idx, w, q_seq, q_pos, scale: float, new_blocks=(0, 0),
            stream=None):
        """One step: pool the blocks completed by this step's tokens, score, select, attend."""
        self.pool(X, new_blocks[0], new_blocks[1], stream=stream)
        if not self.dense:
            self.select(q_idx, w, q_seq, q_pos, stream=stream)
        self.attend(Q, K, V, q_seq, q_pos, scale, stream=stream)
        return self.O
