"""Seeded synthetic inputs for indexer-selected block-sparse attention.

This module is the one piece shared by the CUDA path's tests/bench and the oracle: it
draws inputs and holds none of the method's arithmetic.  Values follow the workloads of
the pages (llama.cpp PR #27970 measures DeepSeek-V4 decode ``tg32@dN`` and prefill
``pp2048@dN``; the QSA commit for qwen4exp sets compress_ratio and indexer_top_k), with
trained weights replaced by seeded draws:

* K cache, Q, index keys X and index queries: N(0, 1) in fp32 from a seeded
  ``torch.Generator``, rounded to bf16 (round to nearest even);
* index head weights w: U(0, 1) fp32;
* decode at depth d: the query sits at position d and sees d + 1 cached tokens;
* prefill of n tokens at depth d: queries at positions d .. d + n - 1 (causal), the cache
  holds d + n tokens.

Every tensor has its own generator seeded from (seed, tensor role, sequence), so a
tensor's values do not depend on which other tensors were drawn, and big caches are drawn
in chunks directly on the target device.
"""
from __future__ import annotations

import dataclasses
import math

import torch

__all__ = ["Workload", "WORKLOADS", "make_case", "draw_normal_bf16", "draw_uniform",
           "make_cell_map", "to_cells"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one workload (names follow the pages' notation)."""
    name: str
    kind: str            # "decode" or "prefill"
    n_seq: int           # independent sequences (streams)
    n_q_per_seq: int     # query tokens per sequence in this step
    depth: int           # cached tokens before the first query token
    h_q: int             # query heads
    h_kv: int            # KV heads (latent heads for MLA-shaped K)
    dkq: int             # K/Q head size
    dv: int              # V head size
    v_is_k: bool         # V is the first dv dims of K (MLA layout)
    h_idx: int           # indexer heads
    d_idx: int           # indexer head size
    compress_ratio: int  # tokens per pooled block
    indexer_top_k: int   # budget in blocks (the tail is kept on top of it)
    seed: int = 0

    @property
    def n_q(self) -> int:
        return self.n_seq * self.n_q_per_seq

    @property
    def n_tok(self) -> int:
        return self.depth + self.n_q_per_seq

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dkq)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The synthetic workloads: three decode shapes (1 sequence at depth 4096; 32 sequences at
# depth 131072; 4 sequences of two KV heads at depth 1048576) and two prefill shapes
# (512 tokens at depth 8192, also at depth 1000 where every block fits the budget; 2048
# tokens at depth 131072, the pp2048@d131072 shape); and token-level selection
# (compress_ratio 1) at 32 sequences of depth 32768.
WORKLOADS = {
    "decode_1x4096": Workload("decode_1x4096", "decode", 1, 1, 4096, 16, 1, 576, 512, True,
                              4, 64, 4, 256, seed=1000),
    "prefill_512x8192": Workload("prefill_512x8192", "prefill", 1, 512, 8192, 16, 1, 576, 512,
                                 True, 4, 64, 4, 512, seed=1001),
    "prefill_512x1000": Workload("prefill_512x1000", "prefill", 1, 512, 1000, 16, 1, 576, 512,
                                 True, 4, 64, 4, 512, seed=1011),
    "decode_32x131072": Workload("decode_32x131072", "decode", 32, 1, 131072, 16, 1, 576, 512,
                                 True, 8, 128, 4, 512, seed=1002),
    "pp2048_131072": Workload("pp2048_131072", "prefill", 1, 2048, 131072, 16, 1, 576, 512,
                              True, 8, 128, 4, 512, seed=1003),
    "decode_4x1048576": Workload("decode_4x1048576", "decode", 4, 1, 1048576, 16, 2, 512, 512,
                                 False, 8, 128, 8, 256, seed=1004),
    # token-level selection (compress_ratio 1: every token its own block, a budget of 2048
    # tokens), at 32 sequences of depth 32768
    "decode_cr1_32x32768": Workload("decode_cr1_32x32768", "decode", 32, 1, 32768, 16, 1, 576,
                                    512, True, 16, 128, 1, 2048, seed=1005),
}

_ROLE = {"K": 1, "V": 2, "X": 3, "Q": 4, "QI": 5, "W": 6}
_CHUNK = 1 << 26


def _gen(seed: int, role: str, part: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + _ROLE[role] * 7919 + part) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def draw_normal_bf16(shape, seed: int, role: str, part: int, device, out=None):
    """N(0,1) fp32 draws rounded to bf16, drawn in chunks (same values on any chunking of
    the caller's side: the chunk size is fixed here)."""
    device = torch.device(device)
    n = math.prod(shape)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    g = _gen(seed, role, part, device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        flat[s:e].copy_(torch.randn(e - s, generator=g, device=device, dtype=torch.float32))
    return out


def draw_uniform(shape, seed: int, role: str, part: int, device):
    g = _gen(seed, role, part, torch.device(device))
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def make_case(w: Workload, device="cpu", dtype=torch.bfloat16, n_tok_cap: int | None = None):
    """Draw one step's inputs for workload ``w`` on ``device``.

    Returns a dict of tensors (all contiguous):
      X     [n_seq][n_tok_cap][d_idx]   bf16 raw index keys (rows >= n_tok are zero)
      K     [n_seq][n_tok_cap][h_kv][dkq] ``dtype``
      V     [n_seq][n_tok_cap][h_kv][dv]  ``dtype`` or None (V = K[..., :dv])
      Q     [n_q][h_q][dkq] ``dtype``;  q_idx [n_q][h_idx][d_idx] bf16;  w [n_q][h_idx] f32
      q_seq, q_pos [n_q] int32
    ``dtype`` float32 gives the fp32-input variant (values are the same bf16-rounded draws).
    """
    cap = n_tok_cap or w.n_tok
    assert cap >= w.n_tok
    dev = torch.device(device)
    X = torch.zeros((w.n_seq, cap, w.d_idx), dtype=torch.bfloat16, device=dev)
    K = torch.zeros((w.n_seq, cap, w.h_kv, w.dkq), dtype=dtype, device=dev)
    V = None if w.v_is_k else torch.zeros((w.n_seq, cap, w.h_kv, w.dv), dtype=dtype, device=dev)
    for s in range(w.n_seq):
        draw_normal_bf16((w.n_tok, w.d_idx), w.seed, "X", s, dev, out=X[s, : w.n_tok])
        if dtype == torch.bfloat16:
            draw_normal_bf16((w.n_tok, w.h_kv, w.dkq), w.seed, "K", s, dev, out=K[s, : w.n_tok])
            if V is not None:
                draw_normal_bf16((w.n_tok, w.h_kv, w.dv), w.seed, "V", s, dev, out=V[s, : w.n_tok])
        else:
            K[s, : w.n_tok] = draw_normal_bf16((w.n_tok, w.h_kv, w.dkq), w.seed, "K", s, dev).to(dtype)
            if V is not None:
                V[s, : w.n_tok] = draw_normal_bf16((w.n_tok, w.h_kv, w.dv), w.seed, "V", s, dev).to(dtype)
    Q = draw_normal_bf16((w.n_q, w.h_q, w.dkq), w.seed, "Q", 0, dev).to(dtype)
    q_idx = draw_normal_bf16((w.n_q, w.h_idx, w.d_idx), w.seed, "QI", 0, dev)
    wts = draw_uniform((w.n_q, w.h_idx), w.seed, "W", 0, dev)
    q_seq = torch.arange(w.n_seq, dtype=torch.int32, device=dev).repeat_interleave(w.n_q_per_seq)
    q_pos = (w.depth + torch.arange(w.n_q_per_seq, dtype=torch.int32, device=dev)).repeat(w.n_seq)
    return {"X": X, "K": K, "V": V, "Q": Q, "q_idx": q_idx, "w": wts, "q_seq": q_seq,
            "q_pos": q_pos}


def make_cell_map(n_seq: int, n_pos: int, page: int = 64, spare_pages: int = 0, seed: int = 0,
                  device="cpu"):
    """A paged cache layout: each sequence's positions fill pages of ``page`` consecutive
    cells, dealt from a seeded random permutation of n_seq * ceil(n_pos / page) + spare_pages
    pages (the spare pages stay unused).  Returns (cell_of [n_seq][n_pos] int32, n_cells)."""
    pps = -(-n_pos // page)
    n_pages = n_seq * pps + spare_pages
    g = torch.Generator()
    g.manual_seed(seed)
    perm = torch.randperm(n_pages, generator=g)[: n_seq * pps].view(n_seq, pps)
    t = torch.arange(n_pos)
    cell_of = perm[:, t // page] * page + t % page
    return cell_of.to(torch.int32).to(device), n_pages * page


def to_cells(x, cell_of, n_cells: int):
    """The flat cell array of the per-sequence tensor x [n_seq][n_pos][...]: row cell_of[s][t]
    holds x[s][t]; unused cells are zero."""
    tail = tuple(x.shape[2:])
    cells = torch.zeros((n_cells,) + tail, dtype=x.dtype, device=x.device)
    cells.index_copy_(0, cell_of.reshape(-1).to(x.device).long(), x.reshape((-1,) + tail))
    return cells
