"""Paged (non-contiguous) cell layout: the pool and the attention read each position's rows
through a per-stream position -> cell map.  Blocks stay cuts of the position line, so the
paged calls must give bit for bit what the per-sequence calls give on the gathered layout, and
match the oracle run through the same map."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, TOL_F32, np32, row_rel_err

pytestmark = pytest.mark.gpu

sfa = pytest.importorskip("indexer_selected_sparse_block_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _randn(shape, gen, dtype):
    return torch.randn(shape, generator=gen).to(torch.bfloat16).to(dtype)


def _cell_map(n_seq, n_pos, layout, rng, page=16, spare=5):
    """[n_seq][n_pos] int32 map and the cell count.  "pages": each sequence's positions fill
    pages of `page` consecutive cells, the pages shuffled over the array with `spare` unused
    ones among them (a serving cache's page table); "cells": every position in a random cell."""
    if layout == "pages":
        pps = -(-n_pos // page)
        n_cells = (n_seq * pps + spare) * page
        perm = rng.permutation(n_seq * pps + spare)[: n_seq * pps].reshape(n_seq, pps)
        t = np.arange(n_pos)
        cell_of = perm[:, t // page] * page + (t % page)[None, :]
    else:
        n_cells = n_seq * n_pos + spare * page
        cell_of = rng.permutation(n_cells)[: n_seq * n_pos].reshape(n_seq, n_pos)
    return np.ascontiguousarray(cell_of, dtype=np.int32), n_cells


def _scatter(Xc, cell_of, n_cells, gen):
    """The cell array holding Xc[s][t] in cell cell_of[s][t]; cells no position maps to hold
    other random values (a read of a wrong cell shows)."""
    n_seq, n_pos = cell_of.shape
    cells = _randn((n_cells,) + tuple(Xc.shape[2:]), gen, Xc.dtype)
    cells[torch.from_numpy(cell_of.reshape(-1)).long()] = Xc.reshape((n_seq * n_pos,) + tuple(Xc.shape[2:]))
    return cells


# --------------------------------------------------------------------------------- pooling
@pytest.mark.parametrize("layout", ["pages", "cells"])
@pytest.mark.parametrize("cr,d_idx,xdtype", [(4, 128, torch.bfloat16), (1, 64, torch.bfloat16),
                                             (8, 32, torch.float32), (3, 96, torch.bfloat16)])
def test_pool_paged(dev, layout, cr, d_idx, xdtype):
    g = torch.Generator().manual_seed(cr * 100 + d_idx)
    rng = np.random.default_rng(cr + d_idx)
    n_seq, n_pos = 3, 1200 + cr
    Xc = _randn((n_seq, n_pos, d_idx), g, xdtype)
    cell_of, n_cells = _cell_map(n_seq, n_pos, layout, rng)
    cells = _scatter(Xc, cell_of, n_cells, g)
    blk_cap = n_pos // cr + 4
    b0, b1 = 2, n_pos // cr
    with_r = d_idx != 96
    outs = []
    for paged in (False, True):
        Kbar = torch.full(sfa.kbar_shape(n_seq, blk_cap, d_idx), 7.0, dtype=torch.bfloat16, device=dev)
        Kr = torch.full((n_seq, blk_cap), -1.0, device=dev) if with_r else None
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if paged:
            sfa.sfa_pool_index_keys_paged(cells.to(dev), torch.from_numpy(cell_of).to(dev), cr, b0,
                                          b1, Kbar, Kr, dev_status=status)
        else:
            sfa.sfa_pool_index_keys(Xc.to(dev), cr, b0, b1, Kbar, Kr)
        torch.cuda.synchronize()
        assert sfa.sfa_read_device_status(status) == 0
        outs.append((Kbar, Kr))
    assert torch.equal(outs[0][0], outs[1][0])
    if with_r:
        assert torch.equal(outs[0][1], outs[1][1])
    kb = np32(outs[1][0]).astype(np.float64)
    got = kb[..., :d_idx] + kb[..., d_idx:]
    cn = np32(cells)
    for s in range(n_seq):
        ref = oracle.pool_cells(cn, cell_of[s], b1, cr)
        mag = np.abs(cn[cell_of[s, : b1 * cr]].astype(np.float64)).reshape(b1, cr, d_idx).mean(1)
        assert np.all(np.abs(got[s, b0:b1] - ref[b0:b1]) <= 2.0 ** -16 * mag[b0:b1] + 1e-30)
    assert np.all(kb[:, :b0] == 7.0) and np.all(kb[:, b1:] == 7.0)


# ------------------------------------------------------------------------------- attention
def _selection(q_pos, cr, top_k, rng):
    sel = np.full((len(q_pos), top_k), -1, np.int32)
    n_sel = np.zeros(len(q_pos), np.int32)
    for i, p in enumerate(q_pos):
        B = (int(p) + 1) // cr
        n = min(top_k, B)
        sel[i, :n] = np.sort(rng.choice(B, size=n, replace=False)) if n else []
        n_sel[i] = n
    return sel, n_sel


def _attend_inputs(dkq, dv, v_is_k, h_q, h_kv, n_seq, n_pos, n_q, dtype, layout, seed):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    Kc = _randn((n_seq, n_pos, h_kv, dkq), g, dtype)
    Vc = None if v_is_k else _randn((n_seq, n_pos, h_kv, dv), g, dtype)
    Q = _randn((n_q, h_q, dkq), g, dtype)
    cell_of, n_cells = _cell_map(n_seq, n_pos, layout, rng)
    Kp = _scatter(Kc, cell_of, n_cells, g)
    Vp = None if v_is_k else _scatter(Vc, cell_of, n_cells, g)
    return Q, Kc, Vc, Kp, Vp, cell_of, rng


SHAPES = [(576, 512, True, 16, 1), (512, 512, False, 16, 2), (128, 128, False, 8, 2)]


@pytest.mark.parametrize("layout", ["pages", "cells"])
@pytest.mark.parametrize("dkq,dv,v_is_k,h_q,h_kv", SHAPES)
@pytest.mark.parametrize("mode", ["decode", "decode32", "prefill"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_gather_attend_paged(dev, layout, dkq, dv, v_is_k, h_q, h_kv, mode, dtype):
    """Decode rows (2048 kept cells and a tail: 4 queries split over many CTAs and merged by a
    second kernel; 32 queries split over an 8-CTA cluster, the tail folded into the last split
    where V = K) and prefill rows (one CTA each)."""
    cr = 4
    if mode == "decode":
        n_seq, n_pos, top_k = 3, 2600, 512
        q_seq = np.array([0, 1, 2, 1], np.int32)
        q_pos = np.array([2599, 2100, 900, 2], np.int32)
    elif mode == "decode32":
        n_seq, n_pos, top_k = 3, 2600, 512
        q_seq = (np.arange(32) % 3).astype(np.int32)
        q_pos = np.array([2599, 2100, 900, 2, 2598, 2597, 1, 0] * 4, np.int32)
    else:
        n_seq, n_pos, top_k = 1, 700, 40
        q_seq = np.zeros(120, np.int32)
        q_pos = np.arange(580, 700, dtype=np.int32)
    Q, Kc, Vc, Kp, Vp, cell_of, rng = _attend_inputs(dkq, dv, v_is_k, h_q, h_kv, n_seq, n_pos,
                                                     len(q_seq), dtype, layout, dkq + h_q)
    sel, n_sel = _selection(q_pos, cr, top_k, rng)
    scale = 1.0 / math.sqrt(dkq)
    d = lambda a: torch.from_numpy(a).to(dev)
    res = []
    for paged in (False, True):
        O = torch.full((len(q_seq), h_q, dv), float("nan"), device=dev)
        lse = torch.full((len(q_seq), h_q), float("nan"), device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if paged:
            sfa.sfa_gather_attend_paged(Q.to(dev), Kp.to(dev), None if Vp is None else Vp.to(dev),
                                        d(cell_of), d(q_seq), d(q_pos), d(sel), d(n_sel), top_k,
                                        cr, scale, O, lse=lse, dev_status=status)
        else:
            sfa.sfa_gather_attend(Q.to(dev), Kc.to(dev), None if Vc is None else Vc.to(dev),
                                  d(q_seq), d(q_pos), d(sel), d(n_sel), top_k, cr, scale, O,
                                  lse=lse, dev_status=status)
        torch.cuda.synchronize()
        assert sfa.sfa_read_device_status(status) == 0
        res.append((O, lse))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])
    Kn, Vn, Qn = np32(Kp), np32(Vp), np32(Q)
    On, Ln = np32(res[1][0]), np32(res[1][1])
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    for i in range(len(q_seq)):
        s, p = int(q_seq[i]), int(q_pos[i])
        msk = oracle.mask(p, cr, sel[i], int(n_sel[i]))
        ref, rlse = oracle.attend(Qn[i], Kn, Vn, msk, scale, h_kv, dv=dv,
                                  tok_row=cell_of[s, : p + 1])
        assert row_rel_err(On[i], ref).max() < tol, i
        assert np.abs(Ln[i] - rlse).max() < (2e-3 if dtype == torch.bfloat16 else 1e-5), i


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_dense_attend_paged(dev, dtype):
    dkq, dv, h_q, h_kv = 576, 512, 16, 1
    n_seq, n_pos = 2, 1100
    q_seq = np.array([0, 1, 1, 0], np.int32)
    q_pos = np.array([1099, 0, 517, 64], np.int32)
    Q, Kc, _, Kp, _, cell_of, _ = _attend_inputs(dkq, dv, True, h_q, h_kv, n_seq, n_pos,
                                                 len(q_seq), dtype, "pages", 23)
    scale = 1.0 / math.sqrt(dkq)
    d = lambda a: torch.from_numpy(a).to(dev)
    O1 = torch.empty((len(q_seq), h_q, dv), device=dev)
    O2 = torch.empty_like(O1)
    sfa.sfa_dense_attend(Q.to(dev), Kc.to(dev), None, d(q_seq), d(q_pos), n_pos, scale, O1)
    sfa.sfa_dense_attend_paged(Q.to(dev), Kp.to(dev), None, d(cell_of), d(q_seq), d(q_pos), n_pos,
                               scale, O2)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2)
    Kn, Qn, On = np32(Kp), np32(Q), np32(O2)
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    for i in range(len(q_seq)):
        s, p = int(q_seq[i]), int(q_pos[i])
        ref, _ = oracle.attend(Qn[i], Kn, None, oracle.mask(p, 4, dense=True), scale, h_kv, dv=dv,
                               tok_row=cell_of[s, : p + 1])
        assert row_rel_err(On[i], ref).max() < tol


def test_paged_ignores_tcgen05_opt_in(dev, monkeypatch):
    """With the tcgen05 kernel asked for, the paged call still takes the mma.sync kernel and
    gives the default contiguous result bit for bit."""
    dkq, dv, h_q, h_kv, cr, top_k = 576, 512, 16, 1, 4, 512
    q_seq = np.array([0, 1], np.int32)
    q_pos = np.array([2599, 1500], np.int32)
    Q, Kc, _, Kp, _, cell_of, rng = _attend_inputs(dkq, dv, True, h_q, h_kv, 2, 2600, 2,
                                                   torch.bfloat16, "pages", 5)
    sel, n_sel = _selection(q_pos, cr, top_k, rng)
    d = lambda a: torch.from_numpy(a).to(dev)
    O1 = torch.empty((2, h_q, dv), device=dev)
    O2 = torch.empty_like(O1)
    sfa.sfa_gather_attend(Q.to(dev), Kc.to(dev), None, d(q_seq), d(q_pos), d(sel), d(n_sel),
                          top_k, cr, 0.04, O1)
    monkeypatch.setenv("SFA_ATTEND_KERNEL", "tcgen05")
    sfa.sfa_gather_attend_paged(Q.to(dev), Kp.to(dev), None, d(cell_of), d(q_seq), d(q_pos),
                                d(sel), d(n_sel), top_k, cr, 0.04, O2)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2)


def test_bad_cells_are_flagged_and_left_out(dev):
    """Map entries outside [0, n_cells) raise SFA_DEV_BAD_CELL without being read: the pool
    counts such a position as a zero row, the attention leaves it out of the softmax."""
    dkq, dv, h_q, h_kv, cr, top_k = 576, 512, 16, 1, 4, 64
    n_seq, n_pos = 2, 604
    q_seq = np.array([0, 1], np.int32)
    q_pos = np.array([602, 602], np.int32)          # 150 whole blocks and a 3-cell tail
    Q, _, _, Kp, _, cell_of, rng = _attend_inputs(dkq, dv, True, h_q, h_kv, n_seq, n_pos, 2,
                                                  torch.bfloat16, "cells", 31)
    n_cells = Kp.shape[0]
    sel, n_sel = _selection(q_pos, cr, top_k, rng)
    bad = cell_of.copy()
    hit = [int(sel[0, 3]) * cr + 1, 601]            # a kept block's cell and a tail cell
    bad[0, hit[0]] = -5
    bad[0, hit[1]] = n_cells + 3
    d = lambda a: torch.from_numpy(a).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    O = torch.empty((2, h_q, dv), device=dev)
    sfa.sfa_gather_attend_paged(Q.to(dev), Kp.to(dev), None, d(bad), d(q_seq), d(q_pos), d(sel),
                                d(n_sel), top_k, cr, 0.04, O, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) & sfa.SFA_DEV_BAD_CELL
    Kn, Qn, On = np32(Kp), np32(Q), np32(O)
    for i in range(2):
        msk = oracle.mask(602, cr, sel[i], int(n_sel[i]))
        if i == 0:   # both bad positions are attended by query 0, and then left out
            assert msk[hit].all()
            msk[hit] = 0
        rows = cell_of[i, :603]
        ref, _ = oracle.attend(Qn[i], Kn, None, msk, 0.04, h_kv, dv=dv, tok_row=rows)
        assert row_rel_err(On[i], ref).max() < TOL_BF16, i
    # the pool: sequence 0's rows through the map with the bad positions as zero rows
    X = _randn((n_cells, 64), torch.Generator().manual_seed(2), torch.bfloat16)
    Kbar = torch.zeros(sfa.kbar_shape(n_seq, 150, 64), dtype=torch.bfloat16, device=dev)
    status.zero_()
    sfa.sfa_pool_index_keys_paged(X.to(dev), d(bad), cr, 0, 150, Kbar, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) & sfa.SFA_DEV_BAD_CELL
    Xn = np32(X).astype(np.float64)
    rows = np.where((bad[0] >= 0) & (bad[0] < n_cells), bad[0], 0)
    G = Xn[rows]
    G[(bad[0] < 0) | (bad[0] >= n_cells)] = 0.0
    want = G[:600].reshape(150, cr, 64).mean(1)
    kb = np32(Kbar).astype(np.float64)
    got = kb[0, :, :64] + kb[0, :, 64:]
    assert np.all(np.abs(got - want) <= 2.0 ** -16 * np.abs(G[:600]).reshape(150, cr, 64).mean(1) + 1e-30)


# ------------------------------------------------------------------------------ whole step
STEPS = [("decode_1x4096", True, {}),                                   # bounded selection
         ("decode_32x131072", False, {"n_seq": 4, "depth": 20000}),    # exact, 4 sequences
         ("prefill_512x1000", None, {}),                                # below budget: dense
         ("decode_4x1048576", None, {"n_seq": 2, "depth": 70000})]      # separate V, cr 8


@pytest.mark.parametrize("name,bounded,shrink", STEPS, ids=[s[0] for s in STEPS])
def test_step_paged_equals_contiguous(dev, name, bounded, shrink):
    """SfaStep on a paged cache (64-cell pages, shuffled) keeps the same blocks and gives the
    same outputs, bit for bit, as on the per-sequence cache."""
    w = sfa.WORKLOADS[name]
    if shrink:
        w = w.with_(**shrink)
    case = sfa.make_case(w, device=dev)
    cell_of, n_cells = sfa.make_cell_map(w.n_seq, w.n_tok, page=64, spare_pages=w.n_seq, seed=3,
                                         device=dev)
    paged = {n: None if case[n] is None else sfa.to_cells(case[n], cell_of, n_cells)
             for n in ("X", "K", "V")}
    n_blk_max = w.n_tok // w.compress_ratio
    runs = []
    for cm in (None, cell_of):
        st = sfa.SfaStep(n_seq=w.n_seq, n_tok_cap=w.n_tok, n_q=w.n_q, h_q=w.h_q, h_kv=w.h_kv,
                         dkq=w.dkq, dv=w.dv, h_idx=w.h_idx, d_idx=w.d_idx,
                         compress_ratio=w.compress_ratio, indexer_top_k=w.indexer_top_k,
                         n_blk_max=n_blk_max, q_group=w.n_q_per_seq, bounded=bounded,
                         cell_of=cm, device=dev)
        src = case if cm is None else paged
        st.run(src["X"], src["K"], src["V"], case["Q"], case["q_idx"], case["w"], case["q_seq"],
               case["q_pos"], w.scale, new_blocks=(0, n_blk_max))
        torch.cuda.synchronize()
        assert sfa.sfa_read_device_status(st.status) == 0
        runs.append(st)
    a, b = runs
    assert a.dense == b.dense and a.bounded == b.bounded
    assert torch.equal(a.Kbar, b.Kbar)
    if not a.dense:
        assert torch.equal(a.n_sel, b.n_sel)
        for i in range(w.n_q):
            n = int(a.n_sel[i])
            assert torch.equal(a.blk_idx[i, :n], b.blk_idx[i, :n])
    assert torch.equal(a.O, b.O) and torch.equal(a.lse, b.lse)
