"""Quantized KV cache (q8_0): the quantization kernel against the oracle's rule bit for bit, and
the attention over q8_0 rows (gathered, dense, paged, whole steps) against the oracle's
attention over the values the codes stand for."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, np32, row_rel_err

pytestmark = pytest.mark.gpu

sfa = pytest.importorskip("indexer_selected_sparse_block_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _randn(shape, gen, dtype=torch.bfloat16):
    return torch.randn(shape, generator=gen).to(torch.bfloat16).to(dtype)


def _quantize(x, dev):
    """GPU q8_0 rows of x [..., d] (any leading shape, contiguous) -> uint8 [..., row_bytes]."""
    d = x.shape[-1]
    rb = sfa.sfa_q8_0_row_bytes(d)
    xd = x.to(dev).contiguous()
    y = torch.empty(x.shape[:-1] + (rb,), dtype=torch.uint8, device=dev)
    sfa.sfa_quantize_kv_q8_0(xd.view(1, -1, d), y.view(1, -1, rb))
    return y


def _split_rows(y, d):
    """(codes int8 [..., d], scale bits uint16 [..., d/32], padding bytes) of q8_0 rows."""
    a = y.cpu().numpy()
    codes = a[..., :d].view(np.int8)
    scales = np.ascontiguousarray(a[..., d: d + d // 16]).view(np.uint16)
    return codes, scales, a[..., d + d // 16:]


def _oracle_values(x):
    """The values the oracle's q8_0 codes of x stand for (float32, same shape)."""
    q, s = oracle.quantize_q8_0(np32(x))
    return oracle.dequantize_q8_0(q, s)


# ------------------------------------------------------------------------------ quantization
@pytest.mark.parametrize("d", [576, 512, 128, 64])
@pytest.mark.parametrize("xdtype", [torch.bfloat16, torch.float32])
def test_quantize_matches_oracle(dev, d, xdtype):
    g = torch.Generator().manual_seed(d)
    n_outer, n_inner = 3, 70
    X = torch.randn((n_outer, n_inner, d), generator=g)
    X *= 10.0 ** torch.randint(-7, 4, (n_outer, n_inner, 1), generator=g).float()
    X[0, 3] = 0.0                                           # all-zero row: scales 0
    X[1, 5, :32] = 0.0                                      # one zero block
    X[2, 7, :8] = torch.tensor([127, 0.5, -0.5, 1.5, -2.5, 2.49, -126.5, 3.5])   # ties
    X[2, 7, 8:32] = 0.0
    X = X.to(xdtype)
    rb = sfa.sfa_q8_0_row_bytes(d)
    # the outer stride of Y leaves a gap after each outer group, which must stay untouched
    Yb = torch.full((n_outer, n_inner * rb + 64), 0xAB, dtype=torch.uint8, device=dev)
    Y = Yb[:, : n_inner * rb].view(n_outer, n_inner, rb)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_quantize_kv_q8_0(X.to(dev), Y, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    codes, scales, pad = _split_rows(Y, d)
    q, s = oracle.quantize_q8_0(np32(X))
    assert np.array_equal(codes, q) and np.array_equal(scales, s)
    assert not pad.any()
    assert np.all(Yb[:, n_inner * rb:].cpu().numpy() == 0xAB)
    assert codes[2, 7, :8].tolist() == [127, 1, -1, 2, -3, 2, -127, 4]


def test_quantize_flags_binary16_overflow(dev):
    X = torch.ones((1, 2, 64), device=dev)
    X[0, 1, 40] = 1e7                                       # scale 78740 > 65504
    Y = torch.empty((1, 2, sfa.sfa_q8_0_row_bytes(64)), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_quantize_kv_q8_0(X, Y, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) & sfa.SFA_DEV_FP16_RANGE


# --------------------------------------------------------------------------------- attention
def _selection(q_pos, cr, top_k, rng):
    sel = np.full((len(q_pos), top_k), -1, np.int32)
    n_sel = np.zeros(len(q_pos), np.int32)
    for i, p in enumerate(q_pos):
        B = (int(p) + 1) // cr
        n = min(top_k, B)
        sel[i, :n] = np.sort(rng.choice(B, size=n, replace=False)) if n else []
        n_sel[i] = n
    return sel, n_sel


SHAPES = [(576, 512, True, 16, 1), (512, 512, False, 16, 2), (512, 512, True, 8, 1),
          (128, 128, False, 8, 2), (64, 64, True, 4, 1)]


@pytest.mark.parametrize("dkq,dv,v_is_k,h_q,h_kv", SHAPES)
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_gather_attend_q8_matches_oracle(dev, dkq, dv, v_is_k, h_q, h_kv, mode):
    cr = 4
    if mode == "decode":   # 2048 kept cells split over a cluster, a shorter list, a tail only
        n_seq, n_tok, top_k = 3, 2600, 512
        q_seq = np.array([0, 1, 2, 1], np.int32)
        q_pos = np.array([2599, 2100, 900, 2], np.int32)
    else:
        n_seq, n_tok, top_k = 1, 700, 40
        q_seq = np.zeros(100, np.int32)
        q_pos = np.arange(600, 700, dtype=np.int32)
    g = torch.Generator().manual_seed(dkq + h_q + len(q_seq))
    rng = np.random.default_rng(dkq)
    K = _randn((n_seq, n_tok, h_kv, dkq), g)
    V = None if v_is_k else _randn((n_seq, n_tok, h_kv, dv), g)
    Q = _randn((len(q_seq), h_q, dkq), g)
    Kq = _quantize(K, dev)
    Vq = None if V is None else _quantize(V, dev)
    sel, n_sel = _selection(q_pos, cr, top_k, rng)
    scale = 1.0 / math.sqrt(dkq)
    d = lambda a: torch.from_numpy(a).to(dev)
    O = torch.full((len(q_seq), h_q, dv), float("nan"), device=dev)
    lse = torch.full((len(q_seq), h_q), float("nan"), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_gather_attend(Q.to(dev), Kq, Vq, d(q_seq), d(q_pos), d(sel), d(n_sel), top_k, cr,
                          scale, O, lse=lse, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    Kh = _oracle_values(K)
    Vh = None if V is None else _oracle_values(V)
    Qn, On, Ln = np32(Q), np32(O), np32(lse)
    for i in range(len(q_seq)):
        s, p = int(q_seq[i]), int(q_pos[i])
        msk = oracle.mask(p, cr, sel[i], int(n_sel[i]))
        ref, rlse = oracle.attend(Qn[i], Kh[s], None if Vh is None else Vh[s], msk, scale, h_kv,
                                  dv=dv)
        assert row_rel_err(On[i], ref).max() < TOL_BF16, i
        assert np.abs(Ln[i] - rlse).max() < 2e-3, i


def test_dense_and_paged_attend_q8(dev):
    """Dense attention over q8_0 rows matches the oracle; the paged calls on the same rows in
    shuffled 16-cell pages give the per-sequence results bit for bit."""
    dkq, dv, h_q, h_kv = 576, 512, 16, 1
    n_seq, n_tok = 2, 1100
    q_seq = np.array([0, 1, 1, 0], np.int32)
    q_pos = np.array([1099, 0, 517, 64], np.int32)
    g = torch.Generator().manual_seed(77)
    K = _randn((n_seq, n_tok, h_kv, dkq), g)
    Q = _randn((len(q_seq), h_q, dkq), g)
    Kq = _quantize(K, dev)
    scale = 1.0 / math.sqrt(dkq)
    d = lambda a: torch.from_numpy(a).to(dev)
    O1 = torch.empty((len(q_seq), h_q, dv), device=dev)
    sfa.sfa_dense_attend(Q.to(dev), Kq, None, d(q_seq), d(q_pos), n_tok, scale, O1)
    cell_of, n_cells = sfa.make_cell_map(n_seq, n_tok, page=16, spare_pages=3, seed=4, device=dev)
    Kp = sfa.to_cells(Kq, cell_of, n_cells)
    O2 = torch.empty_like(O1)
    sfa.sfa_dense_attend_paged(Q.to(dev), Kp, None, cell_of, d(q_seq), d(q_pos), n_tok, scale, O2)
    # gathered, per sequence and paged
    rng = np.random.default_rng(5)
    sel, n_sel = _selection(q_pos, 4, 64, rng)
    O3, O4 = torch.empty_like(O1), torch.empty_like(O1)
    sfa.sfa_gather_attend(Q.to(dev), Kq, None, d(q_seq), d(q_pos), d(sel), d(n_sel), 64, 4,
                          scale, O3)
    sfa.sfa_gather_attend_paged(Q.to(dev), Kp, None, cell_of, d(q_seq), d(q_pos), d(sel),
                                d(n_sel), 64, 4, scale, O4)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(O3, O4)
    Kh, Qn, On = _oracle_values(K), np32(Q), np32(O1)
    for i in range(len(q_seq)):
        s, p = int(q_seq[i]), int(q_pos[i])
        ref, _ = oracle.attend(Qn[i], Kh[s], None, oracle.mask(p, 4, dense=True), scale, h_kv,
                               dv=dv)
        assert row_rel_err(On[i], ref).max() < TOL_BF16, i


def test_q8_flags_query_beyond_binary16(dev):
    dkq, dv, h_q = 64, 64, 4
    g = torch.Generator().manual_seed(3)
    K = _randn((1, 64, 1, dkq), g)
    Q = _randn((1, h_q, dkq), g)
    Q[0, 1, 5] = 1e5
    Kq = _quantize(K, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    O = torch.empty((1, h_q, dv), device=dev)
    d = lambda a: torch.from_numpy(np.asarray(a, np.int32)).to(dev)
    sfa.sfa_dense_attend(Q.to(dev), Kq, None, d([0]), d([63]), 64, 0.125, O, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) & sfa.SFA_DEV_FP16_RANGE


# -------------------------------------------------------------------------------- whole step
@pytest.mark.parametrize("name,shrink", [("decode_1x4096", {}),
                                         ("decode_32x131072", {"n_seq": 4, "depth": 30000}),
                                         ("decode_4x1048576", {"n_seq": 2, "depth": 50000})])
def test_step_on_q8_cache(dev, name, shrink):
    """A whole step on q8_0 caches: the kept blocks are those of the bf16 step (the index keys
    are unchanged) and the outputs match the oracle's attention over the dequantized cache."""
    w = sfa.WORKLOADS[name]
    if shrink:
        w = w.with_(**shrink)
    case = sfa.make_case(w, device=dev)
    n_blk_max = w.n_tok // w.compress_ratio
    Kq = _quantize(case["K"], dev)
    Vq = None if case["V"] is None else _quantize(case["V"], dev)
    steps = []
    for K, V in ((case["K"], case["V"]), (Kq, Vq)):
        st = sfa.SfaStep(n_seq=w.n_seq, n_tok_cap=w.n_tok, n_q=w.n_q, h_q=w.h_q, h_kv=w.h_kv,
                         dkq=w.dkq, dv=w.dv, h_idx=w.h_idx, d_idx=w.d_idx,
                         compress_ratio=w.compress_ratio, indexer_top_k=w.indexer_top_k,
                         n_blk_max=n_blk_max, q_group=w.n_q_per_seq, device=dev)
        st.run(case["X"], K, V, case["Q"], case["q_idx"], case["w"], case["q_seq"],
               case["q_pos"], w.scale, new_blocks=(0, n_blk_max))
        torch.cuda.synchronize()
        assert sfa.sfa_read_device_status(st.status) == 0
        steps.append(st)
    a, b = steps
    assert torch.equal(a.n_sel, b.n_sel) and torch.equal(a.blk_idx, b.blk_idx)
    Qn, On, Ln = np32(case["Q"]), np32(b.O), np32(b.lse)
    sel, n_sel = np32(b.blk_idx), np32(b.n_sel)
    for i in range(w.n_q):
        s, p = int(case["q_seq"][i]), int(case["q_pos"][i])
        Kh = _oracle_values(case["K"][s, : p + 1])
        Vh = None if case["V"] is None else _oracle_values(case["V"][s, : p + 1])
        msk = oracle.mask(p, w.compress_ratio, sel[i], int(n_sel[i]))
        ref, rlse = oracle.attend(Qn[i], Kh, Vh, msk, w.scale, w.h_kv, dv=w.dv)
        assert row_rel_err(On[i], ref).max() < TOL_BF16, i
        assert np.abs(Ln[i] - rlse).max() < 2e-3, i
