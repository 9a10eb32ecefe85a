"""The dense window + sparse selection variant against the oracle (its attended set: the kept
blocks, the tail and the `window` most recent positions; llama.cpp PR #27970's review
discussion: dense attention over the continuous block of keys, sparse attention over the
selected keys, the two results combined).

Stage level: the whole set in one pass, and the kept part and the window part attended apart
and merged by sfa_combine_attention, for several compress ratios and windows, including no
window (equal to sfa_gather_attend bit for bit) and a window reaching position 0 (dense).
Full size: the decode_32x131072 step with a 128-position window, both ways, every query."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, np32, row_rel_err
from test_gpu_pipeline import _check_queries, _run
from test_gpu_stages import _attend_case, _random_selection

pytestmark = pytest.mark.gpu

sfa = pytest.importorskip("indexer_selected_sparse_block_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _setup(dev, cr, seed, dkq=576, dv=512, v_is_k=True, h_q=16, h_kv=1):
    top_k = 40
    n_seq, n_tok = 3, 900
    q_seq = np.array([0, 1, 2, 0, 1], np.int32)
    q_pos = np.array([899, 161, 2, 500, 30], np.int32)
    Q, K, V = _attend_case(dev, dkq, dv, v_is_k, h_q, h_kv, n_seq, n_tok, q_seq, q_pos,
                           torch.bfloat16, seed)
    sel, n_sel = _random_selection(q_pos, cr, top_k, seed)
    return dict(Q=Q, K=K, V=V, q_seq=q_seq, q_pos=q_pos, sel=sel, n_sel=n_sel, top_k=top_k,
                cr=cr, dv=dv, h_q=h_q, h_kv=h_kv, scale=1.0 / math.sqrt(dkq))


def _attend(dev, c, window, part):
    n_q = len(c["q_seq"])
    O = torch.full((n_q, c["h_q"], c["dv"]), float("nan"), device=dev)
    lse = torch.full((n_q, c["h_q"]), float("nan"), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_gather_attend_window(c["Q"], c["K"], c["V"], torch.from_numpy(c["q_seq"]).to(dev),
                                 torch.from_numpy(c["q_pos"]).to(dev),
                                 torch.from_numpy(c["sel"]).to(dev),
                                 torch.from_numpy(c["n_sel"]).to(dev), c["top_k"], c["cr"],
                                 window, c["scale"], O, lse=lse, part=part, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    return O, lse


def _check(c, window, O, lse):
    Kn, Qn = np32(c["K"]), np32(c["Q"])
    Vn = None if c["V"] is None else np32(c["V"])
    On, Ln = np32(O), np32(lse)
    for i in range(len(c["q_seq"])):
        s, p = int(c["q_seq"][i]), int(c["q_pos"][i])
        msk = oracle.mask(p, c["cr"], c["sel"][i], int(c["n_sel"][i]), window=window)
        ref, rlse = oracle.attend(Qn[i], Kn[s], None if Vn is None else Vn[s], msk, c["scale"],
                                  c["h_kv"], dv=c["dv"])
        assert row_rel_err(On[i], ref).max() < TOL_BF16, (i, window)
        assert np.abs(Ln[i] - rlse).max() < 2e-3, (i, window)


@pytest.mark.parametrize("cr", [4, 3, 8])
@pytest.mark.parametrize("window", [1, 7, 37, 300, 5000])
def test_window_one_pass_and_split_match_oracle(dev, cr, window):
    c = _setup(dev, cr, 100 + cr + window)
    O, lse = _attend(dev, c, window, sfa.SFA_PART_ALL)
    _check(c, window, O, lse)
    Oa, la = _attend(dev, c, window, sfa.SFA_PART_SELECTED)
    Ob, lb = _attend(dev, c, window, sfa.SFA_PART_WINDOW)
    sfa.sfa_combine_attention(Oa, la, Ob, lb, Oa, la)   # in place
    torch.cuda.synchronize()
    _check(c, window, Oa, la)


def test_window_separate_v(dev):
    c = _setup(dev, 8, 7, dkq=512, dv=512, v_is_k=False, h_q=16, h_kv=2)
    for window in (5, 64):
        O, lse = _attend(dev, c, window, sfa.SFA_PART_ALL)
        _check(c, window, O, lse)


def test_no_window_is_the_gathered_attention(dev):
    c = _setup(dev, 4, 3)
    O, lse = _attend(dev, c, 0, sfa.SFA_PART_ALL)
    O2 = torch.empty_like(O)
    l2 = torch.empty_like(lse)
    sfa.sfa_gather_attend(c["Q"], c["K"], c["V"], torch.from_numpy(c["q_seq"]).to(dev),
                          torch.from_numpy(c["q_pos"]).to(dev), torch.from_numpy(c["sel"]).to(dev),
                          torch.from_numpy(c["n_sel"]).to(dev), c["top_k"], c["cr"], c["scale"],
                          O2, lse=l2)
    torch.cuda.synchronize()
    assert torch.equal(O, O2) and torch.equal(lse, l2)


def test_empty_parts(dev):
    """A window that reaches position 0 leaves every query an empty kept part: O = 0 and
    lse = -inf (the combine with such a part is checked above, window 5000)."""
    c = _setup(dev, 4, 9)
    O, lse = _attend(dev, c, 5000, sfa.SFA_PART_SELECTED)
    assert bool(torch.all(O == 0)) and bool(torch.all(torch.isneginf(lse)))


@pytest.mark.parametrize("mode", ["single", "split"])
def test_window_step_full_size(dev, mode):
    w = sfa.WORKLOADS["decode_32x131072"]
    case, step = _run(w, dev, window=128, window_mode=mode)
    _check_queries(w, case, step, window=128)
