"""Parity of the tcgen05 attention kernel (selected with SFA_ATTEND_KERNEL=tcgen05) against the
oracle: the stage-level gathered and dense cases of the 512-wide heads, and the full-size
decode and prefill workloads on every query.  The default path (the warp-level kernel) is
covered by test_gpu_stages / test_gpu_pipeline."""
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

TC_SHAPES = [(576, 512, True, 16, 1), (512, 512, False, 16, 2), (512, 512, True, 8, 1)]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.fixture
def tcgen05(monkeypatch):
    monkeypatch.setenv("SFA_ATTEND_KERNEL", "tcgen05")


@pytest.mark.parametrize("dkq,dv,v_is_k,h_q,h_kv", TC_SHAPES)
@pytest.mark.parametrize("mode", ["decode", "prefill"])
@pytest.mark.parametrize("cr", [4, 3])
def test_tcgen05_gather_attend_matches_oracle(dev, tcgen05, dkq, dv, v_is_k, h_q, h_kv, mode, cr):
    top_k = 40
    if mode == "decode":
        n_seq, n_tok = 3, 900
        q_seq = np.array([0, 1, 2], np.int32)
        q_pos = np.array([899, 161, 2], np.int32)
    else:
        n_seq, n_tok = 1, 700
        q_seq = np.zeros(150, np.int32)
        q_pos = np.arange(550, 700, dtype=np.int32)
    Q, K, V = _attend_case(dev, dkq, dv, v_is_k, h_q, h_kv, n_seq, n_tok, q_seq, q_pos,
                           torch.bfloat16, dkq + h_q + cr)
    sel, n_sel = _random_selection(q_pos, cr, top_k, 5)
    scale = 1.0 / math.sqrt(dkq)
    O = torch.empty((len(q_seq), h_q, dv), device=dev)
    lse = torch.empty((len(q_seq), h_q), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_gather_attend(Q, K, V, torch.from_numpy(q_seq).to(dev), torch.from_numpy(q_pos).to(dev),
                          torch.from_numpy(sel).to(dev), torch.from_numpy(n_sel).to(dev), top_k,
                          cr, scale, O, lse=lse, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    Kn, Vn, Qn, On, Ln = np32(K), np32(V), np32(Q), np32(O), np32(lse)
    for i in range(len(q_seq)):
        s, p = q_seq[i], int(q_pos[i])
        msk = oracle.mask(p, cr, sel[i], int(n_sel[i]))
        ref, rlse = oracle.attend(Qn[i], Kn[s], None if Vn is None else Vn[s], msk, scale, h_kv,
                                  dv=dv)
        assert row_rel_err(On[i], ref).max() < TOL_BF16, i
        assert np.abs(Ln[i] - rlse).max() < 2e-3


@pytest.mark.parametrize("dkq,dv,v_is_k,h_q,h_kv", TC_SHAPES[:2])
def test_tcgen05_dense_attend_matches_oracle(dev, tcgen05, dkq, dv, v_is_k, h_q, h_kv):
    n_seq, n_tok = 2, 1100
    q_seq = np.array([0, 1, 1, 0], np.int32)
    q_pos = np.array([1099, 0, 517, 64], np.int32)
    Q, K, V = _attend_case(dev, dkq, dv, v_is_k, h_q, h_kv, n_seq, n_tok, q_seq, q_pos,
                           torch.bfloat16, 11)
    scale = 1.0 / math.sqrt(dkq)
    O = torch.empty((len(q_seq), h_q, dv), device=dev)
    sfa.sfa_dense_attend(Q, K, V, torch.from_numpy(q_seq).to(dev), torch.from_numpy(q_pos).to(dev),
                         n_tok, scale, O)
    torch.cuda.synchronize()
    Kn, Vn, Qn, On = np32(K), np32(V), np32(Q), np32(O)
    for i in range(len(q_seq)):
        s, p = q_seq[i], int(q_pos[i])
        ref, _ = oracle.attend(Qn[i], Kn[s], None if Vn is None else Vn[s],
                               oracle.mask(p, 4, dense=True), scale, h_kv, dv=dv)
        assert row_rel_err(On[i], ref).max() < TOL_BF16


def test_tcgen05_matches_default_kernel(dev, monkeypatch):
    """Both kernels attend the same kept cells: outputs agree within the bf16 tolerance."""
    w = sfa.WORKLOADS["decode_1x4096"].with_(n_seq=5, seed=91)
    case, step = _run(w, dev)
    O_default = np32(step.O)
    monkeypatch.setenv("SFA_ATTEND_KERNEL", "tcgen05")
    step.attend(case["Q"], case["K"], case["V"], case["q_seq"], case["q_pos"], w.scale)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(step.status) == 0
    assert row_rel_err(np32(step.O), O_default).max() < TOL_BF16


@pytest.mark.parametrize("name", ["decode_32x131072", "pp2048_131072", "decode_4x1048576"])
def test_tcgen05_full_size_all(dev, tcgen05, name):
    w = sfa.WORKLOADS[name]
    case, step = _run(w, dev)
    _check_queries(w, case, step)
