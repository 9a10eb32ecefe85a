"""Parity of the warp-specialised bulk-copy attention kernel (selected with
SFA_ATTEND_KERNEL=ws) against the oracle.  The kernel is opt-in: on the measured workloads it
is slower than the default warp-level kernel (see the design notes), and these tests keep it
correct: every shape and mode of the stage-level gathered and dense cases, the cluster and
combine merges, bad-list flags, the paged layout, and the full-size decode and prefill
workloads on every query."""
import pytest
import torch

import test_gpu_paged as P
import test_gpu_stages as S
from test_gpu_pipeline import _check_queries, _run

pytestmark = pytest.mark.gpu

sfa = pytest.importorskip("indexer_selected_sparse_block_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.fixture
def ws(monkeypatch):
    monkeypatch.setenv("SFA_ATTEND_KERNEL", "ws")


@pytest.mark.parametrize("dkq,dv,v_is_k,h_q,h_kv", S.ATTN_SHAPES)
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_ws_gather_attend_matches_oracle(dev, ws, dkq, dv, v_is_k, h_q, h_kv, mode):
    S.test_gather_attend_matches_oracle(dev, dkq, dv, v_is_k, h_q, h_kv, mode, torch.bfloat16)


@pytest.mark.parametrize("n_q", [32, 76, 128])
def test_ws_cluster_and_combine_merges(dev, ws, n_q):
    S.test_gather_attend_cluster_merge(dev, n_q)


@pytest.mark.parametrize("dkq,dv,v_is_k,h_q,h_kv", S.ATTN_SHAPES[:2])
def test_ws_dense_attend_matches_oracle(dev, ws, dkq, dv, v_is_k, h_q, h_kv):
    S.test_dense_attend_matches_oracle(dev, dkq, dv, v_is_k, h_q, h_kv, torch.bfloat16)


def test_ws_flags_bad_block_lists(dev, ws):
    S.test_attend_flags_bad_block_lists(dev)


@pytest.mark.parametrize("layout", ["pages", "cells"])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_ws_gather_attend_paged(dev, ws, layout, mode):
    dkq, dv, v_is_k, h_q, h_kv = P.SHAPES[0]
    P.test_gather_attend_paged(dev, layout, dkq, dv, v_is_k, h_q, h_kv, mode, torch.bfloat16)


@pytest.mark.parametrize("name", ["decode_32x131072", "pp2048_131072", "decode_4x1048576"])
def test_ws_full_size_all(dev, ws, name):
    w = sfa.WORKLOADS[name]
    case, step = _run(w, dev)
    _check_queries(w, case, step)


@pytest.mark.parametrize("name", ["decode_1x4096", "decode_4x1048576"])
def test_gather_kv_bandwidth_moves_the_attended_rows(dev, name):
    """The gather-only measurement kernel copies exactly the attended rows: the sum of the
    first 32-bit word of every attended K row (V rows are copied beside them) equals the same
    sum taken on the host over the kept blocks and the tail."""
    w = sfa.WORKLOADS[name].with_(n_seq=3) if name == "decode_1x4096" else sfa.WORKLOADS[name]
    case, step = _run(w, dev)
    chk = torch.zeros(1, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_gather_kv_bandwidth(case["K"], case["V"], case["q_seq"], case["q_pos"], step.blk_idx,
                                step.n_sel, step.top_k, w.compress_ratio, w.dkq, w.dv, chk,
                                dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    words = case["K"].view(torch.int32)[..., 0]            # [n_seq][n_tok][h_kv]: first word
    total = 0
    sel, ns = step.blk_idx.cpu().numpy(), step.n_sel.cpu().numpy()
    for i in range(w.n_q):
        s, p = int(case["q_seq"][i]), int(case["q_pos"][i])
        cr = w.compress_ratio
        toks = [b * cr + r for b in sel[i, : ns[i]] for r in range(cr)]
        toks += list(range(((p + 1) // cr) * cr, p + 1))
        rows = words[s].index_select(0, torch.tensor(toks, device=dev))
        total += int(rows.to(torch.int64).sum().item())
    assert (int(chk.item()) & 0xFFFFFFFF) == (total & 0xFFFFFFFF)
