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
