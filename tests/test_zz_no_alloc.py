"""sfa_gather_attend_noalloc, called through the C ABI, against sfa_gather_attend.

The no-allocation entry point exists for callers that cannot allocate device memory when
they call (an application that owns all device memory through its own allocator, or a decode
loop that must not pay cudaFree's device-wide synchronisation).  It must give the same result
as the workspace entry point, call after call, although every call reuses one fixed scratch
array inside the library.  This file is collected last on purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, np32, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from indexer_selected_sparse_block_gb300 import _binding
    return _binding.lib()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _case(seed, dev, n_seq=3, n_tok=2100, h_q=16, h_kv=1, dkq=576, dv=512, cr=4, top_k=256):
    g = torch.Generator().manual_seed(seed)
    K = torch.randn((n_seq, n_tok, h_kv, dkq), generator=g).to(torch.bfloat16).to(dev)
    Q = torch.randn((n_seq, h_q, dkq), generator=g).to(torch.bfloat16).to(dev)
    q_seq = torch.arange(n_seq, dtype=torch.int32)
    q_pos = torch.tensor([n_tok - 1 - 7 * i for i in range(n_seq)], dtype=torch.int32)
    sel = np.full((n_seq, top_k), -1, np.int32)
    n_sel = np.zeros(n_seq, np.int32)
    rng = np.random.default_rng(seed)
    for i, p in enumerate(q_pos.tolist()):
        B = (p + 1) // cr
        n = min(top_k, B)
        sel[i, :n] = np.sort(rng.choice(B, size=n, replace=False))
        n_sel[i] = n
    return dict(Q=Q, K=K, q_seq=q_seq.to(dev), q_pos=q_pos.to(dev),
                sel=torch.from_numpy(sel).to(dev), n_sel=torch.from_numpy(n_sel).to(dev),
                dims=(n_seq, n_tok, n_seq, h_q, h_kv, dkq, dv), cr=cr, top_k=top_k,
                scale=1.0 / math.sqrt(dkq))


def _call_noalloc(L, c, O, lse, status):
    n_seq, n_tok, n_q, h_q, h_kv, dkq, dv = c["dims"]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.sfa_gather_attend_noalloc(_ptr(c["Q"]), _ptr(c["K"]), None, 0, n_seq, n_tok, n_q,
                                       h_q, h_kv, dkq, dv, c["scale"], _ptr(c["q_seq"]),
                                       _ptr(c["q_pos"]), _ptr(c["sel"]), _ptr(c["n_sel"]),
                                       c["top_k"], c["cr"], _ptr(O), _ptr(lse), _ptr(status),
                                       stream)


def _call_workspace(L, c, O, lse, status):
    n_seq, n_tok, n_q, h_q, h_kv, dkq, dv = c["dims"]
    n_kv = c["top_k"] * c["cr"] + c["cr"] - 1
    need = L.sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv)
    assert need > 0, "this case must exercise the split-KV scratch"
    ws = torch.empty(need, dtype=torch.uint8, device=O.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.sfa_gather_attend(_ptr(c["Q"]), _ptr(c["K"]), None, 0, n_seq, n_tok, n_q, h_q,
                               h_kv, dkq, dv, c["scale"], _ptr(c["q_seq"]), _ptr(c["q_pos"]),
                               _ptr(c["sel"]), _ptr(c["n_sel"]), c["top_k"], c["cr"], _ptr(O),
                               _ptr(lse), _ptr(ws), need, _ptr(status), stream)


def _plan(L, c):
    """(splits per list, kernels per call) of the attention call of case c."""
    n_seq, n_tok, n_q, h_q, h_kv, dkq, dv = c["dims"]
    ns, nk = ctypes.c_int(0), ctypes.c_int(0)
    n_kv = c["top_k"] * c["cr"] + c["cr"] - 1
    assert L.sfa_attend_plan(0, n_q, h_kv, dkq, 0, ctypes.c_int64(n_kv), c["cr"], 0,
                             ctypes.byref(ns), ctypes.byref(nk)) == 0
    return ns.value, nk.value


def _oracle_outputs(c):
    """The oracle's attention of every query of case c over its kept blocks and tail."""
    n_seq, n_tok, n_q, h_q, h_kv, dkq, dv = c["dims"]
    K, Q = np32(c["K"]), np32(c["Q"])
    sel, n_sel, q_pos = np32(c["sel"]), np32(c["n_sel"]), np32(c["q_pos"])
    out = []
    for i in range(n_q):
        msk = oracle.mask(int(q_pos[i]), c["cr"], sel[i], int(n_sel[i]))
        out.append(oracle.attend(Q[i], K[i], None, msk, c["scale"], h_kv, dv=dv))
    return np.stack([o for o, _ in out]), np.stack([l for _, l in out])


def test_noalloc_matches_workspace_entry_point_twice(L):
    dev = torch.device("cuda:0")
    for seed in (11, 12):   # two calls in a row, different data, one shared scratch array
        c = _case(seed, dev)
        # the plan splits each list over several CTAs and merges them through the scratch
        # (a second kernel), so the shared array is really written and read
        n_split, kernels = _plan(L, c)
        assert n_split > 1 and kernels == 2, (n_split, kernels)
        n_q, h_q, dv = c["dims"][2], c["dims"][3], c["dims"][6]
        O1 = torch.empty((n_q, h_q, dv), device=dev)
        O2 = torch.full((n_q, h_q, dv), float("nan"), device=dev)
        l1 = torch.empty((n_q, h_q), device=dev)
        l2 = torch.full((n_q, h_q), float("nan"), device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        assert _call_workspace(L, c, O1, l1, st) == 0
        assert _call_noalloc(L, c, O2, l2, st) == 0
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert row_rel_err(np32(O2), np32(O1)).max() < TOL_BF16
        assert np.abs(np32(l2) - np32(l1)).max() < 2e-3
        ref_o, ref_l = _oracle_outputs(c)
        assert row_rel_err(np32(O2), ref_o).max() < TOL_BF16
        assert np.abs(np32(l2) - ref_l).max() < 2e-3


def test_noalloc_scratch_bound(L):
    """The split-KV scratch a shape needs either fits the fixed array, or the call is refused
    with SFA_ERR_WORKSPACE before anything is enqueued.  With one-wave split sizing the need
    is bounded by about (SM count) x 16 heads x (dv + 2) x 4 bytes, so on this GPU every
    supported shape fits; any shape that did not would take the refusal path."""
    dev = torch.device("cuda:0")
    limit = 16 << 20
    h_q, h_kv, dkq, dv, cr, top_k = 16, 1, 576, 512, 4, 512
    n_kv = top_k * cr + cr - 1
    over = [n for n in range(1, 2048)
            if L.sfa_attend_workspace_bytes(n, h_q, h_kv, dv, n_kv) > limit]
    if not over:
        assert all(L.sfa_attend_workspace_bytes(n, 16, hk, 512, 1 << 20) <= limit
                   for n in range(1, 512) for hk in (1, 2, 4))
        return
    n_q = over[0]
    n_tok = 4096
    K = torch.zeros((1, n_tok, h_kv, dkq), dtype=torch.bfloat16, device=dev)
    Q = torch.zeros((n_q, h_q, dkq), dtype=torch.bfloat16, device=dev)
    q_seq = torch.zeros(n_q, dtype=torch.int32, device=dev)
    q_pos = torch.full((n_q,), n_tok - 1, dtype=torch.int32, device=dev)
    sel = torch.arange(top_k, dtype=torch.int32, device=dev).repeat(n_q, 1).contiguous()
    n_sel = torch.full((n_q,), top_k, dtype=torch.int32, device=dev)
    O = torch.full((n_q, h_q, dv), 5.0, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.sfa_gather_attend_noalloc(_ptr(Q), _ptr(K), None, 0, 1, n_tok, n_q, h_q, h_kv, dkq,
                                     dv, 1.0 / 24.0, _ptr(q_seq), _ptr(q_pos), _ptr(sel),
                                     _ptr(n_sel), top_k, cr, _ptr(O), None, None, stream)
    torch.cuda.synchronize()
    assert rc == 4                          # SFA_ERR_WORKSPACE
    assert bool(torch.all(O == 5.0))        # nothing ran
