"""Stage-by-stage parity of the CUDA path (through the C ABI) against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_BF16, TOL_F32, check_selection, np32, row_rel_err

pytestmark = pytest.mark.gpu

sfa = pytest.importorskip("indexer_selected_sparse_block_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _randn_bf16(shape, gen, dev, scale=1.0):
    return (torch.randn(shape, generator=gen, device="cpu") * scale).to(torch.bfloat16).to(dev)


# -------------------------------------------------------------------------------- pooling
@pytest.mark.parametrize("cr", [1, 3, 4, 8])
@pytest.mark.parametrize("d_idx", [32, 64, 128])
@pytest.mark.parametrize("xdtype", [torch.bfloat16, torch.float32])
def test_pool_matches_oracle(dev, cr, d_idx, xdtype):
    g = torch.Generator().manual_seed(cr * 1000 + d_idx)
    n_seq, n_tok = 3, 1000 + cr
    X = _randn_bf16((n_seq, n_tok, d_idx), g, dev).to(xdtype)
    blk_cap = n_tok // cr + 5
    Kbar = torch.full(sfa.kbar_shape(n_seq, blk_cap, d_idx), 7.0, dtype=torch.bfloat16, device=dev)
    b0, b1 = 3, n_tok // cr
    sfa.sfa_pool_index_keys(X, cr, b0, b1, Kbar)
    torch.cuda.synchronize()
    kb = np32(Kbar).astype(np.float64)
    got = kb[..., :d_idx] + kb[..., d_idx:]
    Xn = np32(X)
    for s in range(n_seq):
        ref = oracle.pool(Xn[s], b1, cr)
        mag = np.abs(Xn[s, : b1 * cr].astype(np.float64)).reshape(b1, cr, d_idx).mean(1)
        err = np.abs(got[s, b0:b1] - ref[b0:b1])
        assert np.all(err <= 2.0 ** -16 * mag[b0:b1] + 1e-30), err.max()
    assert np.all(kb[:, :b0] == 7.0) and np.all(kb[:, b1:] == 7.0)  # other rows untouched


# ---------------------------------------------------------------------------------- scores
def _oracle_scores(Xn, qi, w, q_seq, q_pos, cr):
    out = []
    for i in range(len(q_seq)):
        B = (int(q_pos[i]) + 1) // cr
        kb = oracle.pool(Xn[q_seq[i]], B, cr)
        s = oracle.index_scores(qi[i], w[i], kb)
        mag = np.abs(kb) @ np.abs(qi[i].astype(np.float64)).T @ np.abs(w[i].astype(np.float64))
        out.append((s, mag))
    return out


@pytest.mark.parametrize("d_idx,h_idx", [(64, 4), (128, 8), (64, 16), (128, 4)])
@pytest.mark.parametrize("mode", ["decode", "prefill", "prefill_wide"])
def test_scores_match_oracle(dev, d_idx, h_idx, mode):
    """decode: one query per tile; prefill: 70 queries in tiles of 2 (narrow B tiles);
    prefill_wide: 96 queries in tiles of 16 or 32 (B tiles of 128 or 256 columns, the
    prefill workloads' shape), causal over a ragged last block tile."""
    g = torch.Generator().manual_seed(d_idx + h_idx)
    cr = 4
    if mode == "decode":
        n_seq, n_tok, n_q, q_group = 5, 1500, 5, 1
        q_seq = torch.arange(5, dtype=torch.int32)
        q_pos = torch.tensor([1499, 700, 3, 1023, 511], dtype=torch.int32)
    elif mode == "prefill_wide":
        n_seq, n_tok, n_q, q_group = 1, 2100, 96, 96
        q_seq = torch.zeros(n_q, dtype=torch.int32)
        q_pos = torch.arange(2100 - n_q, 2100, dtype=torch.int32)
    else:
        n_seq, n_tok, n_q, q_group = 1, 2100, 70, 70
        q_seq = torch.zeros(n_q, dtype=torch.int32)
        q_pos = torch.arange(2100 - n_q, 2100, dtype=torch.int32)
    X = _randn_bf16((n_seq, n_tok, d_idx), g, dev)
    qi = _randn_bf16((n_q, h_idx, d_idx), g, dev)
    w = torch.rand((n_q, h_idx), generator=g).to(dev)
    blk_cap = n_tok // cr
    Kbar = torch.zeros(sfa.kbar_shape(n_seq, blk_cap, d_idx), dtype=torch.bfloat16, device=dev)
    sfa.sfa_pool_index_keys(X, cr, 0, blk_cap, Kbar)
    n_blk_max = int((q_pos.max() + 1) // cr)
    scores = torch.full((n_q, n_blk_max + 3), float("nan"), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores(qi, w, q_seq.to(dev), q_pos.to(dev), Kbar, cr, n_blk_max, scores,
                         q_group=q_group, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    got = np32(scores)
    ref = _oracle_scores(np32(X), np32(qi), np32(w), q_seq.numpy(), q_pos.numpy(), cr)
    for i, (s, mag) in enumerate(ref):
        B = s.shape[0]
        err = np.abs(got[i, :B] - s)
        assert np.all(err <= 1e-5 * mag + 1e-30), (i, err.max(), mag.max())
        assert np.all(np.isnan(got[i, B:])), i   # entries at b >= B_i untouched


def test_scores_flag_query_group_violation(dev):
    """A query that breaks the q_group promise is skipped and flagged, never misread."""
    g = torch.Generator().manual_seed(5)
    X = _randn_bf16((2, 600, 64), g, dev)
    Kbar = torch.zeros(sfa.kbar_shape(2, 150, 64), dtype=torch.bfloat16, device=dev)
    sfa.sfa_pool_index_keys(X, 4, 0, 150, Kbar)
    qi = _randn_bf16((4, 4, 64), g, dev)
    w = torch.rand((4, 4), generator=g).to(dev)
    q_seq = torch.tensor([0, 0, 0, 1], dtype=torch.int32, device=dev)
    q_pos = torch.full((4,), 599, dtype=torch.int32, device=dev)
    scores = torch.full((4, 150), float("nan"), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores(qi, w, q_seq, q_pos, Kbar, 4, 150, scores, q_group=4, dev_status=status)
    st = sfa.sfa_read_device_status(status)
    assert st & sfa.SFA_DEV_BAD_QUERY
    got = np32(scores)
    assert np.all(np.isnan(got[3])) and not np.any(np.isnan(got[:3]))


# ------------------------------------------------------------------------------------ top-k
@pytest.mark.parametrize("top_k", [1, 7, 256, 512, 2048])
@pytest.mark.parametrize("pattern", ["coarse", "continuous", "dup_at_cut", "odd_stride"])
def test_topk_bit_exact(dev, top_k, pattern):
    """Kept sets equal the oracle's full sort exactly, for rows that fit the budget, rows of
    one chunk and rows cut into chunks; coarse values (many ties: the fallback radix select),
    continuous values (the two-digit path), continuous values with a run of exact ties
    across the cut (ranked by index), and continuous values in rows whose starts are not
    16-byte aligned (a row pitch of n_blk_max + 1 scores: the staging's single-word head)."""
    g = torch.Generator().manual_seed(top_k * 3 + len(pattern))
    cr = 4
    Bs = [0, 1, top_k - 1, top_k, top_k + 1, 3000, 8192, 8193, 20000, 70000]
    Bs = [b for b in Bs if b >= 0]
    n_q = len(Bs)
    q_pos = torch.tensor([b * cr + (i % (cr - 1)) for i, b in enumerate(Bs)], dtype=torch.int32)
    n_blk_max = max(Bs)
    raw = torch.randn((n_q, n_blk_max), generator=g)
    if pattern == "coarse":
        vals = torch.round(raw * 4) / 4          # many exact ties
        vals[vals == 0] = -0.0                   # signed zeros must tie with +0.0
        vals[1::2, ::3] = 0.0
    elif pattern in ("continuous", "odd_stride"):
        vals = torch.relu(raw) * 3 + torch.rand((n_q, n_blk_max), generator=g)
    else:
        vals = torch.relu(raw) * 3 + torch.rand((n_q, n_blk_max), generator=g)
        for i, b in enumerate(Bs):
            if b > top_k:
                row = vals[i, :b]
                cut = torch.sort(row, descending=True).values[top_k - 1].item()
                idx = torch.randperm(b, generator=g)[:40]
                row[idx] = cut                   # 40 exact copies of the cut value
    if pattern == "odd_stride":
        wide = torch.full((n_q, n_blk_max + 1), float("nan"), device=dev)
        wide[:, :n_blk_max] = vals.to(dev)
        scores = wide[:, :n_blk_max]
    else:
        scores = vals.to(dev)
    blk = torch.full((n_q, top_k), -9, dtype=torch.int32, device=dev)
    n_sel = torch.full((n_q,), -9, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_topk_blocks(scores, q_pos.to(dev), cr, top_k, n_blk_max, blk, n_sel,
                        dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    got, got_n = np32(blk), np32(n_sel)
    sc = vals.double().numpy()
    for i in range(n_q):
        B = (int(q_pos[i]) + 1) // cr
        ref, n = oracle.select(sc[i, :B], top_k)
        assert got_n[i] == n, (i, got_n[i], n)
        assert np.array_equal(got[i], ref), (i, B)


# ----------------------------------------------------------------------------------- attend
def _attend_case(dev, dkq, dv, v_is_k, h_q, h_kv, n_seq, n_tok, q_seq, q_pos, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    K = _randn_bf16((n_seq, n_tok, h_kv, dkq), g, dev).to(dtype)
    V = None if v_is_k else _randn_bf16((n_seq, n_tok, h_kv, dv), g, dev).to(dtype)
    Q = _randn_bf16((len(q_seq), h_q, dkq), g, dev).to(dtype)
    return Q, K, V


def _random_selection(q_pos, cr, top_k, seed):
    rng = np.random.default_rng(seed)
    sel = np.full((len(q_pos), top_k), -1, np.int32)
    n_sel = np.zeros(len(q_pos), np.int32)
    for i, p in enumerate(q_pos):
        B = (int(p) + 1) // cr
        n = min(top_k, B)
        pick = np.sort(rng.choice(B, size=n, replace=False)) if n else np.zeros(0, np.int64)
        sel[i, :n] = pick
        n_sel[i] = n
    return sel, n_sel


ATTN_SHAPES = [(576, 512, True, 16, 1), (512, 512, False, 16, 2), (128, 128, False, 8, 2),
               (64, 64, True, 4, 1)]


@pytest.mark.parametrize("dkq,dv,v_is_k,h_q,h_kv", ATTN_SHAPES)
@pytest.mark.parametrize("mode", ["decode", "prefill"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_gather_attend_matches_oracle(dev, dkq, dv, v_is_k, h_q, h_kv, mode, dtype):
    cr, top_k = 4, 40
    if mode == "decode":
        n_seq, n_tok = 3, 900
        q_seq = np.array([0, 1, 2], np.int32)
        q_pos = np.array([899, 161, 2], np.int32)    # long list, just over budget, tail only
    else:
        n_seq, n_tok = 1, 700
        q_seq = np.zeros(150, np.int32)
        q_pos = np.arange(550, 700, dtype=np.int32)
    Q, K, V = _attend_case(dev, dkq, dv, v_is_k, h_q, h_kv, n_seq, n_tok, q_seq, q_pos, dtype,
                           dkq + h_q)
    sel, n_sel = _random_selection(q_pos, cr, top_k, 3)
    scale = 1.0 / math.sqrt(dkq)
    O = torch.empty((len(q_seq), h_q, dv), device=dev)
    lse = torch.empty((len(q_seq), h_q), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_gather_attend(Q, K, V, torch.from_numpy(q_seq).to(dev), torch.from_numpy(q_pos).to(dev),
                          torch.from_numpy(sel).to(dev), torch.from_numpy(n_sel).to(dev), top_k,
                          cr, scale, O, lse=lse, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    Kn, Vn, Qn = np32(K), np32(V), np32(Q)
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    On, Ln = np32(O), np32(lse)
    for i in range(len(q_seq)):
        s, p = q_seq[i], int(q_pos[i])
        msk = oracle.mask(p, cr, sel[i], int(n_sel[i]))
        ref, rlse = oracle.attend(Qn[i], Kn[s], None if Vn is None else Vn[s], msk, scale, h_kv,
                                  dv=dv)
        err = row_rel_err(On[i], ref)
        assert err.max() < tol, (i, err.max())
        assert np.abs(Ln[i] - rlse).max() < (2e-3 if dtype == torch.bfloat16 else 1e-5)


@pytest.mark.parametrize("n_q", [32, 76, 128])
def test_gather_attend_cluster_merge(dev, n_q):
    """Decode batches whose lists the bf16 kernel splits over 8, 4 or 2 CTAs merged inside a
    cluster (no second kernel): full 512-block lists, shorter ones and tail-only ones (whose
    later splits are empty) all match the oracle, with their log-sum-exp."""
    dkq, dv, h_q, h_kv, cr, top_k = 576, 512, 16, 1, 4, 512
    n_seq, n_tok = 4, 2600
    rng = np.random.default_rng(n_q)
    q_seq = (np.arange(n_q) % n_seq).astype(np.int32)
    kinds = np.arange(n_q) % 4
    q_pos = np.where(kinds == 0, 2599, np.where(kinds == 1, 2100,
                     np.where(kinds == 2, rng.integers(300, 1800, n_q), rng.integers(0, 4, n_q))))
    q_pos = q_pos.astype(np.int32)
    Q, K, V = _attend_case(dev, dkq, dv, True, h_q, h_kv, n_seq, n_tok, q_seq, q_pos,
                           torch.bfloat16, 17 + n_q)
    sel, n_sel = _random_selection(q_pos, cr, top_k, n_q)
    scale = 1.0 / math.sqrt(dkq)
    O = torch.full((n_q, h_q, dv), float("nan"), device=dev)
    lse = torch.full((n_q, h_q), float("nan"), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_gather_attend(Q, K, V, torch.from_numpy(q_seq).to(dev), torch.from_numpy(q_pos).to(dev),
                          torch.from_numpy(sel).to(dev), torch.from_numpy(n_sel).to(dev), top_k,
                          cr, scale, O, lse=lse, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    Kn, Qn, On, Ln = np32(K), np32(Q), np32(O), np32(lse)
    for i in range(n_q):
        s, p = q_seq[i], int(q_pos[i])
        msk = oracle.mask(p, cr, sel[i], int(n_sel[i]))
        ref, rlse = oracle.attend(Qn[i], Kn[s], None, msk, scale, h_kv, dv=dv)
        assert row_rel_err(On[i], ref).max() < TOL_BF16, i
        assert np.abs(Ln[i] - rlse).max() < 2e-3, i


@pytest.mark.parametrize("cr,top_k", [(8, 512), (16, 128)])
def test_gather_attend_cluster_merge_long_tails(dev, cr, top_k):
    """32 decode queries split over 8-CTA clusters with the tail folded into the last split, at
    block sizes whose tails reach 7 and 15 tokens (every tail length occurs), against the
    oracle."""
    dkq, dv, h_q, h_kv = 576, 512, 16, 1
    n_q, n_seq = 32, 4
    n_tok = top_k * cr + 2 * cr
    q_seq = (np.arange(n_q) % n_seq).astype(np.int32)
    # full lists with every tail length, and a few short ones (later splits empty)
    q_pos = np.array([top_k * cr + (i % cr) for i in range(24)] + [cr * 3 + 1, cr - 1, 5, 2,
                     top_k * cr // 2 + 3, 0, 7, cr * 10 + cr - 2], np.int32)
    Q, K, V = _attend_case(dev, dkq, dv, True, h_q, h_kv, n_seq, n_tok, q_seq, q_pos,
                           torch.bfloat16, 31 + cr)
    sel, n_sel = _random_selection(q_pos, cr, top_k, cr)
    scale = 1.0 / math.sqrt(dkq)
    O = torch.full((n_q, h_q, dv), float("nan"), device=dev)
    lse = torch.full((n_q, h_q), float("nan"), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_gather_attend(Q, K, V, torch.from_numpy(q_seq).to(dev), torch.from_numpy(q_pos).to(dev),
                          torch.from_numpy(sel).to(dev), torch.from_numpy(n_sel).to(dev), top_k,
                          cr, scale, O, lse=lse, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    Kn, Qn, On, Ln = np32(K), np32(Q), np32(O), np32(lse)
    for i in range(n_q):
        s, p = q_seq[i], int(q_pos[i])
        msk = oracle.mask(p, cr, sel[i], int(n_sel[i]))
        ref, rlse = oracle.attend(Qn[i], Kn[s], None, msk, scale, h_kv, dv=dv)
        assert row_rel_err(On[i], ref).max() < TOL_BF16, i
        assert np.abs(Ln[i] - rlse).max() < 2e-3, i


@pytest.mark.parametrize("dkq,dv,v_is_k,h_q,h_kv", ATTN_SHAPES[:2])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_dense_attend_matches_oracle(dev, dkq, dv, v_is_k, h_q, h_kv, dtype):
    n_seq, n_tok = 2, 1100
    q_seq = np.array([0, 1, 1, 0], np.int32)
    q_pos = np.array([1099, 0, 517, 64], np.int32)
    Q, K, V = _attend_case(dev, dkq, dv, v_is_k, h_q, h_kv, n_seq, n_tok, q_seq, q_pos, dtype, 9)
    scale = 1.0 / math.sqrt(dkq)
    O = torch.empty((len(q_seq), h_q, dv), device=dev)
    sfa.sfa_dense_attend(Q, K, V, torch.from_numpy(q_seq).to(dev), torch.from_numpy(q_pos).to(dev),
                         n_tok, scale, O)
    torch.cuda.synchronize()
    Kn, Vn, Qn, On = np32(K), np32(V), np32(Q), np32(O)
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    for i in range(len(q_seq)):
        s, p = q_seq[i], int(q_pos[i])
        ref, _ = oracle.attend(Qn[i], Kn[s], None if Vn is None else Vn[s],
                               oracle.mask(p, 4, dense=True), scale, h_kv, dv=dv)
        assert row_rel_err(On[i], ref).max() < tol


def test_attend_flags_bad_block_lists(dev):
    """Out-of-range, repeated or descending block ids and bad n_sel are skipped and flagged;
    the result equals attention over the valid part of the list."""
    dkq, dv, h_q, h_kv, cr, top_k = 64, 64, 4, 1, 4, 6
    q_seq = np.array([0, 0, 0], np.int32)
    q_pos = np.array([99, 99, 99], np.int32)   # B = 25
    Q, K, V = _attend_case(dev, dkq, dv, True, h_q, h_kv, 1, 100, q_seq, q_pos, torch.bfloat16, 4)
    sel = np.array([[2, 5, 30, 7, -1, -1], [3, 3, 9, 12, -1, -1], [1, 2, 3, 4, 5, 6]], np.int32)
    n_sel = np.array([4, 4, 9], np.int32)
    O = torch.empty((3, h_q, dv), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_gather_attend(Q, K, None, torch.from_numpy(q_seq).to(dev),
                          torch.from_numpy(q_pos).to(dev), torch.from_numpy(sel).to(dev),
                          torch.from_numpy(n_sel).to(dev), top_k, cr, 0.125, O, dev_status=status)
    st = sfa.sfa_read_device_status(status)
    assert st & sfa.SFA_DEV_BAD_BLOCK and st & sfa.SFA_DEV_BAD_NSEL
    Kn, Qn, On = np32(K), np32(Q), np32(O)
    for i in range(3):
        valid = []
        for j in range(min(int(n_sel[i]), top_k)):
            b = int(sel[i, j])
            ok = 0 <= b < 25 and (j == 0 or b > int(sel[i, j - 1]))
            if ok:
                valid.append(b)
        msk = oracle.mask(99, cr, np.array(valid, np.int32), len(valid))
        ref, _ = oracle.attend(Qn[i], Kn[0], None, msk, 0.125, h_kv, dv=dv)
        assert row_rel_err(On[i], ref).max() < TOL_BF16


# ---------------------------------------------------------------------- key transform
@pytest.mark.parametrize("norm", [0, 1, 2])
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("d_idx,n_rot", [(128, 64), (64, 64), (32, 16)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_pool_transform_matches_oracle(dev, norm, neox, d_idx, n_rot, dtype):
    """Pooled keys normalised and rotated on the GPU (hi + lo) match the fp64 oracle, at block
    positions past 1e5 where only double-precision angles keep the rotation exact enough."""
    g = torch.Generator().manual_seed(norm * 10 + d_idx + int(neox))
    cr, n_seq, n_tok, b0 = 4, 2, 4 * 30000, 29500
    blk_cap = n_tok // cr
    X = (torch.randn((n_seq, n_tok, d_idx), generator=g) * 3 + 0.5).to(dtype).to(dev)
    gamma = (torch.rand(d_idx, generator=g) + 0.5).to(dev)
    beta = torch.randn(d_idx, generator=g).to(dev)
    Kbar = torch.zeros(sfa.kbar_shape(n_seq, blk_cap, d_idx), dtype=torch.bfloat16, device=dev)
    Kr = torch.zeros((n_seq, blk_cap), device=dev)
    tf = dict(norm=norm, gamma=gamma if norm else None, beta=beta if norm == 2 else None,
              eps=1e-5, n_rot=n_rot, rope_base=10000.0, rope_neox=neox, pos_offset=3)
    sfa.sfa_pool_index_keys_transformed(X, cr, b0, blk_cap, Kbar, Kr, **tf)
    torch.cuda.synchronize()
    kb = Kbar.float().cpu().double().numpy()
    got = kb[..., :d_idx] + kb[..., d_idx:]
    Xh = np32(X)
    for s in range(n_seq):
        pooled = oracle.pool(Xh[s], blk_cap, cr)
        ref = oracle.key_transform(pooled, cr, norm=norm, gamma=np32(gamma), beta=np32(beta),
                                   eps=1e-5, n_rot=n_rot, rope_base=10000.0, rope_neox=neox,
                                   pos_offset=3)[b0:]
        err = np.abs(got[s, b0:] - ref).max(axis=1) / np.abs(ref).max(axis=1)
        assert err.max() < 2e-5, (s, err.max())
        assert np.all(got[s, :b0] == 0)                       # rows outside the range untouched
        hi, lo = kb[s, b0:, :d_idx], kb[s, b0:, d_idx:]
        bound = np.sqrt((lo ** 2).sum(1)) + 2.0 ** -14 * np.sqrt((hi ** 2).sum(1))
        assert np.all(np32(Kr)[s, b0:] >= bound)


def test_step_with_key_transform_matches_oracle(dev):
    """A decode step whose pooled index keys are RMS-normalised and rotated: its selections
    follow the agreement rule against the oracle's selection on the transformed keys, and
    its outputs match the oracle attending the same cells."""
    w = sfa.WORKLOADS["decode_32x131072"].with_(n_seq=4, depth=40000, seed=21)
    case = sfa.make_case(w, device=dev)
    g = torch.Generator().manual_seed(4)
    gamma = (torch.rand(w.d_idx, generator=g) + 0.5).to(dev)
    tf = dict(norm=1, gamma=gamma, eps=1e-6, n_rot=64, rope_base=10000.0, rope_neox=True,
              pos_offset=0)
    n_blk_max = w.n_tok // w.compress_ratio
    step = sfa.SfaStep(n_seq=w.n_seq, n_tok_cap=w.n_tok, n_q=w.n_q, h_q=w.h_q, h_kv=w.h_kv,
                       dkq=w.dkq, dv=w.dv, h_idx=w.h_idx, d_idx=w.d_idx,
                       compress_ratio=w.compress_ratio, indexer_top_k=w.indexer_top_k,
                       n_blk_max=n_blk_max, key_transform=tf, device=dev)
    step.pool(case["X"], 0, n_blk_max)
    step.run(case["X"], case["K"], case["V"], case["Q"], case["q_idx"], case["w"],
             case["q_seq"], case["q_pos"], w.scale)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(step.status) == 0
    c = {k: np32(v) for k, v in case.items() if v is not None}
    got_sel, got_n, O = np32(step.blk_idx), np32(step.n_sel), np32(step.O)
    cr, n_exact = w.compress_ratio, 0
    for i in range(w.n_q):
        s, p = int(c["q_seq"][i]), int(c["q_pos"][i])
        B = (p + 1) // cr
        kbar = oracle.key_transform(oracle.pool(c["X"][s], B, cr), cr, norm=1, gamma=np32(gamma),
                                    eps=1e-6, n_rot=64, rope_base=10000.0, rope_neox=True)
        sc = oracle.index_scores(c["q_idx"][i], c["w"][i], kbar)
        ok, exact = check_selection(got_sel[i], int(got_n[i]), sc, w.indexer_top_k)
        assert ok, i
        n_exact += exact
        msk = oracle.mask(p, cr, got_sel[i], int(got_n[i]))
        ref, _ = oracle.attend(c["Q"][i], c["K"][s], None, msk, w.scale, w.h_kv, dv=w.dv)
        assert row_rel_err(O[i], ref).max() < TOL_BF16, i
    assert n_exact >= w.n_q - 1


@pytest.mark.parametrize("kernel", ["default", "mma"])
def test_dense_query_past_the_bound_is_flagged(dev, monkeypatch, kernel):
    """A dense query whose q_pos + 1 exceeds the n_kv_max the call was given: SFA_DEV_BAD_QUERY
    is raised, and the query attends its first n_kv_max keys (the other queries are exact)."""
    if kernel == "mma":
        monkeypatch.setenv("SFA_ATTEND_KERNEL", "mma")
    dkq, dv, h_q, h_kv = 576, 512, 16, 1
    n_seq, n_tok = 2, 700
    q_seq = np.array([0, 1], np.int32)
    q_pos = np.array([699, 200], np.int32)      # query 0 sees 700 keys, the bound is 500
    n_kv_max = 500
    Q, K, V = _attend_case(dev, dkq, dv, True, h_q, h_kv, n_seq, n_tok, q_seq, q_pos,
                           torch.bfloat16, 77)
    O = torch.empty((2, h_q, dv), device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_dense_attend(Q, K, V, torch.from_numpy(q_seq).to(dev),
                         torch.from_numpy(q_pos).to(dev), n_kv_max, 1.0 / math.sqrt(dkq), O,
                         dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) & sfa.SFA_DEV_BAD_QUERY
    Kn, Qn, On = np32(K), np32(Q), np32(O)
    for i, keys in ((0, n_kv_max), (1, 201)):
        msk = np.zeros(int(q_pos[i]) + 1, np.uint8)
        msk[:keys] = 1
        ref, _ = oracle.attend(Qn[i], Kn[q_seq[i]], None, msk, 1.0 / math.sqrt(dkq), h_kv, dv=dv)
        assert row_rel_err(On[i], ref).max() < TOL_BF16, i
