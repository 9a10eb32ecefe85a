"""The bounded selection (sfa_index_scores_bounded -> sfa_topk_blocks_refine): the bounds hold
against the hi + lo scores, and the refined kept sets follow the oracle's agreement rule
(the same bar as sfa_index_scores -> sfa_topk_blocks)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_selection, np32
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


def _case(dev, seed, n_seq, n_tok, d_idx, h_idx, cr, q_pos, constant_keys=False):
    g = torch.Generator().manual_seed(seed)
    if constant_keys:   # every pooled key equal: every score ties
        X = torch.ones((n_seq, n_tok, d_idx)).to(torch.bfloat16).to(dev)
    else:
        X = torch.randn((n_seq, n_tok, d_idx), generator=g).to(torch.bfloat16).to(dev)
    n_q = len(q_pos)
    qi = torch.randn((n_q, h_idx, d_idx), generator=g).to(torch.bfloat16).to(dev)
    w = torch.rand((n_q, h_idx), generator=g).to(dev)
    q_seq = torch.arange(n_q, dtype=torch.int32) % n_seq
    q_pos = torch.tensor(q_pos, dtype=torch.int32)
    blk_cap = n_tok // cr
    Kbar = torch.zeros(sfa.kbar_shape(n_seq, blk_cap, d_idx), dtype=torch.bfloat16, device=dev)
    Kr = torch.zeros((n_seq, blk_cap), dtype=torch.float32, device=dev)
    sfa.sfa_pool_index_keys(X, cr, 0, blk_cap, Kbar, Kr)
    return X, qi, w, q_seq.to(dev), q_pos.to(dev), (Kbar, Kr)


@pytest.mark.parametrize("d_idx", [128, 64, 32])
def test_pool_bound_factors(dev, d_idx):
    """r_b from the pooling pass bounds (|lo_b|_2 + 2^-14 |hi_b|_2) of the stored halves from
    above, within the fp32 margin, for bf16 and fp32 raw keys."""
    for dtype in (torch.bfloat16, torch.float32):
        g = torch.Generator().manual_seed(d_idx)
        cr, n_seq, n_tok = 3, 2, 3000
        X = (torch.randn((n_seq, n_tok, d_idx), generator=g) * 5).to(dtype).to(dev)
        blk_cap = n_tok // cr
        Kbar = torch.zeros(sfa.kbar_shape(n_seq, blk_cap, d_idx), dtype=torch.bfloat16, device=dev)
        Kr = torch.full((n_seq, blk_cap), -1.0, device=dev)
        sfa.sfa_pool_index_keys(X, cr, 7, blk_cap - 5, Kbar, Kr)
        torch.cuda.synchronize()
        kb = Kbar.float().cpu().double().numpy()
        r = np32(Kr).astype(np.float64)
        hi, lo = kb[..., :d_idx], kb[..., d_idx:]
        ref = np.sqrt((lo ** 2).sum(-1)) + 2.0 ** -14 * np.sqrt((hi ** 2).sum(-1))
        inside = slice(7, blk_cap - 5)
        assert np.all(r[:, inside] >= ref[:, inside])
        assert np.all(r[:, inside] <= ref[:, inside] * (1 + 2.0 ** -14) + 1e-30)
        assert np.all(r[:, :7] == -1.0) and np.all(r[:, blk_cap - 5:] == -1.0)   # untouched


@pytest.mark.parametrize("d_idx,h_idx", [(128, 8), (64, 4), (128, 16)])
def test_bounds_hold(dev, d_idx, h_idx):
    cr, n_seq, n_tok = 4, 3, 6000
    X, qi, w, q_seq, q_pos, Kb = _case(dev, d_idx + h_idx, n_seq, n_tok, d_idx, h_idx, cr,
                                         [5999, 4003, 1299])
    n_blk_max = 1500
    exact = torch.full((3, n_blk_max), float("nan"), device=dev)
    lower = torch.full_like(exact, float("nan"))
    upper = torch.full_like(exact, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores(qi, w, q_seq, q_pos, Kb[0], cr, n_blk_max, exact, dev_status=status)
    sfa.sfa_index_scores_bounded(qi, w, q_seq, q_pos, *Kb, cr, n_blk_max, lower, upper,
                                 dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    e, lo, up = np32(exact), np32(lower), np32(upper)
    for i, p in enumerate([5999, 4003, 1299]):
        B = (p + 1) // cr
        assert np.all(lo[i, :B] <= e[i, :B]) and np.all(e[i, :B] <= up[i, :B]), i
        assert np.all(np.isnan(lo[i, B:])) and np.all(np.isnan(up[i, B:]))
        # tight enough to be useful: a few per cent of the typical score
        half = 0.5 * (up[i, :B] - lo[i, :B])
        assert np.median(half) < 0.1 * np.median(np.abs(e[i, :B]) + 1e-30)


@pytest.mark.parametrize("d_idx,h_idx", [(128, 8), (64, 16), (128, 4)])
def test_bounds_hold_wide_tiles(dev, d_idx, h_idx):
    """The bound pass on prefill-shaped query tiles (96 queries of one sequence: tiles of 16 or
    32 queries, B operands of 128 or 256 columns, twelve epilogue warps): lower <= exact <=
    upper on every visible block, nothing written past a query's blocks."""
    cr, n_tok = 4, 6000
    pos = list(range(5999 - 95, 6000))
    X, qi, w, q_seq, q_pos, Kb = _case(dev, 5 + d_idx + h_idx, 1, n_tok, d_idx, h_idx, cr, pos)
    n_q, n_blk_max = len(pos), 1500
    exact = torch.full((n_q, n_blk_max), float("nan"), device=dev)
    lower = torch.full_like(exact, float("nan"))
    upper = torch.full_like(exact, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores(qi, w, q_seq, q_pos, Kb[0], cr, n_blk_max, exact, q_group=n_q,
                         dev_status=status)
    sfa.sfa_index_scores_bounded(qi, w, q_seq, q_pos, *Kb, cr, n_blk_max, lower, upper,
                                 q_group=n_q, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    e, lo, up = np32(exact), np32(lower), np32(upper)
    for i, p in enumerate(pos):
        B = (p + 1) // cr
        assert np.all(lo[i, :B] <= e[i, :B]) and np.all(e[i, :B] <= up[i, :B]), i
        assert np.all(np.isnan(lo[i, B:])) and np.all(np.isnan(up[i, B:])), i


@pytest.mark.parametrize("top_k", [1, 64, 512, 2048])
def test_refine_follows_agreement_rule(dev, top_k):
    cr, d_idx, h_idx = 4, 128, 8
    pos = [11999, 9000, 2047, 700, 3, 8191]
    X, qi, w, q_seq, q_pos, Kb = _case(dev, top_k, 2, 12000, d_idx, h_idx, cr, pos)
    n_q, n_blk_max = len(pos), 3000
    lower = torch.empty((n_q, n_blk_max), device=dev)
    upper = torch.empty_like(lower)
    blk = torch.full((n_q, top_k), -7, dtype=torch.int32, device=dev)
    n_sel = torch.empty(n_q, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores_bounded(qi, w, q_seq, q_pos, *Kb, cr, n_blk_max, lower, upper,
                                 dev_status=status)
    sfa.sfa_topk_blocks_refine(lower, upper, qi, w, q_seq, q_pos, Kb[0], cr, top_k, n_blk_max,
                               blk, n_sel, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    Xh, qh, wh = np32(X), np32(qi), np32(w)
    got, gn = np32(blk), np32(n_sel)
    n_exact = 0
    for i, p in enumerate(pos):
        s = i % 2
        B = (p + 1) // cr
        sc = oracle.index_scores(qh[i], wh[i], oracle.pool(Xh[s], B, cr))
        ok, exact = check_selection(got[i], int(gn[i]), sc, top_k)
        assert ok, (i, p)
        n_exact += exact
        assert np.all(np.diff(got[i, :gn[i]]) > 0)        # ascending
        assert np.all(got[i, gn[i]:] == -1)                # padded
    assert n_exact >= len(pos) - 1


@pytest.mark.parametrize("n_tok", [4000, 24000])
def test_refine_all_tied(dev, n_tok):
    """Every pooled key equal, so every score ties: every block is a candidate and the
    lowest block indices win.  At 6000 blocks the candidate list is longer than the 4096
    resolved in shared memory and takes the global-memory path."""
    cr, d_idx, h_idx, top_k = 4, 64, 4, 100
    pos = [n_tok - 1, n_tok // 2 + 1]
    X, qi, w, q_seq, q_pos, Kb = _case(dev, 3, 2, n_tok, d_idx, h_idx, cr, pos,
                                         constant_keys=True)
    n_q, n_blk_max = 2, n_tok // cr
    lower = torch.empty((n_q, n_blk_max), device=dev)
    upper = torch.empty_like(lower)
    blk = torch.empty((n_q, top_k), dtype=torch.int32, device=dev)
    n_sel = torch.empty(n_q, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores_bounded(qi, w, q_seq, q_pos, *Kb, cr, n_blk_max, lower, upper)
    sfa.sfa_topk_blocks_refine(lower, upper, qi, w, q_seq, q_pos, Kb[0], cr, top_k, n_blk_max,
                               blk, n_sel)
    torch.cuda.synchronize()
    got = np32(blk)
    assert np.array_equal(np32(n_sel), [top_k, top_k])
    for i in range(n_q):
        assert np.array_equal(got[i], np.arange(top_k))


def test_refine_many_rows_per_cluster(dev):
    """More rows than clusters (each cluster loops over several rows), rows below the budget
    (no cluster barrier for them) mixed with rows of every length up to the widest, so that
    some shares of the widest row hold no group of a shorter one."""
    cr, d_idx, h_idx, top_k = 4, 128, 8, 256
    n_tok = 16000
    rng = np.random.default_rng(5)
    pos = [int(x) for x in rng.integers(0, n_tok, size=100)]
    pos[:6] = [3, 1023, 1024, 1027, n_tok - 1, 2 * top_k * cr]   # at and around the budget
    X, qi, w, q_seq, q_pos, Kb = _case(dev, 17, 3, n_tok, d_idx, h_idx, cr, pos)
    n_q, n_blk_max = len(pos), n_tok // cr
    lower = torch.empty((n_q, n_blk_max), device=dev)
    upper = torch.empty_like(lower)
    blk = torch.full((n_q, top_k), -7, dtype=torch.int32, device=dev)
    n_sel = torch.empty(n_q, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores_bounded(qi, w, q_seq, q_pos, *Kb, cr, n_blk_max, lower, upper,
                                 dev_status=status)
    sfa.sfa_topk_blocks_refine(lower, upper, qi, w, q_seq, q_pos, Kb[0], cr, top_k, n_blk_max,
                               blk, n_sel, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    Xh, qh, wh = np32(X), np32(qi), np32(w)
    got, gn = np32(blk), np32(n_sel)
    n_exact = 0
    for i, p in enumerate(pos):
        B = (p + 1) // cr
        if B <= top_k:
            assert gn[i] == B and np.array_equal(got[i, :B], np.arange(B))
            assert np.all(got[i, B:] == -1)
            continue
        sc = oracle.index_scores(qh[i], wh[i], oracle.pool(Xh[i % 3], B, cr))
        ok, exact = check_selection(got[i], int(gn[i]), sc, top_k)
        assert ok, (i, p)
        assert np.all(np.diff(got[i, :gn[i]]) > 0)        # ascending
        n_exact += exact
    assert n_exact >= 0.9 * sum((p + 1) // cr > top_k for p in pos)


def test_refine_below_budget_and_bad_query(dev):
    cr, d_idx, h_idx, top_k = 4, 64, 4, 50
    pos = [150, 2, 3999]
    X, qi, w, q_seq, q_pos, Kb = _case(dev, 9, 1, 4000, d_idx, h_idx, cr, pos)
    n_q, n_blk_max = 3, 1000
    q_pos_bad = q_pos.clone()
    q_pos_bad[2] = -1                                     # a query outside the cache
    lower = torch.empty((n_q, n_blk_max), device=dev)
    upper = torch.empty_like(lower)
    blk = torch.empty((n_q, top_k), dtype=torch.int32, device=dev)
    n_sel = torch.empty(n_q, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores_bounded(qi, w, q_seq, q_pos_bad, *Kb, cr, n_blk_max, lower, upper,
                                 dev_status=status)
    sfa.sfa_topk_blocks_refine(lower, upper, qi, w, q_seq, q_pos_bad, Kb[0], cr, top_k,
                               n_blk_max, blk, n_sel, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) & sfa.SFA_DEV_BAD_QUERY
    got, gn = np32(blk), np32(n_sel)
    assert gn[0] == 37 and np.array_equal(got[0, :37], np.arange(37)) and np.all(got[0, 37:] == -1)
    assert gn[1] == 0 and np.all(got[1] == -1)
    assert gn[2] == 0 and np.all(got[2] == -1)


@pytest.mark.parametrize("name", ["decode_32x131072", "decode_1x4096"])
def test_bounded_step_full_size_all(dev, name):
    """The whole step with the bounded selection (SfaStep(bounded=True)) at full size: every
    query follows the oracle's agreement rule and attends within tolerance."""
    w = sfa.WORKLOADS[name]
    case, step = _run(w, dev, bounded=True)
    assert step.bounded
    _check_queries(w, case, step)


def test_bounded_step_rejects_rows_past_the_limit(dev):
    w = sfa.WORKLOADS["decode_4x1048576"]
    with pytest.raises(ValueError):
        sfa.SfaStep(n_seq=1, n_tok_cap=8 * 131073 + 8, n_q=1, h_q=w.h_q, h_kv=w.h_kv,
                    dkq=w.dkq, dv=w.dv, h_idx=w.h_idx, d_idx=w.d_idx,
                    compress_ratio=w.compress_ratio, indexer_top_k=w.indexer_top_k,
                    n_blk_max=131073, q_group=1, bounded=True, device=dev)


@pytest.mark.parametrize("pos", [[1048575, 1000000, 600000, 296000]])
def test_refine_long_rows(dev, pos):
    """Rows past one selection piece (up to 131072 blocks at cr 8): each CTA of the row's
    cluster takes eight rounds of 4096 blocks; selections follow the agreement rule."""
    cr, d_idx, h_idx, top_k = 8, 128, 8, 256
    X, qi, w, q_seq, q_pos, Kb = _case(dev, 778, 1, 1048576, d_idx, h_idx, cr, pos)
    n_q, n_blk_max = len(pos), 131072
    lower = torch.empty((n_q, n_blk_max), device=dev)
    upper = torch.empty_like(lower)
    blk = torch.empty((n_q, top_k), dtype=torch.int32, device=dev)
    n_sel = torch.empty(n_q, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores_bounded(qi, w, q_seq, q_pos, *Kb, cr, n_blk_max, lower, upper,
                                 dev_status=status)
    sfa.sfa_topk_blocks_refine(lower, upper, qi, w, q_seq, q_pos, Kb[0], cr, top_k, n_blk_max,
                               blk, n_sel, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    Xh, qh, wh = np32(X), np32(qi), np32(w)
    got, gn = np32(blk), np32(n_sel)
    kb = oracle.pool(Xh[0], (max(pos) + 1) // cr, cr)
    n_exact = 0
    for i, p in enumerate(pos):
        B = (p + 1) // cr
        sc = oracle.index_scores(qh[i], wh[i], kb[:B])
        ok, exact = check_selection(got[i], int(gn[i]), sc, top_k)
        assert ok, (i, p)
        n_exact += exact
    assert n_exact >= len(pos) - 1


def test_refine_longest_rows(dev):
    """Rows of up to the 36864-block limit: each CTA of the cluster takes three rounds of
    groups, and blocks past 32768 are candidates like any other."""
    cr, d_idx, h_idx, top_k = 4, 128, 8, 512
    pos = [147455, 144003, 131075, 40000]   # B = 36864, 36001, 32769, 10000
    X, qi, w, q_seq, q_pos, Kb = _case(dev, 777, 1, 147456, d_idx, h_idx, cr, pos)
    n_q, n_blk_max = len(pos), 36864
    lower = torch.empty((n_q, n_blk_max), device=dev)
    upper = torch.empty_like(lower)
    blk = torch.empty((n_q, top_k), dtype=torch.int32, device=dev)
    n_sel = torch.empty(n_q, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores_bounded(qi, w, q_seq, q_pos, *Kb, cr, n_blk_max, lower, upper,
                                 dev_status=status)
    sfa.sfa_topk_blocks_refine(lower, upper, qi, w, q_seq, q_pos, Kb[0], cr, top_k, n_blk_max,
                               blk, n_sel, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    Xh, qh, wh = np32(X), np32(qi), np32(w)
    got, gn = np32(blk), np32(n_sel)
    n_exact = 0
    for i, p in enumerate(pos):
        B = (p + 1) // cr
        sc = oracle.index_scores(qh[i], wh[i], oracle.pool(Xh[0], B, cr))
        ok, exact = check_selection(got[i], int(gn[i]), sc, top_k)
        assert ok, (i, p)
        n_exact += exact
        # the selection reaches past block 32768 when the best blocks are there
        top = np.argsort(-sc, kind="stable")[:top_k]
        if exact and (top >= 32768).any():
            assert (got[i] >= 32768).any()
    assert n_exact >= len(pos) - 1


# ------------------------------------------------------------------ the 8-bit bound pass
def _k8(dev, Kbar, blk_cap, d_idx, b0, b1):
    n_seq = Kbar.shape[0]
    k8s, srs = sfa.k8_shapes(n_seq, blk_cap, d_idx)
    K8 = torch.zeros(k8s, dtype=torch.int8, device=dev)
    sr = torch.full(srs, -1.0, dtype=torch.float32, device=dev)
    sfa.sfa_quantize_pooled_keys_i8(Kbar, b0, b1, K8, sr)
    return K8, sr


@pytest.mark.parametrize("d_idx", [128, 64])
def test_quantize_pooled_keys_i8(dev, d_idx):
    """Codes, scale and bound factor per row, checked against their definition in float64:
    sc = max|m| / 127 (m = hi + lo), |m - sc c| <= sc / 2 elementwise, and the stored factor
    covers |m - sc c|_2 + 2^-14 sc |c|_2 by at most a few ulps; rows outside the range are not
    written, and a zero row gives zero codes, scale and factor."""
    cr, n_seq, n_tok = 4, 2, 4000
    X, qi, w, q_seq, q_pos, Kb = _case(dev, 31 + d_idx, n_seq, n_tok, d_idx, 4, cr, [3999, 17])
    Kbar = Kb[0]
    blk_cap = n_tok // cr
    Kbar[1, 500].zero_()                                   # a zero row
    b0, b1 = 3, blk_cap - 2
    K8, sr = _k8(dev, Kbar, blk_cap, d_idx, b0, b1)
    torch.cuda.synchronize()
    kb = np32(Kbar).astype(np.float64)
    m = kb[..., :d_idx] + kb[..., d_idx:]
    c = K8.cpu().numpy().view(np.uint8).astype(np.float64) - 128.0   # stored as c + 128
    s = np32(sr).astype(np.float64)
    sc, r = s[..., 0], s[..., 1]
    rows = slice(b0, b1)
    mx = np.abs(m[:, rows]).max(-1)
    assert np.allclose(sc[:, rows], mx / 127, rtol=2 ** -22, atol=0)
    assert np.all(np.abs(c[:, rows]) <= 127)
    res = m[:, rows] - sc[:, rows, None] * c[:, rows]
    assert np.all(np.abs(res) <= 0.5 * sc[:, rows, None] * (1 + 2 ** -14) + 1e-38)
    need = np.linalg.norm(res, axis=-1) + 2 ** -14 * sc[:, rows] * np.linalg.norm(c[:, rows], axis=-1)
    assert np.all(r[:, rows] >= need)
    assert np.all(r[:, rows] <= need * (1 + 2 ** -12) + 1e-38)
    assert sc[1, 500] == 0 and r[1, 500] == 0 and np.all(c[1, 500] == 0)
    raw = K8.cpu().numpy()
    assert np.all(raw[:, :b0] == 0) and np.all(raw[:, b1:] == 0)      # not written
    assert np.all(s[:, :b0] == -1.0) and np.all(s[:, b1:] == -1.0)


@pytest.mark.parametrize("d_idx,h_idx", [(128, 8), (64, 4), (128, 16), (64, 16)])
def test_bounds_hold_i8(dev, d_idx, h_idx):
    """The 8-bit bounds bracket the hi + lo scores the exact pass computes, for every visible
    block of queries of several lengths (partial last tiles included)."""
    cr, n_seq, n_tok = 4, 3, 6000
    pos = [5999, 4003, 1299, 511, 5000]
    X, qi, w, q_seq, q_pos, Kb = _case(dev, 7 * d_idx + h_idx, n_seq, n_tok, d_idx, h_idx, cr,
                                         pos)
    n_blk_max = 1500
    K8, sr = _k8(dev, Kb[0], n_tok // cr, d_idx, 0, n_blk_max)
    exact = torch.full((len(pos), n_blk_max), float("nan"), device=dev)
    lower = torch.full_like(exact, float("nan"))
    upper = torch.full_like(exact, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores(qi, w, q_seq, q_pos, Kb[0], cr, n_blk_max, exact, dev_status=status)
    sfa.sfa_index_scores_bounded_i8(qi, w, q_seq, q_pos, K8, sr, cr, n_blk_max, lower, upper,
                                    dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    e, lo, up = np32(exact), np32(lower), np32(upper)
    for i, p in enumerate(pos):
        B = (p + 1) // cr
        assert np.all(lo[i, :B] <= e[i, :B]) and np.all(e[i, :B] <= up[i, :B]), i
        assert np.all(np.isnan(lo[i, B:])) and np.all(np.isnan(up[i, B:]))
        # useful, if looser than the hi-only bounds (a fifth of the typical score)
        half = 0.5 * (up[i, :B] - lo[i, :B])
        assert np.median(half) < 0.3 * np.median(np.abs(e[i, :B]) + 1e-30)


@pytest.mark.parametrize("top_k", [64, 512, 2048])
def test_refine_follows_agreement_rule_i8(dev, top_k):
    cr, d_idx, h_idx = 4, 128, 8
    pos = [11999, 9000, 2047, 700, 3, 8191]
    X, qi, w, q_seq, q_pos, Kb = _case(dev, top_k + 3, 2, 12000, d_idx, h_idx, cr, pos)
    n_q, n_blk_max = len(pos), 3000
    K8, sr = _k8(dev, Kb[0], 3000, d_idx, 0, n_blk_max)
    lower = torch.empty((n_q, n_blk_max), device=dev)
    upper = torch.empty_like(lower)
    blk = torch.full((n_q, top_k), -7, dtype=torch.int32, device=dev)
    n_sel = torch.empty(n_q, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores_bounded_i8(qi, w, q_seq, q_pos, K8, sr, cr, n_blk_max, lower, upper,
                                    dev_status=status)
    sfa.sfa_topk_blocks_refine(lower, upper, qi, w, q_seq, q_pos, Kb[0], cr, top_k, n_blk_max,
                               blk, n_sel, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    Xh, qh, wh = np32(X), np32(qi), np32(w)
    got, gn = np32(blk), np32(n_sel)
    n_exact = 0
    for i, p in enumerate(pos):
        B = (p + 1) // cr
        sc = oracle.index_scores(qh[i], wh[i], oracle.pool(Xh[i % 2], B, cr))
        ok, exact = check_selection(got[i], int(gn[i]), sc, top_k)
        assert ok, (i, p)
        assert np.all(np.diff(got[i, :gn[i]]) > 0)
        assert np.all(got[i, gn[i]:] == -1)
        n_exact += exact
    assert n_exact >= len(pos) - 1


@pytest.mark.parametrize("n_tok", [4000, 24000])
def test_refine_all_tied_i8(dev, n_tok):
    """Every pooled key equal: the 8-bit bounds are equal too, every block is a candidate
    (past 4096 of them, the global-memory list) and the lowest block indices win."""
    cr, d_idx, h_idx, top_k = 4, 64, 4, 100
    pos = [n_tok - 1, n_tok // 2 + 1]
    X, qi, w, q_seq, q_pos, Kb = _case(dev, 5, 2, n_tok, d_idx, h_idx, cr, pos,
                                         constant_keys=True)
    n_q, n_blk_max = 2, n_tok // cr
    K8, sr = _k8(dev, Kb[0], n_blk_max, d_idx, 0, n_blk_max)
    lower = torch.empty((n_q, n_blk_max), device=dev)
    upper = torch.empty_like(lower)
    blk = torch.empty((n_q, top_k), dtype=torch.int32, device=dev)
    n_sel = torch.empty(n_q, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sfa.sfa_index_scores_bounded_i8(qi, w, q_seq, q_pos, K8, sr, cr, n_blk_max, lower, upper,
                                    dev_status=status)
    sfa.sfa_topk_blocks_refine(lower, upper, qi, w, q_seq, q_pos, Kb[0], cr, top_k, n_blk_max,
                               blk, n_sel, dev_status=status)
    torch.cuda.synchronize()
    assert sfa.sfa_read_device_status(status) == 0
    assert np.array_equal(np32(n_sel), [top_k, top_k])
    got = np32(blk)
    for i in range(n_q):
        assert np.array_equal(got[i], np.arange(top_k))


@pytest.mark.parametrize("name,bound_pass", [("decode_32x131072", "hi"),
                                             ("decode_4x1048576", "hi"),
                                             ("decode_cr1_32x32768", "i8")])
def test_bound_passes_full_size_all(dev, name, bound_pass):
    """Every query of the full-size decode workloads through either bound pass (the i8 pass is
    the default and the other full-size tests run it)."""
    w = sfa.WORKLOADS[name]
    case, step = _run(w, dev, bound_pass=bound_pass)
    assert step.bound_pass == bound_pass
    _check_queries(w, case, step)
