"""Pins of the oracle to facts fixed outside itself (CPU only).

Each ``pin_*`` function checks the oracle against a closed form, a hand-derived worked
example (``tests/golden``), brute force, an invariant the pages state, or an independent
library routine (numpy / torch fp64).  ``test_mutants_are_caught`` plants plausible
mistakes in a copy of the oracle's C source and checks that some pin fails for each one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16(a):
    """Round an fp32 array to bf16 values (the inputs of the method are bf16)."""
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


# --------------------------------------------------------------------------------- pool
def pin_pool_closed_forms(lib):
    # cr = 1: the pooled key is the key itself.
    X = _bf16(_rng(1).standard_normal((37, 8)))
    assert np.array_equal(oracle.pool(X, 37, 1, lib=lib), X.astype(np.float64))
    # a constant key pools to the same constant
    C = np.full((24, 5), 0.375, np.float32)
    assert np.array_equal(oracle.pool(C, 6, 4, lib=lib), np.full((6, 5), 0.375))
    # ramp X[t][d] = t + d/4: mean over block b is b*cr + (cr-1)/2 + d/4 (exact)
    for cr in (2, 3, 4, 8):
        nb = 5
        t = np.arange(nb * cr + 3, dtype=np.float32)[:, None]
        d = np.arange(6, dtype=np.float32)[None, :]
        R = t + d / 4
        want = (np.arange(nb)[:, None] * cr + (cr - 1) / 2 + np.arange(6)[None, :] / 4)
        assert np.array_equal(oracle.pool(R, nb, cr, lib=lib), want)
    # against numpy's own mean (independent library routine)
    X = _bf16(_rng(2).standard_normal((64 * 4 + 3, 16)))
    want = X[: 64 * 4].astype(np.float64).reshape(64, 4, 16).mean(axis=1)
    np.testing.assert_allclose(oracle.pool(X, 64, 4, lib=lib), want, rtol=0, atol=1e-15)


def pin_pool_cells(lib):
    # Worked example of the paged layout: four cells, position t held in cell [2, 0, 3, 1][t],
    # cr 2.  Block 0 covers positions 0 and 1 (cells 2 and 0): (4 + 1)/2, (40 + 10)/2; block 1
    # covers positions 2 and 3 (cells 3 and 1): (8 + 2)/2, (80 + 20)/2.  Reading the map the
    # wrong way round (cell -> position) or ignoring it gives other values.
    X = np.array([[1, 10], [2, 20], [4, 40], [8, 80]], np.float32)
    assert np.array_equal(oracle.pool_cells(X, [2, 0, 3, 1], 2, 2, lib=lib),
                          [[2.5, 25.0], [5.0, 50.0]])
    # the identity map is the per-sequence layout
    Y = _bf16(_rng(40).standard_normal((130, 16)))
    assert np.array_equal(oracle.pool_cells(Y, np.arange(130), 32, 4, lib=lib),
                          oracle.pool(Y, 32, 4, lib=lib))
    # a shuffled page table (10 of 14 pages of 16 cells, the rest unused), against numpy's
    # block means of the gathered rows
    r = _rng(41)
    page = 16
    pages = r.permutation(14)[:10]
    cell_of = (pages[:, None] * page + np.arange(page)[None, :]).reshape(-1)
    cells = _bf16(r.standard_normal((14 * page, 8)))
    want = cells[cell_of].astype(np.float64)[:160].reshape(40, 4, 8).mean(axis=1)
    np.testing.assert_allclose(oracle.pool_cells(cells, cell_of, 40, 4, lib=lib), want,
                               rtol=0, atol=1e-15)
    # an entry outside the cell array is an error, not a read
    with pytest.raises(ValueError):
        oracle.pool_cells(X, [2, 0, 4, 1], 2, 2, lib=lib)


# ----------------------------------------------------------------------- q8_0 KV blocks
def pin_q8_0(lib):
    # Worked example: amax 127 gives delta = 1 exactly; codes round half away from zero.
    x = np.zeros((1, 64), np.float32)
    x[0, :7] = [127, 0.5, -0.5, 1.5, -2.5, 2.49, -126.5]
    q, s = oracle.quantize_q8_0(x, lib=lib)
    assert q[0, :7].tolist() == [127, 1, -1, 2, -3, 2, -127] and not q[0, 7:].any()
    assert s.tolist() == [[0x3C00, 0x0000]]                # 1.0; the all-zero block has scale 0
    assert oracle.dequantize_q8_0(q, s, lib=lib)[0, :7].tolist() == [127, 1, -1, 2, -3, 2, -127]
    # Codes are taken with the unrounded delta.  amax = 127 (1 + 2^-12) gives delta = 1 + 2^-12,
    # stored as binary16 1.0; x = 2.5 + 2^-11 is 2.4999 deltas (code 2), but 2.5005 stored scales.
    y = np.zeros((1, 32), np.float32)
    y[0, 0], y[0, 1] = 127 * (1 + 2.0 ** -12), 2.5 + 2.0 ** -11
    q, s = oracle.quantize_q8_0(y, lib=lib)
    assert q[0, :2].tolist() == [127, 2] and s[0, 0] == 0x3C00
    # Scales that fall exactly between two binary16 values round to the even one.
    for delta, bits in [(1 + 2.0 ** -11, 0x3C00), (1 + 3 * 2.0 ** -11, 0x3C02),
                        (2.0 ** -24 * 1.5, 0x0002), (2.0 ** -24 * 2.5, 0x0002)]:
        z = np.zeros((1, 32), np.float32)
        z[0, 0] = 127 * delta
        assert np.float32(z[0, 0]) / np.float32(127) == np.float32(delta)
        assert oracle.quantize_q8_0(z, lib=lib)[1][0, 0] == bits, delta
    # Values on the code grid come back exactly: x = k * 2^-3, one |k| = 127 per block.
    k = _rng(50).integers(-127, 128, (20, 96))
    k[:, ::32] = 127 * np.sign(k[:, ::32] + 0.5).astype(np.int64)
    g = (k * 0.125).astype(np.float32)
    q, s = oracle.quantize_q8_0(g, lib=lib)
    assert np.array_equal(q, k) and np.all(s == 0x3000)      # 2^-3
    assert np.array_equal(oracle.dequantize_q8_0(q, s, lib=lib), g)
    # binary16 rounding of the scale against numpy's conversion, over many binades
    r = _rng(51)
    v = (r.standard_normal(50000) * 10.0 ** r.integers(-10, 6, 50000)).astype(np.float32)
    with np.errstate(over="ignore"):                          # large values go to infinity
        want = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.fp16_bits(v, lib=lib), want)
    # Error bound on random rows: |s q - x| <= delta / 2 (rounding of the code, plus the binary32
    # division) + 127 |s - delta| (the binary16 scale).
    X = (r.standard_normal((300, 128)) * 10.0 ** r.integers(-6, 5, (300, 1))).astype(np.float32)
    q, s = oracle.quantize_q8_0(X, lib=lib)
    assert np.abs(q.astype(np.int64)).max() <= 127
    xb = X.astype(np.float64).reshape(300, 4, 32)
    delta = (np.float32(1) * np.abs(X).reshape(300, 4, 32).max(-1) / np.float32(127)).astype(np.float64)
    sv = s.view(np.float16).astype(np.float64)
    err = np.abs(oracle.dequantize_q8_0(q, s, lib=lib).astype(np.float64).reshape(300, 4, 32) - xb)
    bound = delta * 0.5 * (1 + 2.0 ** -20) + 127 * np.abs(sv - delta)
    assert np.all(err <= bound[..., None])
    # a scale that overflows binary16 is an error
    with pytest.raises(ValueError):
        oracle.quantize_q8_0(np.full((1, 32), 1e7, np.float32), lib=lib)


# -------------------------------------------------------------------------------- score
def pin_scores(lib):
    g = _golden("qsa_tiny_relu.json")
    kbar = oracle.pool(np.array(g["X"], np.float32), 2, g["compress_ratio"], lib=lib)
    assert np.array_equal(kbar, np.array(g["expect"]["kbar"], np.float64))
    s = oracle.index_scores(np.array(g["q_idx"]), np.array(g["w"]), kbar, lib=lib)
    assert np.array_equal(s, np.array(g["expect"]["score"], np.float64))
    # one head, unit weight: ReLU(q . kbar), checked against numpy's einsum
    r = _rng(3)
    kb = r.standard_normal((50, 32))
    q = _bf16(r.standard_normal((1, 32)))
    want = np.maximum(np.einsum("bd,d->b", kb, q[0].astype(np.float64)), 0.0)
    np.testing.assert_allclose(oracle.index_scores(q, np.ones(1), kb, lib=lib), want,
                               rtol=1e-14, atol=1e-14)
    # heads enter with their weights: w = e_j selects head j alone
    qs = _bf16(r.standard_normal((4, 32)))
    for j in range(4):
        w = np.zeros(4)
        w[j] = 1.0
        want = np.maximum(kb @ qs[j].astype(np.float64), 0.0)
        np.testing.assert_allclose(oracle.index_scores(qs, w, kb, lib=lib), want, rtol=1e-14,
                                   atol=1e-14)
    # all-positive keys and queries: every dot is positive; negated queries rectify to 0
    kp = np.abs(kb) + 0.1
    qp = np.abs(qs) + 0.1
    assert np.all(oracle.index_scores(qp, np.full(4, 0.5), kp, lib=lib) > 0)
    assert np.all(oracle.index_scores(-qp, np.full(4, 0.5), kp, lib=lib) == 0.0)
    # positive homogeneity in w (power of two: exact)
    w = np.abs(r.standard_normal(4)).astype(np.float32)
    s1 = oracle.index_scores(qs, w, kb, lib=lib)
    s2 = oracle.index_scores(qs, 2 * w, kb, lib=lib)
    assert np.array_equal(2 * s1, s2)


# ------------------------------------------------------------------------------- select
def _brute_force_select(score, k):
    """Max-sum k-subset, ties broken by the lexicographically smallest ascending ids."""
    best = None
    for c in itertools.combinations(range(len(score)), k):
        key = (-sum(score[i] for i in c), c)
        if best is None or key < best:
            best = key
    return list(best[1])


def pin_select(lib):
    g = _golden("qsa_tie_cut.json")
    sel, n = oracle.select(np.array(g["score"], np.float64), g["indexer_top_k"], lib=lib)
    assert n == g["expect"]["n_sel"] and list(sel[:n]) == g["expect"]["sel"]
    g1 = _golden("qsa_tiny_relu.json")
    sel, n = oracle.select(np.array(g1["expect"]["score"], np.float64), 1, lib=lib)
    assert n == 1 and list(sel) == g1["expect"]["sel"]
    # every block fits the budget: all blocks, ascending, -1 padded
    sel, n = oracle.select(np.array([3.0, 1.0, 2.0]), 5, lib=lib)
    assert n == 3 and list(sel) == [0, 1, 2, -1, -1]
    sel, n = oracle.select(np.zeros(0), 4, lib=lib)
    assert n == 0 and list(sel) == [-1] * 4
    # brute force over all subsets (integer scores: sums exact, many ties)
    r = _rng(4)
    for trial in range(60):
        B = int(r.integers(1, 12))
        k = int(r.integers(1, B + 1))
        score = r.integers(0, 4, size=B).astype(np.float64)
        sel, n = oracle.select(score, k, lib=lib)
        assert n == k
        assert list(sel[:n]) == _brute_force_select(list(score), k), (score, k)
    # all-equal scores: the lowest k blocks
    sel, n = oracle.select(np.zeros(40), 7, lib=lib)
    assert list(sel) == list(range(7))


def pin_token_expanded(lib):
    """The graph formulation: expand block scores to tokens, token-level top-(k*cr) with the
    lower token winning ties.  It must keep exactly the tokens of the kept blocks."""
    r = _rng(5)
    for trial in range(40):
        cr = int(r.choice([1, 2, 4, 8]))
        B = int(r.integers(1, 60))
        k = int(r.integers(1, 70))
        score = np.round(r.standard_normal(B), 1)   # coarse: ties are common
        sel, n = oracle.select(score, k, lib=lib)
        tok_score = np.repeat(score, cr)
        order = np.lexsort((np.arange(B * cr), -tok_score))   # score desc, token asc
        tokens = np.sort(order[: min(k, B) * cr])
        want = np.concatenate([np.arange(b * cr, b * cr + cr) for b in sel[:n]]) if n else []
        assert np.array_equal(tokens, np.asarray(want, dtype=tokens.dtype))


# --------------------------------------------------------------------------------- mask
def pin_mask(lib):
    g = _golden("qsa_tie_cut.json")
    m = oracle.mask(g["p"], g["compress_ratio"], np.array(g["expect"]["sel"]), 3, lib=lib)
    assert list(np.nonzero(m)[0]) == g["expect"]["attended"]
    r = _rng(6)
    for trial in range(40):
        cr = int(r.choice([1, 2, 3, 4, 8]))
        p = int(r.integers(0, 200))
        B = (p + 1) // cr
        k = int(r.integers(1, 40))
        score = r.standard_normal(B)
        sel, n = oracle.select(score, k, lib=lib)
        m = oracle.mask(p, cr, sel, n, lib=lib)
        assert m.shape == (p + 1,)
        assert int(m.sum()) == n * cr + (p + 1) % cr          # |A| = n_sel*cr + |tail|
        assert np.all(m[B * cr:] == 1)                        # the tail is always kept
        assert n == min(k, B)
    assert np.all(oracle.mask(9, 4, dense=True, lib=lib) == 1)


def pin_mask_window(lib):
    """The windowed attended set (dense window + kept blocks + tail): hand-derived sets; no
    window is the plain set; a window reaching position 0 is every position; the set only
    grows with the window; and the window suffix with the kept tokens before it is a disjoint
    cover of the set, over which attention splits exactly into two log-sum-exp-combined
    parts (the decomposition the dense + sparse variant computes)."""
    for c in _golden("qsa_window.json")["cases"]:
        sel = np.array(c["sel"], np.int32)
        m = oracle.mask(c["p"], c["compress_ratio"], sel, len(sel), window=c["window"], lib=lib)
        assert list(np.nonzero(m)[0]) == c["attended"], c["derivation"][0]
    r = _rng(17)
    for trial in range(30):
        cr = int(r.choice([1, 2, 3, 4, 8]))
        p = int(r.integers(0, 160))
        B = (p + 1) // cr
        k = int(r.integers(1, 20))
        sel, n = oracle.select(r.standard_normal(B), k, lib=lib)
        plain = oracle.mask(p, cr, sel, n, lib=lib)
        assert np.array_equal(oracle.mask(p, cr, sel, n, window=0, lib=lib), plain)
        assert np.all(oracle.mask(p, cr, sel, n, window=p + 1 + int(r.integers(0, 5)), lib=lib) == 1)
        prev = plain
        for W in sorted(r.integers(1, p + 2, 4)):
            cur = oracle.mask(p, cr, sel, n, window=int(W), lib=lib)
            assert np.all(cur >= prev) and cur.sum() >= prev.sum()
            prev = cur
    # attention over the set == the two parts combined by their log-sum-exp
    r = _rng(19)
    h_q, h_kv, dkq, dv, cr, p, W = 4, 2, 32, 16, 4, 70, 13
    K = r.standard_normal((p + 1, h_kv, dkq)).astype(np.float32)
    V = r.standard_normal((p + 1, h_kv, dv)).astype(np.float32)
    q = r.standard_normal((h_q, dkq)).astype(np.float32)
    sel, n = oracle.select(r.standard_normal((p + 1) // cr), 5, lib=lib)
    full = oracle.mask(p, cr, sel, n, window=W, lib=lib)
    s0 = min(((p + 1) // cr) * cr, p - W + 1)
    suffix = np.zeros(p + 1, np.uint8)
    suffix[s0:] = 1
    before = oracle.mask(p, cr, sel, n, lib=lib).copy()
    before[s0:] = 0
    assert np.array_equal(suffix | before, full) and not np.any(suffix & before)
    O, lse = oracle.attend(q, K, V, full, 0.2, h_kv, lib=lib)
    Oa, la = oracle.attend(q, K, V, suffix, 0.2, h_kv, lib=lib)
    Ob, lb = oracle.attend(q, K, V, before, 0.2, h_kv, lib=lib)
    M = np.maximum(la, lb)
    wa, wb = np.exp(la - M), np.exp(lb - M)
    np.testing.assert_allclose(O, (wa[:, None] * Oa + wb[:, None] * Ob) / (wa + wb)[:, None],
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, M + np.log(wa + wb), rtol=1e-13)


# ------------------------------------------------------------------------------- attend
def _sdpa_fp64(q, K, V, msk, scale, group):
    """torch's scaled_dot_product_attention in fp64 over the masked tokens."""
    qt = torch.from_numpy(q.astype(np.float64))[:, None, :]          # [h][1][d]
    Kt = torch.from_numpy(K.astype(np.float64)).repeat_interleave(group, dim=1).permute(1, 0, 2)
    Vt = torch.from_numpy(V.astype(np.float64)).repeat_interleave(group, dim=1).permute(1, 0, 2)
    am = torch.from_numpy(msk.astype(bool))[None, None, :].expand(qt.shape[0], 1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=am, scale=scale)
    logits = (qt @ Kt.transpose(1, 2))[:, 0, :] * scale
    lse = torch.logsumexp(logits.masked_fill(~am[:, 0, :], -math.inf), dim=-1)
    return o[:, 0, :].numpy(), lse.numpy()


def pin_attend(lib):
    g = _golden("qsa_tiny_relu.json")
    e = math.e
    Q = np.array(g["Q"], np.float32)
    K = np.array(g["K"], np.float32)[:, None, :]
    V = np.array(g["V"], np.float32)[:, None, :]
    O, lse = oracle.attend(Q, K, V, np.array(g["expect"]["mask"]), 1.0, 1, lib=lib)
    den = e + 1 + e * e
    np.testing.assert_allclose(O[0], [(7 * e + e * e) / den, (7 + e * e) / den], rtol=1e-14)
    np.testing.assert_allclose(lse[0], math.log(den), rtol=1e-14)
    O, _ = oracle.attend(Q, K, V, np.ones(5), 1.0, 1, lib=lib)
    den = 3 + e + e * e
    np.testing.assert_allclose(O[0], [(9 + 7 * e + e * e) / den, (9 + 7 + e * e) / den],
                               rtol=1e-14)
    r = _rng(7)
    for (h_q, h_kv, dkq, dv, v_is_k) in [(16, 1, 576, 512, True), (16, 2, 512, 512, False),
                                         (8, 1, 64, 32, False), (4, 4, 16, 16, True)]:
        n = 45
        q = _bf16(r.standard_normal((h_q, dkq)))
        K = _bf16(r.standard_normal((n, h_kv, dkq)))
        V = None if v_is_k else _bf16(r.standard_normal((n, h_kv, dv)))
        msk = (r.random(n) < 0.6).astype(np.uint8)
        msk[-1] = 1
        scale = 1.0 / math.sqrt(dkq)
        O, lse = oracle.attend(q, K, V, msk, scale, h_kv, dv=dv, lib=lib)
        Vf = K[..., :dv] if v_is_k else V
        want, want_lse = _sdpa_fp64(q, K, Vf, msk, scale, h_q // h_kv)
        np.testing.assert_allclose(O, want, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, want_lse, rtol=1e-12, atol=1e-13)
        # compacted rows: token t reads row tok_row[t]
        idx = np.nonzero(msk)[0]
        rows = np.full(n, -1, np.int64)
        rows[idx] = np.arange(len(idx))
        O2, _ = oracle.attend(q, np.ascontiguousarray(K[idx]),
                              None if V is None else np.ascontiguousarray(V[idx]), msk, scale,
                              h_kv, dv=dv, tok_row=rows, lib=lib)
        assert np.array_equal(O, O2)
    # q = 0: the plain mean of V over the attended set
    K = _bf16(r.standard_normal((30, 1, 8)))
    V = _bf16(r.standard_normal((30, 1, 4)))
    msk = (np.arange(30) % 3 == 0).astype(np.uint8)
    O, lse = oracle.attend(np.zeros((2, 8)), K, V, msk, 0.5, 1, lib=lib)
    np.testing.assert_allclose(O[1], V[msk == 1, 0].astype(np.float64).mean(0), rtol=1e-14,
                               atol=1e-15)
    np.testing.assert_allclose(lse, math.log(10), rtol=1e-15)
    # identical V rows: the output is that row whatever the logits
    Vc = np.repeat(V[:1], 30, axis=0)
    O, _ = oracle.attend(_bf16(r.standard_normal((2, 8))), K, Vc, msk, 0.5, 1, lib=lib)
    np.testing.assert_allclose(O, np.repeat(Vc[0], 2, axis=0), rtol=1e-14)
    # one attended token: the output is its V row
    one = np.zeros(30, np.uint8)
    one[17] = 1
    O, _ = oracle.attend(_bf16(r.standard_normal((2, 8))), K, V, one, 0.5, 1, lib=lib)
    assert np.array_equal(O, np.repeat(V[17].astype(np.float64), 2, axis=0))


# ----------------------------------------------------------------------------- pipeline
def _small_case(seed, n_seq=2, n_tok=70, h_q=4, h_kv=2, dkq=16, dv=8, v_is_k=False, h_idx=3,
                d_idx=8):
    r = _rng(seed)
    n_q = 5
    X = _bf16(r.standard_normal((n_seq, n_tok, d_idx)))
    K = _bf16(r.standard_normal((n_seq, n_tok, h_kv, dkq)))
    V = None if v_is_k else _bf16(r.standard_normal((n_seq, n_tok, h_kv, dv)))
    Q = _bf16(r.standard_normal((n_q, h_q, dkq)))
    qi = _bf16(r.standard_normal((n_q, h_idx, d_idx)))
    w = r.random((n_q, h_idx)).astype(np.float32)
    q_seq = np.array([0, 1, 1, 0, 1], np.int32)[:n_q] % n_seq
    q_pos = np.array([n_tok - 1, 0, 2, 40, 47], np.int32)
    return dict(X=X, q_idx=qi, w=w, Q=Q, K=K, V=V, q_seq=q_seq, q_pos=q_pos, dv=dv)


def pin_pipeline(lib):
    g = _golden("qsa_tiny_relu.json")
    X = np.array(g["X"], np.float32)[None]
    K = np.array(g["K"], np.float32)[None, :, None, :]
    V = np.array(g["V"], np.float32)[None, :, None, :]
    out = oracle.run(X, np.array(g["q_idx"], np.float32)[None], np.array(g["w"])[None],
                     np.array(g["Q"], np.float32)[None], K, V, [0], [g["p"]], cr=2, top_k=1,
                     scale=1.0, want_scores=True, lib=lib)
    assert list(out["sel"][0]) == [1] and list(out["score"][0, :2]) == [2.0, 3.0]
    e = math.e
    den = e + 1 + e * e
    np.testing.assert_allclose(out["O"][0, 0], [(7 * e + e * e) / den, (7 + e * e) / den],
                               rtol=1e-14)
    c = _small_case(11)
    cr = 4
    # below the budget (B_i <= top_k for every query) sparse is exactly dense
    big_k = (int(c["q_pos"].max()) + 1) // cr
    sp = oracle.run(**c, cr=cr, top_k=big_k, scale=0.25, lib=lib)
    de = oracle.run(**c, cr=cr, top_k=0, scale=0.25, lib=lib)
    assert np.array_equal(sp["O"], de["O"]) and np.array_equal(sp["lse"], de["lse"])
    # above it, the output is attention over the brute-force best block subset + tail
    k = 3
    sp = oracle.run(**c, cr=cr, top_k=k, scale=0.25, want_scores=True, lib=lib)
    for i in range(5):
        s, p = int(c["q_seq"][i]), int(c["q_pos"][i])
        B = (p + 1) // cr
        if B > 12:
            continue
        if B > 0:
            kb = c["X"][s, : B * cr].astype(np.float64).reshape(B, cr, -1).mean(1)
            sc = np.einsum("jd,bd->bj", c["q_idx"][i].astype(np.float64), kb)
            sc = (np.maximum(sc, 0) * c["w"][i].astype(np.float64)).sum(1)
            best = _brute_force_select(list(sc), min(k, B))
        else:
            best = []
        assert list(sp["sel"][i][: min(k, B)]) == best
        msk = np.zeros(p + 1, np.uint8)
        for b in best:
            msk[b * cr: b * cr + cr] = 1
        msk[B * cr:] = 1
        want, _ = _sdpa_fp64(c["Q"][i], c["K"][s, : p + 1], c["V"][s, : p + 1], msk, 0.25, 2)
        np.testing.assert_allclose(sp["O"][i], want, rtol=1e-12, atol=1e-13)
    # stream isolation: changing sequence 1's data leaves sequence 0's queries bit-identical
    c2 = dict(c)
    c2["X"] = c["X"].copy()
    c2["K"] = c["K"].copy()
    c2["V"] = c["V"].copy()
    c2["X"][1] *= -1
    c2["K"][1] += 1
    c2["V"][1] += 1
    sp2 = oracle.run(**c2, cr=cr, top_k=k, scale=0.25, lib=lib)
    for i in range(5):
        same = np.array_equal(sp["O"][i], sp2["O"][i])
        assert same == (c["q_seq"][i] == 0)


# ------------------------------------------------------------------------ key transform
def pin_key_transform(lib):
    kt = lambda k, cr, **kw: oracle.key_transform(k, cr, lib=lib, **kw)  # noqa: E731
    rng = _rng(31)
    K = rng.standard_normal((6, 16))
    # nothing to do: the identity
    assert np.array_equal(kt(K, 4), K)
    # a rotation at position 0 (block 0, no offset) is the identity
    for neox in (True, False):
        assert np.allclose(kt(K[:1], 4, n_rot=16, rope_neox=neox), K[:1], rtol=0, atol=1e-15)
    # rotations preserve every row's length
    R = kt(K, 3, n_rot=16, pos_offset=11)
    np.testing.assert_allclose(np.linalg.norm(R, axis=1), np.linalg.norm(K, axis=1), rtol=1e-13)
    # dot products of rotated vectors depend only on their position difference
    q, k = rng.standard_normal(16), rng.standard_normal(16)
    rows = np.zeros((13, 16))
    rows[5], rows[2], rows[12], rows[9] = q, k, q, k
    for neox in (True, False):
        Rr = kt(rows, 1, n_rot=16, rope_base=50.0, rope_neox=neox)
        assert abs(Rr[5] @ Rr[2] - Rr[12] @ Rr[9]) < 1e-12
        same = np.zeros((4, 16))
        same[3] = q
        a = kt(same, 1, n_rot=16, rope_neox=neox)[3]
        same[3] = k
        b = kt(same, 1, n_rot=16, rope_neox=neox)[3]
        assert abs(a @ b - q @ k) < 1e-12
    # closed forms: block 1 at cr = 4 sits at position 4; pair 0 turns by 4 rad, pair 1 of
    # n_rot = 4 by 4 / sqrt(base) rad
    base = 100.0
    e = np.zeros((2, 4))
    e[1, 0] = 1.0                                   # dim 0: pair 0 in both pairings
    r = kt(e, 4, n_rot=4, rope_base=base, rope_neox=True)[1]
    np.testing.assert_allclose(r, [math.cos(4), 0, math.sin(4), 0], atol=1e-15)   # (0, 2)
    r = kt(e, 4, n_rot=4, rope_base=base, rope_neox=False)[1]
    np.testing.assert_allclose(r, [math.cos(4), math.sin(4), 0, 0], atol=1e-15)   # (0, 1)
    e = np.zeros((2, 4))
    e[1, 1] = 1.0                                   # dim 1: NeoX pair 1 (1, 3); adjacent pair 0
    t1 = 4 / math.sqrt(base)
    np.testing.assert_allclose(kt(e, 4, n_rot=4, rope_base=base, rope_neox=True)[1],
                               [0, math.cos(t1), 0, math.sin(t1)], atol=1e-15)
    np.testing.assert_allclose(kt(e, 4, n_rot=4, rope_base=base, rope_neox=False)[1],
                               [-math.sin(4), math.cos(4), 0, 0], atol=1e-15)
    # the norms: statistics of the result (eps = 0, unit gain)
    y = kt(K, 4, norm=1, eps=0.0)
    np.testing.assert_allclose((y ** 2).mean(1), 1.0, rtol=1e-13)
    y = kt(K, 4, norm=2, eps=0.0)
    np.testing.assert_allclose(y.mean(1), 0.0, atol=1e-13)
    np.testing.assert_allclose((y ** 2).mean(1), 1.0, rtol=1e-13)
    # a constant row: RMS norm gives gamma * sign, layer norm gives beta
    g = rng.uniform(0.5, 2, 16).astype(np.float32)
    bt = rng.standard_normal(16).astype(np.float32)
    c = np.full((1, 16), -3.0)
    np.testing.assert_allclose(kt(c, 1, norm=1, gamma=g, eps=0.0)[0], -g.astype(np.float64),
                               rtol=1e-14)
    np.testing.assert_allclose(kt(c, 1, norm=2, gamma=g, beta=bt, eps=1e-6)[0],
                               bt.astype(np.float64), rtol=0, atol=0)
    # the norm comes before the rotation (with a non-uniform gain the two do not commute)
    both = kt(K, 2, norm=1, gamma=g, n_rot=16, pos_offset=3)
    step = kt(kt(K, 2, norm=1, gamma=g), 2, n_rot=16, pos_offset=3)
    np.testing.assert_allclose(both, step, rtol=1e-14)
    rot_first = kt(kt(K, 2, n_rot=16, pos_offset=3), 2, norm=1, gamma=g)
    assert not np.allclose(both, rot_first, rtol=1e-6)


PINS = [pin_pool_closed_forms, pin_pool_cells, pin_q8_0, pin_scores, pin_select, pin_token_expanded, pin_mask,
        pin_mask_window, pin_attend, pin_pipeline, pin_key_transform]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, olib):
    pin(olib)


# Plausible mistakes, planted in a copy of the oracle source (never in the real one).
MUTANTS = {
    "no_relu": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "ties_to_higher_block": ("return (a->b < b->b) ? -1 : (a->b > b->b);",
                             "return (a->b > b->b) ? -1 : (a->b < b->b);"),
    "tail_dropped": ("for (int64_t t = n_blk * cr; t < n_vis; ++t) mask[t] = 1;", ""),
    "sum_not_mean": ("(int64_t)d_idx + d];\n            kbar[b * d_idx + d] = sum / (double)cr;",
                     "(int64_t)d_idx + d];\n            kbar[b * d_idx + d] = sum;"),
    "pool_window_shifted": ("X[(b * cr + t) * (int64_t)d_idx + d]",
                            "X[(b * cr + t + 1) * (int64_t)d_idx + d]"),
    "cell_map_ignored": ("sum += (double)X[(int64_t)cell_of[b * cr + t] * d_idx + d];",
                         "sum += (double)X[(b * cr + t) * (int64_t)d_idx + d];"),
    "q8_truncated_codes": ("qb[j] = delta == 0.0f ? 0 : (int8_t)roundf(xb[j] / delta);",
                           "qb[j] = delta == 0.0f ? 0 : (int8_t)truncf(xb[j] / delta);"),
    "q8_codes_from_stored_scale": ("qb[j] = delta == 0.0f ? 0 : (int8_t)roundf(xb[j] / delta);",
                                   "qb[j] = delta == 0.0f ? 0 : (int8_t)roundf(xb[j] / fp16_value(fp16_bits(delta)));"),
    "q8_amax_over_128": ("const float delta = amax / 127.0f;", "const float delta = amax / 128.0f;"),
    "fp16_ties_away": ("double frac = nearbyint(ldexp(m, 11));", "double frac = round(ldexp(m, 11));"),
    "scale_dropped": ("logit[t] = scale * dot;", "logit[t] = dot;"),
    "wrong_kv_head": ("const int g = h / group;", "const int g = h % h_kv;"),
    "weight_outside_relu": ("s += (double)w[j] * relu;", "s += relu;"),
    "budget_short_by_one": ("n_sel = top_k;", "n_sel = top_k - 1;"),
    "ascending_score": ("if (a->s > b->s) return -1;\n    if (a->s < b->s) return 1;",
                        "if (a->s < b->s) return -1;\n    if (a->s > b->s) return 1;"),
    "no_max_subtract_sign": ("const double e = exp(logit[t] - m);",
                             "const double e = exp(m - logit[t]);"),
    "v_from_wrong_offset": ("K + r * k_row_stride + (int64_t)g * dkq;\n            const double e",
                            "K + r * k_row_stride + (int64_t)g * dkq + 1;\n            const double e"),
    "rope_sin_sign": ("x[ia] = xa * cos(theta) - xb * sin(theta);",
                      "x[ia] = xa * cos(theta) + xb * sin(theta);"),
    "rope_neox_partner": ("ib = rope_neox ? j + n_rot / 2 : 2 * j + 1;",
                          "ib = rope_neox ? j + 1 : 2 * j + 1;"),
    "rms_without_root": ("const double r = sqrt(ss / d_idx + eps);",
                         "const double r = ss / d_idx + eps;"),
    "position_ignores_cr": ("const double p = (double)(b * cr + pos_offset);",
                            "const double p = (double)(b + pos_offset);"),
    "window_one_too_long": ("int64_t first = p - window + 1;", "int64_t first = p - window;"),
    "window_ignored": ("for (int64_t t = first; t <= p; ++t) mask[t] = 1;", ""),
    "lse_without_max": ("if (lse) lse[h] = m + log(denom);", "if (lse) lse[h] = log(denom);"),
    "kept_block_short_by_one": ("t < (int64_t)sel[i] * cr + cr; ++t) mask[t] = 1;",
                                "t < (int64_t)sel[i] * cr + cr - 1; ++t) mask[t] = 1;"),
    "one_head_weight": ("s += (double)w[j] * relu;", "s += (double)w[0] * relu;"),
    "one_index_query": ("dot += (double)q_idx[j * d_idx + d] * kbar[b * d_idx + d];",
                        "dot += (double)q_idx[d] * kbar[b * d_idx + d];"),
    "kept_ids_unsorted": ("qsort(sel, (size_t)n_sel, sizeof(int32_t), ascending_i32);", ""),
}


def test_mutants_are_caught(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "sfa_oracle.c")).read()
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, name
        path = str(tmp_path / f"mut_{name}.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load(oracle.build(force=True, src=path, out=str(tmp_path / f"{name}.so")))
        caught = []
        for pin in PINS:
            try:
                pin(lib)
            except AssertionError:
                caught.append(pin.__name__)
        assert caught, f"planted mistake '{name}' passed every pin"
