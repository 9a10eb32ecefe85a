"""Calibration of the parity harness with planted mistakes.

The GPU parity tests check the library in two ways: the selection-agreement rule on the
kept blocks (``check_selection``) and the per-row relative error of the outputs
(``row_rel_err`` against ``TOL_BF16``).  A harness that cannot fail proves nothing, so this
file plants the plausible mistakes of the method -- a kept block swapped for the first one
below the cut, a kept block dropped, the tail left out, a tie at the cut broken the wrong
way -- into otherwise correct results and checks that the harness rejects each one.  This
follows the noise-floor check the qwen4exp commit text describes (llama.cpp commit "model:
add Qwen3.8-Flash-Next (qwen4exp)": deliberate bugs planted to see that the comparison
catches them).

The CPU tests plant the mistakes in the oracle's own results.  The GPU test plants them in
the kept-block list the GPU selected (a data corruption on the host: every id stays in range)
and feeds the corrupted list through ``sfa_gather_attend``.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import GAP_REL, TOL_BF16, check_selection, np32, row_rel_err

sfa = pytest.importorskip("indexer_selected_sparse_block_gb300")


def _oracle_case(depth=3000, top_k=256, seed=31):
    """One decode query (576/512, V = K, cr 4) at the given depth, drawn on the CPU."""
    w = sfa.WORKLOADS["decode_1x4096"].with_(depth=depth, indexer_top_k=top_k, seed=seed)
    c = {k: np32(v) for k, v in sfa.make_case(w, device="cpu").items()}
    p = int(c["q_pos"][0])
    B = (p + 1) // w.compress_ratio
    kb = oracle.pool(c["X"][0], B, w.compress_ratio)
    sc = oracle.index_scores(c["q_idx"][0], c["w"][0], kb)
    sel, n = oracle.select(sc, top_k)
    return w, c, p, sc, sel, n


def _attend(w, c, p, msk):
    O, lse = oracle.attend(c["Q"][0], c["K"][0], None, msk, w.scale, w.h_kv, dv=w.dv)
    return O, lse


def _cut(sc, top_k):
    order = np.lexsort((np.arange(sc.shape[0]), -sc))
    return order[top_k - 1], order[top_k]


def test_harness_accepts_the_correct_result():
    w, c, p, sc, sel, n = _oracle_case()
    ok, exact = check_selection(sel, n, sc, w.indexer_top_k)
    assert ok and exact
    O, _ = _attend(w, c, p, oracle.mask(p, w.compress_ratio, sel, n))
    assert row_rel_err(O, O).max() == 0.0


def test_harness_rejects_a_swapped_block():
    """The k-th kept block replaced by the (k+1)-th: the selection check fails (the gap at
    the cut exceeds 1e-4) and the attention over the wrong set is far outside tolerance."""
    w, c, p, sc, sel, n = _oracle_case()
    kth, k1th = _cut(sc, w.indexer_top_k)
    assert (sc[kth] - sc[k1th]) / abs(sc[kth]) > GAP_REL
    bad = np.sort(np.where(sel[:n] == kth, k1th, sel[:n])).astype(np.int32)
    ok, _ = check_selection(bad, n, sc, w.indexer_top_k)
    assert not ok
    ref, _ = _attend(w, c, p, oracle.mask(p, w.compress_ratio, sel, n))
    got, _ = _attend(w, c, p, oracle.mask(p, w.compress_ratio, bad, n))
    assert row_rel_err(got, ref).max() > 5 * TOL_BF16


def test_harness_rejects_a_dropped_block():
    w, c, p, sc, sel, n = _oracle_case()
    ok, _ = check_selection(sel[: n - 1], n - 1, sc, w.indexer_top_k)
    assert not ok
    ref, _ = _attend(w, c, p, oracle.mask(p, w.compress_ratio, sel, n))
    got, _ = _attend(w, c, p, oracle.mask(p, w.compress_ratio, sel, n - 1))
    assert row_rel_err(got, ref).max() > 5 * TOL_BF16


@pytest.mark.parametrize("depth", [3000, 3002])
def test_harness_rejects_a_dropped_tail(depth):
    """The tail (the tokens after the last complete block) left out of the attended set:
    one token at depth 3000, three at depth 3002."""
    w, c, p, sc, sel, n = _oracle_case(depth=depth)
    full = oracle.mask(p, w.compress_ratio, sel, n)
    no_tail = full.copy()
    no_tail[((p + 1) // w.compress_ratio) * w.compress_ratio:] = 0
    assert no_tail.sum() < full.sum()
    ref, _ = _attend(w, c, p, full)
    got, _ = _attend(w, c, p, no_tail)
    assert row_rel_err(got, ref).max() > TOL_BF16


def test_harness_rejects_a_flipped_tie():
    """Ties at the cut broken toward the higher block index: the agreement rule accepts it
    (both sets are correct up to the tie), so the tie rule is enforced where the tests compare
    selections bit for bit (the top-k stage tests) -- and that comparison fails here."""
    rng = np.random.default_rng(5)
    top_k, B = 64, 500
    sc = rng.random(B) * 3.0
    cut = np.sort(sc)[::-1][top_k - 1]
    tied = rng.choice(B, size=12, replace=False)
    sc[tied] = cut
    ref, n = oracle.select(sc, top_k)
    order_flipped = np.lexsort((-np.arange(B), -sc))   # higher index first among ties
    flipped = np.sort(order_flipped[:top_k]).astype(np.int32)
    assert not np.array_equal(flipped, ref[:n])
    ok, exact = check_selection(flipped, top_k, sc, top_k)
    assert ok and not exact


def test_harness_rejects_an_output_off_by_the_tolerance():
    """An output perturbed by 1.5x the tolerance in one element of one row fails the row
    check; one perturbed by half the tolerance passes."""
    w, c, p, sc, sel, n = _oracle_case()
    ref, _ = _attend(w, c, p, oracle.mask(p, w.compress_ratio, sel, n))
    for factor, fails in ((1.5, True), (0.5, False)):
        got = ref.copy()
        got[3, 100] += factor * TOL_BF16 * np.abs(ref[3]).max()
        assert (row_rel_err(got, ref).max() > TOL_BF16) == fails


@pytest.mark.gpu
def test_gpu_harness_rejects_corrupted_kept_lists():
    """The GPU's own kept list, corrupted on the host (k-th block swapped for the (k+1)-th; last
    kept block dropped) and attended by sfa_gather_attend: the harness flags both, while the
    uncorrupted list passes."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    w = sfa.WORKLOADS["decode_1x4096"].with_(depth=3000, seed=31)
    case = sfa.make_case(w, device=dev)
    step = sfa.SfaStep(n_seq=w.n_seq, n_tok_cap=w.n_tok, n_q=w.n_q, h_q=w.h_q, h_kv=w.h_kv,
                       dkq=w.dkq, dv=w.dv, h_idx=w.h_idx, d_idx=w.d_idx,
                       compress_ratio=w.compress_ratio, indexer_top_k=w.indexer_top_k,
                       n_blk_max=w.n_tok // w.compress_ratio, device=dev)
    step.pool(case["X"], 0, step.n_blk_max)
    step.run(case["X"], case["K"], case["V"], case["Q"], case["q_idx"], case["w"],
             case["q_seq"], case["q_pos"], w.scale)
    torch.cuda.synchronize()
    c = {k: np32(v) for k, v in case.items()}
    p = int(c["q_pos"][0])
    kb = oracle.pool(c["X"][0], (p + 1) // w.compress_ratio, w.compress_ratio)
    sc = oracle.index_scores(c["q_idx"][0], c["w"][0], kb)
    sel, n = oracle.select(sc, w.indexer_top_k)
    ref, _ = _attend(w, c, p, oracle.mask(p, w.compress_ratio, sel, n))
    gsel, gn = np32(step.blk_idx)[0], int(np32(step.n_sel)[0])
    kth, k1th = _cut(sc, w.indexer_top_k)

    def attend_list(lst, n_kept):
        blk = torch.full((1, w.indexer_top_k), -1, dtype=torch.int32)
        blk[0, :n_kept] = torch.from_numpy(np.asarray(lst[:n_kept], np.int32))
        n_sel = torch.tensor([n_kept], dtype=torch.int32)
        O = torch.empty((1, w.h_q, w.dv), device=dev)
        sfa.sfa_gather_attend(case["Q"], case["K"], case["V"], case["q_seq"], case["q_pos"],
                              blk.to(dev), n_sel.to(dev), w.indexer_top_k, w.compress_ratio,
                              w.scale, O)
        torch.cuda.synchronize()
        return np32(O)[0]

    assert check_selection(gsel, gn, sc, w.indexer_top_k) == (True, True)
    assert row_rel_err(attend_list(gsel, gn), ref).max() < TOL_BF16
    swapped = np.sort(np.where(gsel[:gn] == kth, k1th, gsel[:gn])).astype(np.int32)
    assert not check_selection(swapped, gn, sc, w.indexer_top_k)[0]
    assert row_rel_err(attend_list(swapped, gn), ref).max() > 5 * TOL_BF16
    assert not check_selection(gsel[: gn - 1], gn - 1, sc, w.indexer_top_k)[0]
    assert row_rel_err(attend_list(gsel, gn - 1), ref).max() > 5 * TOL_BF16
