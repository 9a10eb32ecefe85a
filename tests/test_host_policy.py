"""The step's choice of selection path (host logic, CPU): the bounded pair for decode-like steps
that would stream at least 96 MiB of pooled keys through the exact scores, with rows of at most
131072 blocks and at most four queries per sequence; the 8-bit bound pass up to a budget of
1024 blocks and the hi-only pass above it; the exact pair otherwise, and the dense path below
the budget.  A step built with device="cpu" allocates its buffers and launches nothing."""
import pytest


@pytest.fixture(scope="module")
def sfa():
    import __graft_entry__
    __graft_entry__.build()
    import indexer_selected_sparse_block_gb300
    return indexer_selected_sparse_block_gb300


def _step(sfa, w, **kw):
    return sfa.SfaStep(n_seq=w.n_seq, n_tok_cap=w.n_tok, n_q=w.n_q, h_q=w.h_q, h_kv=w.h_kv,
                       dkq=w.dkq, dv=w.dv, h_idx=w.h_idx, d_idx=w.d_idx,
                       compress_ratio=w.compress_ratio, indexer_top_k=w.indexer_top_k,
                       n_blk_max=w.n_tok // w.compress_ratio, q_group=w.n_q_per_seq,
                       device="cpu", **kw)


@pytest.mark.parametrize("name,bounded,bound_pass,dense", [
    ("decode_1x4096", False, None, False),          # 0.5 MB of pooled keys: exact
    ("prefill_512x8192", False, None, False),       # 512 queries per sequence: exact
    ("prefill_512x1000", False, None, True),        # below the budget: dense
    ("decode_32x131072", True, "i8", False),        # 537 MB: bounded, 8-bit pass
    ("pp2048_131072", False, None, False),          # prefill: exact
    ("decode_4x1048576", True, "i8", False),        # 268 MB, 131072-block rows: bounded
    ("decode_cr1_32x32768", True, "hi", False),     # budget 2048 > 1024: hi-only pass
])
def test_default_selection_path(sfa, name, bounded, bound_pass, dense):
    st = _step(sfa, sfa.WORKLOADS[name])
    assert (st.bounded, st.bound_pass, st.dense) == (bounded, bound_pass, dense)


def test_threshold_and_overrides(sfa):
    w = sfa.WORKLOADS["decode_32x131072"]
    # the same decode with a quarter of the queries streams 134 MB (bounded), with a
    # sixteenth 33.5 MB (exact)
    assert _step(sfa, w.with_(n_seq=8)).bounded
    assert not _step(sfa, w.with_(n_seq=2)).bounded
    # explicit choices win over the default
    assert not _step(sfa, w, bounded=False).bounded
    assert _step(sfa, w.with_(n_seq=2), bounded=True).bounded
    assert _step(sfa, w, bound_pass="hi").bound_pass == "hi"
    with pytest.raises(ValueError):
        _step(sfa, w, bound_pass="fp8")
