"""Helpers shared by the GPU parity tests: tensor marshalling for the oracle, the error
metrics, and the selection-agreement rule.  No arithmetic of the method lives here."""
import numpy as np
import torch

# Attention outputs: max over (query, head) rows of max_d |O - O_ref| / max_d |O_ref|.
TOL_BF16 = 2e-3
TOL_F32 = 1e-5
# Kept-block sets must match exactly where the oracle's k-th / (k+1)-th score gap exceeds
# this relative amount.
GAP_REL = 1e-4


def np32(t):
    """A torch tensor (any device) as a float32 / int numpy array (bf16 -> f32 is exact)."""
    if t is None:
        return None
    t = t.detach().cpu()
    if t.is_floating_point():
        return t.float().numpy()
    return t.numpy()


def row_rel_err(got, ref):
    """Per-row relative error: max_d |got - ref| / max_d |ref| (rows = all leading dims)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.abs(got - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    return num / np.maximum(den, 1e-30)


def check_selection(got_sel, got_n, ref_score, top_k):
    """The selection-agreement rule for one query.

    Returns (ok, exact): exact is True when the oracle's gap at the cut exceeds GAP_REL (the
    sets must then be identical); otherwise every differing block must have an oracle score
    within GAP_REL * |s_(k)| of the cut score s_(k).
    """
    B = ref_score.shape[0]
    got = sorted(int(b) for b in got_sel[:got_n])
    if B <= top_k:
        return got == list(range(B)) and got_n == B, True
    order = np.lexsort((np.arange(B), -ref_score))
    ref = sorted(int(b) for b in order[:top_k])
    sk, sk1 = ref_score[order[top_k - 1]], ref_score[order[top_k]]
    denom = abs(sk) if sk != 0 else 1.0
    exact = (sk - sk1) / denom > GAP_REL
    if exact:
        return got == ref and got_n == top_k, True
    if got_n != top_k or len(set(got)) != top_k or any(b < 0 or b >= B for b in got):
        return False, False
    diff = set(got) ^ set(ref)
    ok = all(abs(ref_score[b] - sk) <= GAP_REL * denom for b in diff)
    return ok, False
