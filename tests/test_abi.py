"""The C ABI on the host (no GPU needed): the library loads, exports every entry point that
include/sfa.h declares, and rejects invalid arguments before enqueuing anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from indexer_selected_sparse_block_gb300 import _binding
    return _binding.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "sfa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sfa_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    from indexer_selected_sparse_block_gb300 import _binding
    assert set(names) <= set(_binding.SIGNATURES)


def test_status_strings(L):
    for code in range(5):
        assert L.sfa_status_string(code).startswith(b"SFA_")
    assert b"unknown" in L.sfa_status_string(99)


FAKE = ctypes.c_void_p(0x10000)     # never dereferenced: every call below is rejected first
ODD = ctypes.c_void_p(0x10008)      # not 16-byte aligned


def test_pool_rejects_bad_arguments(L):
    f = L.sfa_pool_index_keys
    assert f(None, 0, 1024, 1, 64, 4, 0, 4, FAKE, 1024, None, 0, None) == 1
    assert f(FAKE, 2, 1024, 1, 64, 4, 0, 4, FAKE, 1024, None, 0, None) == 1          # dtype
    assert f(FAKE, 0, 1024, 1, 48, 4, 0, 4, FAKE, 1024, None, 0, None) == 2          # d_idx
    assert f(FAKE, 0, 1024, 1, 64, 0, 0, 4, FAKE, 1024, None, 0, None) == 1          # cr
    assert f(FAKE, 0, 1024, 1, 64, 4, 5, 4, FAKE, 1024, None, 0, None) == 1          # begin > end
    assert f(ODD, 0, 1024, 1, 64, 4, 0, 4, FAKE, 1024, None, 0, None) == 1           # alignment
    assert f(FAKE, 0, 100, 1, 64, 4, 0, 4, FAKE, 1024, None, 0, None) == 1           # X too short
    assert f(FAKE, 0, 1024, 1, 64, 4, 0, 4, FAKE, 1024, FAKE, 3, None) == 1          # Kbar_r short
    assert f(FAKE, 0, 1536, 1, 96, 4, 0, 4, FAKE, 1024, FAKE, 4, None) == 2          # r for 96
    assert f(FAKE, 0, 1024, 1, 64, 4, 0, 0, FAKE, 1024, None, 0, None) == 0          # empty: no work


def test_pool_transform_rejects_bad_arguments(L):
    f = L.sfa_pool_index_keys_transformed
    F = ctypes.c_float
    #     X     dt  stride n_seq d   cr b0 b1 norm gamma beta eps      n_rot base      neox off
    ok = [FAKE, 0, 1024, 1, 64, 4, 0, 4, 1, FAKE, None, F(1e-6), 32, F(1e4), 1, 0,
          FAKE, 1024, None, 0, None]
    bad = list(ok); bad[8] = 3
    assert f(*bad) == 1                                                    # norm kind
    bad = list(ok); bad[9] = None
    assert f(*bad) == 1                                                    # RMS norm, no gain
    bad = list(ok); bad[8] = 2
    assert f(*bad) == 1                                                    # layer norm, no bias
    bad = list(ok); bad[11] = F(float("nan"))
    assert f(*bad) == 1                                                    # eps
    bad = list(ok); bad[12] = 33
    assert f(*bad) == 1                                                    # odd n_rot
    bad = list(ok); bad[12] = 128
    assert f(*bad) == 1                                                    # n_rot > d_idx
    bad = list(ok); bad[12] = 24
    assert f(*bad) == 2                                                    # NeoX needs n_rot % 16
    bad = list(ok); bad[13] = F(-1.0)
    assert f(*bad) == 1                                                    # rotary base
    bad = list(ok); bad[4], bad[2] = 96, 1536
    assert f(*bad) == 2                                                    # 96-wide keys
    bad = list(ok); bad[7] = 0
    assert f(*bad) == 0                                                    # empty range: no work


def test_scores_reject_bad_arguments(L):
    f = L.sfa_index_scores
    ok = [FAKE, FAKE, FAKE, FAKE, 4, 1, 8, 128, 4, FAKE, 256 * 100, 1, 100, FAKE, 100, None, None]
    bad = list(ok); bad[7] = 96
    assert f(*bad) == 2                                                    # d_idx
    bad = list(ok); bad[6] = 5
    assert f(*bad) == 2                                                    # h_idx
    bad = list(ok); bad[12] = 101
    assert f(*bad) == 1                                                    # n_blk_max > cap
    bad = list(ok); bad[5] = 0
    assert f(*bad) == 1                                                    # q_group
    bad = list(ok); bad[10] = 250
    assert f(*bad) == 1                                                    # stride % 2*d_idx


def test_bounded_entry_points_reject_bad_arguments(L):
    f = L.sfa_index_scores_bounded
    #     q_idx w     q_seq q_pos n_q grp h  d    cr Kbar  stride     Kbar_r kr   n_seq nbm
    ok = [FAKE, FAKE, FAKE, FAKE, 4, 1, 8, 128, 4, FAKE, 256 * 100, FAKE, 100, 1, 100,
          FAKE, FAKE, 100, None, None]
    bad = list(ok); bad[11] = None
    assert f(*bad) == 1                                                    # no bound factors
    bad = list(ok); bad[12] = 99
    assert f(*bad) == 1                                                    # factor rows short
    bad = list(ok); bad[16] = None
    assert f(*bad) == 1                                                    # no upper array
    g = L.sfa_topk_blocks_refine
    #     lower upper stride q_idx w  q_seq q_pos n_q h  d   Kbar  kstride    n_seq cr top_k nbm
    ok = [FAKE, FAKE, 100, FAKE, FAKE, FAKE, FAKE, 4, 8, 128, FAKE, 256 * 100, 1, 4, 16, 100,
          FAKE, FAKE, FAKE, 1 << 20, None, None]
    bad = list(ok); bad[15] = 131073
    assert g(*bad) == 2                                                    # rows > 131072
    bad = list(ok); bad[14] = 0
    assert g(*bad) == 2                                                    # top_k
    bad = list(ok); bad[10] = ODD
    assert g(*bad) == 1                                                    # Kbar alignment
    bad = list(ok); bad[18] = None
    assert g(*bad) == 4                                                    # workspace
    assert L.sfa_topk_refine_workspace_bytes(4, 100) > 4 * 100 * 8


def test_topk_rejects_bad_arguments(L):
    f = L.sfa_topk_blocks
    assert f(FAKE, 100, FAKE, 4, 4, 0, 100, FAKE, FAKE, None, 0, None, None) == 2     # top_k 0
    assert f(FAKE, 100, FAKE, 4, 4, 4096, 100, FAKE, FAKE, None, 0, None, None) == 2  # > 2048
    assert f(FAKE, 50, FAKE, 4, 4, 16, 100, FAKE, FAKE, None, 0, None, None) == 1     # stride
    assert f(FAKE, 100, FAKE, 4, 0, 16, 100, FAKE, FAKE, None, 0, None, None) == 1    # cr
    need = L.sfa_topk_workspace_bytes(4, 100000, 512)
    assert need > 0
    assert f(FAKE, 100000, FAKE, 4, 4, 512, 100000, FAKE, FAKE, None, 0, None, None) == 4
    assert L.sfa_topk_workspace_bytes(4, 1000, 512) == 0                  # one chunk: none


def test_attend_rejects_bad_arguments(L):
    f = L.sfa_gather_attend
    base = [FAKE, FAKE, None, 0, 1, 4096, 1, 16, 1, 576, 512, ctypes.c_float(0.04), FAKE, FAKE,
            FAKE, FAKE, 256, 4, FAKE, None, None, 0, None, None]
    a = list(base); a[9], a[10] = 320, 256
    assert f(*a) == 2                                                      # head dim
    a = list(base); a[7], a[8] = 12, 5
    assert f(*a) == 1                                                      # h_q % h_kv
    a = list(base); a[7], a[8] = 32, 1
    assert f(*a) == 2                                                      # 32 heads per KV head
    a = list(base); a[11] = ctypes.c_float(float("nan"))
    assert f(*a) == 1                                                      # scale
    a = list(base); a[16] = 0
    assert f(*a) == 1                                                      # top_k
    a = list(base); a[0] = ODD
    assert f(*a) == 1                                                      # alignment
    a = list(base); a[10] = 576; a[9] = 512
    assert f(*a) == 1                                                      # dv > dkq, V NULL
    g = L.sfa_dense_attend
    assert g(FAKE, FAKE, None, 0, 1, 4096, 1, 16, 1, 576, 512, ctypes.c_float(0.04), FAKE, FAKE,
             0, FAKE, None, None, 0, None, None) == 1                      # n_kv_max 0


def test_paged_entry_points_reject_bad_arguments(L):
    f = L.sfa_pool_index_keys_paged
    #       X     dt  n_cells cell_of cap   seq d_idx cr b0 b1 Kbar  stride Kr    kr  status
    base = [FAKE, 0, 5000, FAKE, 4096, 2, 64, 4, 0, 1024, FAKE, 131072, None, 0, None, None]
    assert f(*base[:3], None, *base[4:]) == 1                                     # no map
    a = list(base); a[2] = 0
    assert f(*a) == 1                                                             # no cells
    a = list(base); a[4] = 4095
    assert f(*a) == 1                                                             # map too short
    a = list(base); a[6] = 48
    assert f(*a) == 2                                                             # d_idx
    a = list(base); a[0] = ODD
    assert f(*a) == 1                                                             # alignment
    a = list(base); a[9] = 0
    assert f(*a) == 0                                                             # empty: no work
    g = L.sfa_gather_attend_paged
    base = [FAKE, FAKE, None, 0, 5000, FAKE, 1, 4096, 1, 16, 1, 576, 512, ctypes.c_float(0.04),
            FAKE, FAKE, FAKE, FAKE, 256, 4, FAKE, None, None, 0, None, None]
    a = list(base); a[5] = None
    assert g(*a) == 1                                                             # no map
    a = list(base); a[4] = 0
    assert g(*a) == 1                                                             # no cells
    a = list(base); a[4] = 1 << 31
    assert g(*a) == 1                                                             # cells >= 2^31
    a = list(base); a[11], a[12] = 320, 256
    assert g(*a) == 2                                                             # head dim
    h = L.sfa_dense_attend_paged
    assert h(FAKE, FAKE, None, 0, 5000, None, 1, 4096, 1, 16, 1, 576, 512, ctypes.c_float(0.04),
             FAKE, FAKE, 4096, FAKE, None, None, 0, None, None) == 1               # no map
    assert h(FAKE, FAKE, None, 0, 0, FAKE, 1, 4096, 1, 16, 1, 576, 512, ctypes.c_float(0.04),
             FAKE, FAKE, 4096, FAKE, None, None, 0, None, None) == 1               # no cells


def test_q8_0_entry_points(L):
    assert [L.sfa_q8_0_row_bytes(d) for d in (64, 128, 512, 576, 100, 0)] == [80, 144, 544, 624, 0, 0]
    f = L.sfa_quantize_kv_q8_0
    #       X     dt n_out n_in  d    x_outer Y     y_outer status stream
    base = [FAKE, 0, 2, 100, 576, 57600, FAKE, 62400, None, None]
    assert f(None, *base[1:]) == 1                                                # no X
    a = list(base); a[1] = 2
    assert f(*a) == 1                                                             # x dtype
    a = list(base); a[4] = 96
    assert f(*a) == 2                                                             # d
    a = list(base); a[2] = -1
    assert f(*a) == 1                                                             # n_outer
    a = list(base); a[6] = ODD
    assert f(*a) == 1                                                             # Y alignment
    a = list(base); a[7] = 62400 - 16
    assert f(*a) == 1                                                             # Y groups overlap
    a = list(base); a[5] = 57599
    assert f(*a) == 1                                                             # X groups overlap
    a = list(base); a[3] = 0
    assert f(*a) == 0                                                             # empty: no work
    g = L.sfa_gather_attend
    assert g(FAKE, FAKE, None, 3, 1, 4096, 1, 16, 1, 576, 512, ctypes.c_float(0.04), FAKE, FAKE,
             FAKE, FAKE, 256, 4, FAKE, None, None, 0, None, None) == 1     # dtype 3


def test_copy_cache_rows_rejects_bad_arguments(L):
    f = L.sfa_copy_cache_rows
    #       dst   dpitch src   spitch row  n  stream
    base = [FAKE, 2048, FAKE, 1152, 1152, 32, None]
    a = list(base); a[4] = 0
    assert f(*a) == 1                                                             # no row bytes
    a = list(base); a[1] = 1024
    assert f(*a) == 1                                                             # dst rows overlap
    a = list(base); a[3] = 1000
    assert f(*a) == 1                                                             # src rows overlap
    a = list(base); a[5] = -1
    assert f(*a) == 1                                                             # n_rows
    a = list(base); a[0] = None
    assert f(*a) == 1                                                             # no dst
    a = list(base); a[2] = None
    assert f(*a) == 1                                                             # no src
    a = list(base); a[0] = None; a[5] = 0
    assert f(*a) == 0                                                             # empty: no work


def test_i8_bound_pass_rejects_bad_arguments(L):
    q = L.sfa_quantize_pooled_keys_i8
    #     Kbar  kstride  n_seq d   b0 b1   K8    k8stride  sr    srstride stream
    ok = [FAKE, 256 * 100, 2, 128, 0, 100, FAKE, 128 * 100, FAKE, 200, None]
    bad = list(ok); bad[3] = 96
    assert q(*bad) == 2                                                    # d_idx
    bad = list(ok); bad[7] = 128 * 99
    assert q(*bad) == 1                                                    # code rows short
    bad = list(ok); bad[9] = 199
    assert q(*bad) == 1                                                    # (scale, r) pairs short
    bad = list(ok); bad[6] = ODD
    assert q(*bad) == 1                                                    # K8 alignment
    bad = list(ok); bad[4] = 5; bad[5] = 4
    assert q(*bad) == 1                                                    # begin > end
    bad = list(ok); bad[5] = 0
    assert q(*bad) == 0                                                    # empty: no work
    f = L.sfa_index_scores_bounded_i8
    #     q_idx w     q_seq q_pos n_q h  d    cr K8    k8stride   sr    srstride n_seq nbm
    ok = [FAKE, FAKE, FAKE, FAKE, 4, 8, 128, 4, FAKE, 128 * 100, FAKE, 200, 1, 100,
          FAKE, FAKE, 100, None, None]
    bad = list(ok); bad[5] = 5
    assert f(*bad) == 2                                                    # h_idx
    bad = list(ok); bad[6] = 32
    assert f(*bad) == 2                                                    # d_idx
    bad = list(ok); bad[13] = 101
    assert f(*bad) == 1                                                    # n_blk_max > cap
    bad = list(ok); bad[11] = 198
    assert f(*bad) == 1                                                    # pairs short
    bad = list(ok); bad[9] = 128 * 100 + 8
    assert f(*bad) == 1                                                    # stride % d_idx
    bad = list(ok); bad[15] = None
    assert f(*bad) == 1                                                    # no upper array
    bad = list(ok); bad[4] = 0
    assert f(*bad) == 0                                                    # no queries: no work


def test_copy_cache_rows_multi_rejects_bad_arguments(L):
    from indexer_selected_sparse_block_gb300._binding import _RowCopy, SFA_MAX_ROW_COPIES
    f = L.sfa_copy_cache_rows_multi
    ok = _RowCopy(0x10000, 2048, 0x20000, 1152, 1152, 32)
    bad = _RowCopy(0x10000, 1024, 0x20000, 1152, 1152, 32)       # dst rows overlap
    arr = (_RowCopy * 2)(ok, bad)
    assert f(2, ctypes.cast(arr, ctypes.c_void_p), None) == 1
    assert f(1, None, None) == 1                                  # no list
    assert f(-1, None, None) == 1
    assert f(SFA_MAX_ROW_COPIES + 1, ctypes.cast(arr, ctypes.c_void_p), None) == 1
    assert f(0, None, None) == 0                                  # nothing to copy
    empty = (_RowCopy * 1)(_RowCopy(None, 16, None, 16, 16, 0))
    assert f(1, ctypes.cast(empty, ctypes.c_void_p), None) == 0   # zero rows: skipped


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No CPU fallback: with libsfa.so absent, the first entry-point call raises."""
    import indexer_selected_sparse_block_gb300 as sfa
    from indexer_selected_sparse_block_gb300 import _binding as B
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "libsfa.so"))
    with pytest.raises(RuntimeError, match="not built"):
        sfa.sfa_attend_workspace_bytes(1, 16, 1, 512, 2051)
