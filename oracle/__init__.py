"""Parity oracle for indexer-selected block-sparse attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
this package.  The product library never loads it and shares no code with it.

This module only marshals numpy arrays into the plain-C oracle (``sfa_oracle.c``), which
computes every step in double precision straight from the definition of the method in
the pages (llama.cpp commit "model: add Qwen3.8-Flash-Next (qwen4exp)", QSA indexer
paragraphs; llama.cpp PR #27970 "CUDA + ggml: add sparse-fa for DSV4/GLM").  None of the
method's arithmetic lives here.

Pins: every function is checked against closed forms, brute force, invariants and library
routines by ``tests/test_oracle_pins.py`` (no function is left "parity unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sfa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libsfa_oracle.so")
_lib = None

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_i8p = np.ctypeslib.ndpointer(dtype=np.int8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle with gcc (IEEE double, no FMA contraction, no fast-math)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", out, src, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and type the oracle library."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    lib.sfa_oracle_pool.argtypes = [_f32p, _i64, _int, _int, _f64p]
    lib.sfa_oracle_pool_cells.argtypes = [_f32p, _i64, _i32p, _i64, _int, _int, _f64p]
    lib.sfa_oracle_pool_cells.restype = _int
    lib.sfa_oracle_quantize_q8_0.argtypes = [_f32p, _i64, _int, _i8p, _u16p]
    lib.sfa_oracle_quantize_q8_0.restype = _int
    lib.sfa_oracle_dequantize_q8_0.argtypes = [_i8p, _u16p, _i64, _int, _f32p]
    lib.sfa_oracle_fp16_bits.argtypes = [_f32p, _i64, _u16p]
    lib.sfa_oracle_key_transform.argtypes = [_f64p, _i64, _int, _int, _int, _f32p, _f32p,
                                             ctypes.c_double, _int, ctypes.c_double, _int, _i64]
    lib.sfa_oracle_index_scores.argtypes = [_f32p, _f32p, _int, _int, _f64p, _i64, _f64p]
    lib.sfa_oracle_select.argtypes = [_f64p, _i64, _int, _i32p]
    lib.sfa_oracle_select.restype = _int
    lib.sfa_oracle_mask.argtypes = [_i64, _int, _vp, _int, _int, _u8p]
    lib.sfa_oracle_mask_window.argtypes = [_i64, _int, _vp, _int, _i64, _u8p]
    lib.sfa_oracle_attend.argtypes = [_f32p, _int, _int, _int, _int, ctypes.c_double, _f32p,
                                      _i64, _vp, _i64, _vp, _u8p, _i64, _f64p, _vp]
    lib.sfa_oracle_run.argtypes = [_f32p, _f32p, _f32p, _f32p, _f32p, _vp, _i32p, _i32p,
                                   _int, _int, _int, _int, _int, _int, _int, _int, _int, _int,
                                   ctypes.c_double, _i32p, _i32p, _vp, _i64, _f64p, _f64p, _int]
    if path is None:
        _lib = lib
    return lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def pool(X, n_blk: int, cr: int, lib=None) -> np.ndarray:
    """Block means of one sequence's raw index keys X[n_tok][d_idx] -> [n_blk][d_idx] f64."""
    lib = lib or load()
    X = _f32(X)
    assert n_blk * cr <= X.shape[0]
    out = np.zeros((n_blk, X.shape[1]), np.float64)
    lib.sfa_oracle_pool(X, n_blk, X.shape[1], cr, out)
    return out


def pool_cells(X, cell_of, n_blk: int, cr: int, lib=None) -> np.ndarray:
    """Block means in the paged layout: X[n_cells][d_idx] is the flat cell array and
    cell_of[t] the cell of position t of one sequence -> [n_blk][d_idx] f64."""
    lib = lib or load()
    X = _f32(X)
    cell_of = np.ascontiguousarray(cell_of, dtype=np.int32)
    assert n_blk * cr <= cell_of.shape[0]
    out = np.zeros((n_blk, X.shape[1]), np.float64)
    if lib.sfa_oracle_pool_cells(X, X.shape[0], cell_of, n_blk, X.shape[1], cr, out) != 0:
        raise ValueError("a cell map entry lies outside the cell array")
    return out


def quantize_q8_0(x, lib=None):
    """q8_0 blocks of the rows of x[..., d] (d a multiple of 32): (codes int8 [..., d],
    binary16 scale bits uint16 [..., d/32])."""
    lib = lib or load()
    x = _f32(x)
    d = x.shape[-1]
    assert d % 32 == 0
    rows = x.reshape(-1, d)
    q = np.zeros(rows.shape, np.int8)
    s = np.zeros((rows.shape[0], d // 32), np.uint16)
    if lib.sfa_oracle_quantize_q8_0(rows, rows.shape[0], d, q, s) != 0:
        raise ValueError("a q8_0 scale overflows binary16")
    return q.reshape(x.shape), s.reshape(x.shape[:-1] + (d // 32,))


def dequantize_q8_0(q, scale, lib=None) -> np.ndarray:
    """The values q8_0 codes stand for (float32 [..., d], exact)."""
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    d = q.shape[-1]
    scale = np.ascontiguousarray(scale, dtype=np.uint16)
    out = np.zeros(q.shape, np.float32)
    lib.sfa_oracle_dequantize_q8_0(q.reshape(-1, d), scale.reshape(-1, d // 32),
                                   q.size // d if d else 0, d, out.reshape(-1, d))
    return out


def fp16_bits(x, lib=None) -> np.ndarray:
    """binary16 bits of each element of x (round to nearest, ties to even)."""
    lib = lib or load()
    x = _f32(x).reshape(-1)
    out = np.zeros(x.shape, np.uint16)
    lib.sfa_oracle_fp16_bits(x, x.shape[0], out)
    return out


def key_transform(kbar, cr: int, *, norm: int = 0, gamma=None, beta=None, eps: float = 1e-6,
                  n_rot: int = 0, rope_base: float = 10000.0, rope_neox: bool = True,
                  pos_offset: int = 0, lib=None) -> np.ndarray:
    """The pooled keys kbar[n_blk][d_idx] after the norm (0 none, 1 RMS, 2 layer) and the
    rotation of their first n_rot dims at positions b*cr + pos_offset (a new array)."""
    lib = lib or load()
    out = np.array(kbar, dtype=np.float64, order="C", copy=True)
    d = out.shape[1]
    g = _f32(np.ones(d) if gamma is None else gamma)
    bt = _f32(np.zeros(d) if beta is None else beta)
    lib.sfa_oracle_key_transform(out, out.shape[0], d, cr, norm, g, bt, eps, n_rot, rope_base,
                                 int(rope_neox), pos_offset)
    return out


def index_scores(q_idx, w, kbar, lib=None) -> np.ndarray:
    """Scores of every pooled key kbar[n_blk][d_idx] for one query (q_idx[h][d], w[h])."""
    lib = lib or load()
    q_idx, w = _f32(q_idx), _f32(w)
    kbar = np.ascontiguousarray(kbar, dtype=np.float64)
    out = np.zeros(kbar.shape[0], np.float64)
    lib.sfa_oracle_index_scores(q_idx, w, q_idx.shape[0], q_idx.shape[1], kbar, kbar.shape[0],
                                out)
    return out


def select(score, top_k: int, lib=None):
    """(sel[top_k] ascending, -1 padded; n_sel) for one query's block scores."""
    lib = lib or load()
    score = np.ascontiguousarray(score, dtype=np.float64)
    sel = np.full(top_k, -7, np.int32)
    n = lib.sfa_oracle_select(score, score.shape[0], top_k, sel)
    return sel, int(n)


def mask(p: int, cr: int, sel=None, n_sel: int = 0, dense: bool = False, window: int = 0,
         lib=None):
    """Attended-set mask over positions 0..p (uint8[p+1]); window > 0: the set joined with
    the `window` most recent positions (the dense-window + sparse variant)."""
    lib = lib or load()
    out = np.zeros(p + 1, np.uint8)
    sel_arr = None if sel is None else np.ascontiguousarray(sel, dtype=np.int32)
    ptr = None if sel_arr is None else sel_arr.ctypes.data
    if window > 0 and not dense:
        lib.sfa_oracle_mask_window(p, cr, ptr, n_sel, window, out)
    else:
        lib.sfa_oracle_mask(p, cr, ptr, n_sel, 1 if dense else 0, out)
    return out


def attend(q, K, V, msk, scale: float, h_kv: int, dv: int | None = None, tok_row=None,
           lib=None):
    """Exact attention of one query q[h_q][dkq] over the masked tokens.

    K is [n_rows][h_kv][dkq]; V is [n_rows][h_kv][dv], or None for V = K[..., :dv];
    token t reads row t, or row tok_row[t] when tok_row is given.
    Returns (O[h_q][dv] f64, lse[h_q] f64).
    """
    lib = lib or load()
    q, K = _f32(q), _f32(K)
    h_q, dkq = q.shape
    if V is None:
        assert dv is not None and dv <= dkq
        Vp, v_stride = None, 0
    else:
        V = _f32(V)
        dv = V.shape[-1]
        Vp, v_stride = V.ctypes.data, h_kv * dv
    msk = np.ascontiguousarray(msk, dtype=np.uint8)
    rows = None if tok_row is None else np.ascontiguousarray(tok_row, dtype=np.int64)
    O = np.zeros((h_q, dv), np.float64)
    lse = np.zeros(h_q, np.float64)
    lib.sfa_oracle_attend(q, h_q, h_kv, dkq, dv, float(scale), K, h_kv * dkq, Vp, v_stride,
                          None if rows is None else rows.ctypes.data, msk, msk.shape[0], O,
                          lse.ctypes.data)
    return O, lse


def run(X, q_idx, w, Q, K, V, q_seq, q_pos, *, cr: int, top_k: int, scale: float,
        dv: int | None = None, want_scores: bool = False, n_threads: int | None = None,
        lib=None) -> dict:
    """The whole method for a batch of queries (threads over queries).

    X[n_seq][n_tok][d_idx], q_idx[n_q][h_idx][d_idx], w[n_q][h_idx], Q[n_q][h_q][dkq],
    K[n_seq][n_tok][h_kv][dkq], V[n_seq][n_tok][h_kv][dv] or None.  top_k <= 0: dense.
    """
    lib = lib or load()
    X, q_idx, w, Q, K = _f32(X), _f32(q_idx), _f32(w), _f32(Q), _f32(K)
    q_seq = np.ascontiguousarray(q_seq, dtype=np.int32)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int32)
    n_seq, n_tok, d_idx = X.shape
    n_q, h_idx, _ = q_idx.shape
    _, h_q, dkq = Q.shape
    h_kv = K.shape[2]
    assert K.shape[:2] == (n_seq, n_tok)
    if V is not None:
        V = _f32(V)
        dv = V.shape[-1]
    assert dv is not None and (V is not None or dv <= dkq)
    kk = max(top_k, 1)
    sel = np.full((n_q, kk), -7, np.int32)
    n_sel = np.zeros(n_q, np.int32)
    max_blk = int(q_pos.max() + 1) // cr + 1 if n_q else 1
    score = np.full((n_q, max_blk), np.nan, np.float64) if want_scores else None
    O = np.zeros((n_q, h_q, dv), np.float64)
    lse = np.zeros((n_q, h_q), np.float64)
    n_threads = n_threads or os.cpu_count() or 1
    lib.sfa_oracle_run(X, q_idx, w, Q, K, None if V is None else V.ctypes.data, q_seq, q_pos,
                       n_q, n_tok, h_idx, d_idx, cr, top_k, h_q, h_kv, dkq, dv, float(scale),
                       sel, n_sel, None if score is None else score.ctypes.data, max_blk, O,
                       lse, int(n_threads))
    out = {"O": O, "lse": lse, "threads": min(int(n_threads), max(n_q, 1))}
    if top_k > 0:
        out["sel"] = sel
        out["n_sel"] = n_sel
        if want_scores:
            out["score"] = score
    return out
