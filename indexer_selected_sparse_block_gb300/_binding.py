"""ctypes binding of libsfa (the C ABI in include/sfa.h).

Argument marshalling only: every step of the method runs in libsfa's CUDA kernels.  Tensors
are torch CUDA tensors (torch provides device memory and streams); each function passes
their raw pointers, sizes and the current stream to the C entry point of the same name and
raises ``SfaError`` on a non-zero status.  There is no CPU fallback: if libsfa.so is not
built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsfa.so")

SFA_OK, SFA_ERR_INVALID_ARG, SFA_ERR_UNSUPPORTED, SFA_ERR_CUDA, SFA_ERR_WORKSPACE = range(5)
SFA_BF16, SFA_F32, SFA_Q8_0 = 0, 1, 2
SFA_DEV_BAD_BLOCK, SFA_DEV_BAD_NSEL, SFA_DEV_BAD_QUERY, SFA_DEV_TIMEOUT = 1, 2, 4, 8
SFA_DEV_BAD_CELL, SFA_DEV_FP16_RANGE = 16, 32
SFA_PART_ALL, SFA_PART_SELECTED, SFA_PART_WINDOW = 0, 1, 2
SFA_REFINE_MAX_BLOCKS = 131072  # longest row sfa_topk_blocks_refine takes

_lib = None
_vp, _i64, _int, _f32, _sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                              ctypes.c_size_t)

class _RowCopy(ctypes.Structure):
    """sfa_row_copy of include/sfa.h."""
    _fields_ = [("dst", ctypes.c_void_p), ("dst_pitch", ctypes.c_int64),
                ("src", ctypes.c_void_p), ("src_pitch", ctypes.c_int64),
                ("row_bytes", ctypes.c_int64), ("n_rows", ctypes.c_int64)]


SFA_MAX_ROW_COPIES = 8

# name -> (restype, argtypes); mirrors include/sfa.h
SIGNATURES = {
    "sfa_pool_index_keys": (_int, [_vp, _int, _i64, _int, _int, _int, _i64, _i64, _vp, _i64, _vp,
                                   _i64, _vp]),
    "sfa_pool_index_keys_transformed": (_int, [_vp, _int, _i64, _int, _int, _int, _i64, _i64,
                                               _int, _vp, _vp, _f32, _int, _f32, _int, _i64,
                                               _vp, _i64, _vp, _i64, _vp]),
    "sfa_pool_index_keys_paged": (_int, [_vp, _int, _i64, _vp, _i64, _int, _int, _int, _i64,
                                         _i64, _vp, _i64, _vp, _i64, _vp, _vp]),
    "sfa_index_scores": (_int, [_vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _vp, _i64,
                                _int, _i64, _vp, _i64, _vp, _vp]),
    "sfa_index_scores_bounded": (_int, [_vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _vp,
                                        _i64, _vp, _i64, _int, _i64, _vp, _vp, _i64, _vp, _vp]),
    "sfa_quantize_pooled_keys_i8": (_int, [_vp, _i64, _int, _int, _i64, _i64, _vp, _i64, _vp,
                                           _i64, _vp]),
    "sfa_index_scores_bounded_i8": (_int, [_vp, _vp, _vp, _vp, _int, _int, _int, _int, _vp, _i64,
                                           _vp, _i64, _int, _i64, _vp, _vp, _i64, _vp, _vp]),
    "sfa_topk_workspace_bytes": (_sz, [_int, _i64, _int]),
    "sfa_attend_plan": (_int, [_int, _int, _int, _int, _int, _i64, _int, _int, _vp, _vp]),
    "sfa_topk_refine_workspace_bytes": (_sz, [_int, _i64]),
    "sfa_topk_blocks_refine": (_int, [_vp, _vp, _i64, _vp, _vp, _vp, _vp, _int, _int, _int, _vp,
                                      _i64, _int, _int, _int, _i64, _vp, _vp, _vp, _sz, _vp,
                                      _vp]),
    "sfa_topk_blocks": (_int, [_vp, _i64, _vp, _int, _int, _int, _i64, _vp, _vp, _vp, _sz, _vp,
                               _vp]),
    "sfa_attend_workspace_bytes": (_sz, [_int, _int, _int, _int, _i64]),
    "sfa_gather_attend": (_int, [_vp, _vp, _vp, _int, _int, _i64, _int, _int, _int, _int, _int,
                                 _f32, _vp, _vp, _vp, _vp, _int, _int, _vp, _vp, _vp, _sz, _vp,
                                 _vp]),
    "sfa_dense_attend": (_int, [_vp, _vp, _vp, _int, _int, _i64, _int, _int, _int, _int, _int,
                                _f32, _vp, _vp, _i64, _vp, _vp, _vp, _sz, _vp, _vp]),
    "sfa_window_kv_max": (_i64, [_int, _int, _i64, _int]),
    "sfa_gather_attend_window": (_int, [_vp, _vp, _vp, _int, _int, _i64, _int, _int, _int, _int,
                                        _int, _f32, _vp, _vp, _vp, _vp, _int, _int, _i64, _int,
                                        _vp, _vp, _vp, _sz, _vp, _vp]),
    "sfa_combine_attention": (_int, [_vp, _vp, _vp, _vp, _i64, _int, _vp, _vp, _vp]),
    "sfa_gather_kv_bandwidth": (_int, [_vp, _vp, _int, _i64, _int, _int, _int, _int, _vp, _vp, _vp,
                                       _vp, _int, _int, _vp, _vp, _vp]),
    "sfa_gather_attend_noalloc": (_int, [_vp, _vp, _vp, _int, _int, _i64, _int, _int, _int,
                                         _int, _int, _f32, _vp, _vp, _vp, _vp, _int, _int, _vp,
                                         _vp, _vp, _vp]),
    "sfa_gather_attend_paged": (_int, [_vp, _vp, _vp, _int, _i64, _vp, _int, _i64, _int, _int,
                                       _int, _int, _int, _f32, _vp, _vp, _vp, _vp, _int, _int,
                                       _vp, _vp, _vp, _sz, _vp, _vp]),
    "sfa_dense_attend_paged": (_int, [_vp, _vp, _vp, _int, _i64, _vp, _int, _i64, _int, _int,
                                      _int, _int, _int, _f32, _vp, _vp, _i64, _vp, _vp, _vp, _sz,
                                      _vp, _vp]),
    "sfa_q8_0_row_bytes": (_sz, [_int]),
    "sfa_quantize_kv_q8_0": (_int, [_vp, _int, _i64, _i64, _int, _i64, _vp, _i64, _vp, _vp]),
    "sfa_copy_cache_rows": (_int, [_vp, _i64, _vp, _i64, _i64, _i64, _vp]),
    "sfa_copy_cache_rows_multi": (_int, [_int, _vp, _vp]),
    "sfa_read_device_status": (_int, [_vp, _vp, _vp]),
    "sfa_status_string": (ctypes.c_char_p, [_int]),
}


class SfaError(RuntimeError):
    """A non-zero status returned by libsfa."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {lib().sfa_status_string(status).decode()}")


def lib(path: str | None = None):
    """Loads libsfa.so (built by ``__graft_entry__.build()``); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libsfa.so is not built ({p}); run __graft_entry__.build() first")
    L = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    if path is None:
        _lib = L
    return L


def _p(t, strided=False):
    """Device pointer of t; strided=True when the caller passes t's strides to the library."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libsfa takes CUDA tensors only")
    if not strided and not t.is_contiguous():
        raise ValueError("libsfa takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _p_out(t):
    """Pointer of an attention output: a CUDA tensor, or a page-locked host tensor that the
    device writes directly."""
    if t is not None and not t.is_cuda:
        if not t.is_pinned():
            raise ValueError("an attention output on the host must be in page-locked memory")
        if not t.is_contiguous():
            raise ValueError("libsfa takes contiguous tensors only")
        return ctypes.c_void_p(t.data_ptr())
    return _p(t)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, rc: int):
    if rc != SFA_OK:
        raise SfaError(fn, rc)


def _dtype_code(t) -> int:
    if t.dtype == torch.bfloat16:
        return SFA_BF16
    if t.dtype == torch.float32:
        return SFA_F32
    if t.dtype == torch.uint8:   # q8_0 cache rows
        return SFA_Q8_0
    raise ValueError(f"unsupported dtype {t.dtype}")


def kbar_shape(n_seq: int, blk_cap: int, d_idx: int):
    """Shape of the pooled-key table: [n_seq][blk_cap][2*d_idx] bf16 (hi, lo halves)."""
    return (n_seq, blk_cap, 2 * d_idx)


def sfa_pool_index_keys(X, compress_ratio: int, blk_begin: int, blk_end: int, Kbar,
                        Kbar_r=None, stream=None):
    """X [n_seq][n_tok_cap][d_idx] (bf16/f32) -> rows [blk_begin, blk_end) of Kbar, and of the
    bound factors Kbar_r [n_seq][blk_cap] fp32 when given."""
    n_seq, _, d_idx = X.shape
    rc = lib().sfa_pool_index_keys(_p(X), _dtype_code(X), X.stride(0), n_seq, d_idx,
                                   compress_ratio, blk_begin, blk_end, _p(Kbar), Kbar.stride(0),
                                   _p(Kbar_r), Kbar_r.stride(0) if Kbar_r is not None else 0,
                                   _stream(stream))
    _check("sfa_pool_index_keys", rc)


def sfa_pool_index_keys_transformed(X, compress_ratio: int, blk_begin: int, blk_end: int, Kbar,
                                    Kbar_r=None, *, norm: int = 0, gamma=None, beta=None,
                                    eps: float = 1e-6, n_rot: int = 0, rope_base: float = 10000.0,
                                    rope_neox: bool = True, pos_offset: int = 0, stream=None):
    """sfa_pool_index_keys with the pooled key normalised (norm 0 none, 1 RMS, 2 layer; gamma,
    beta [d_idx] fp32 on the device) and its first n_rot dims rotated at b*cr + pos_offset."""
    n_seq, _, d_idx = X.shape
    rc = lib().sfa_pool_index_keys_transformed(
        _p(X), _dtype_code(X), X.stride(0), n_seq, d_idx, compress_ratio, blk_begin, blk_end,
        norm, _p(gamma), _p(beta), eps, n_rot, rope_base, int(rope_neox), pos_offset, _p(Kbar),
        Kbar.stride(0), _p(Kbar_r), Kbar_r.stride(0) if Kbar_r is not None else 0,
        _stream(stream))
    _check("sfa_pool_index_keys_transformed", rc)


def sfa_index_scores(q_idx, w, q_seq, q_pos, Kbar, compress_ratio: int, n_blk_max: int, scores,
                     q_group: int = 1, dev_status=None, stream=None):
    """scores[i][b] = sum_j w[i][j] * relu(q_idx[i][j] . kbar_b) for b < B_i."""
    n_q, h_idx, d_idx = q_idx.shape
    rc = lib().sfa_index_scores(_p(q_idx), _p(w), _p(q_seq), _p(q_pos), n_q, q_group, h_idx,
                                d_idx, compress_ratio, _p(Kbar), Kbar.stride(0), Kbar.shape[0],
                                n_blk_max, _p(scores), scores.stride(0), _p(dev_status),
                                _stream(stream))
    _check("sfa_index_scores", rc)


def sfa_index_scores_bounded(q_idx, w, q_seq, q_pos, Kbar, Kbar_r, compress_ratio: int,
                             n_blk_max: int, lower, upper, q_group: int = 1, dev_status=None,
                             stream=None):
    """lower[i][b] <= s_ib <= upper[i][b] for the hi + lo score s_ib, from the hi halves of the
    pooled keys and their bound factors Kbar_r only."""
    n_q, h_idx, d_idx = q_idx.shape
    if lower.stride(0) != upper.stride(0):
        raise ValueError("lower and upper must share a row stride")
    rc = lib().sfa_index_scores_bounded(_p(q_idx), _p(w), _p(q_seq), _p(q_pos), n_q, q_group,
                                        h_idx, d_idx, compress_ratio, _p(Kbar), Kbar.stride(0),
                                        _p(Kbar_r), Kbar_r.stride(0), Kbar.shape[0], n_blk_max,
                                        _p(lower), _p(upper), lower.stride(0), _p(dev_status),
                                        _stream(stream))
    _check("sfa_index_scores_bounded", rc)


def k8_shapes(n_seq: int, blk_cap: int, d_idx: int):
    """Shapes of the 8-bit pooled-key copy: codes [n_seq][blk_cap][d_idx] (int8 storage of the
    bytes c + 128) and (scale, bound factor) pairs [n_seq][blk_cap][2] fp32."""
    return (n_seq, blk_cap, d_idx), (n_seq, blk_cap, 2)


def sfa_quantize_pooled_keys_i8(Kbar, blk_begin: int, blk_end: int, K8, K8_sr, stream=None):
    """Rows [blk_begin, blk_end) of the 8-bit copy (K8 codes, K8_sr scale and bound factor) of
    the pooled keys m = hi + lo in Kbar."""
    n_seq, _, two_d = Kbar.shape
    if K8.dtype != torch.int8 or K8_sr.dtype != torch.float32:
        raise ValueError("K8 must be int8 and K8_sr float32")
    rc = lib().sfa_quantize_pooled_keys_i8(_p(Kbar), Kbar.stride(0), n_seq, two_d // 2,
                                           blk_begin, blk_end, _p(K8), K8.stride(0), _p(K8_sr),
                                           K8_sr.stride(0), _stream(stream))
    _check("sfa_quantize_pooled_keys_i8", rc)


def sfa_index_scores_bounded_i8(q_idx, w, q_seq, q_pos, K8, K8_sr, compress_ratio: int,
                                n_blk_max: int, lower, upper, dev_status=None, stream=None):
    """lower[i][b] <= s_ib <= upper[i][b] for the hi + lo score s_ib, from the 8-bit copy of the
    pooled keys (sfa_quantize_pooled_keys_i8)."""
    n_q, h_idx, d_idx = q_idx.shape
    if lower.stride(0) != upper.stride(0):
        raise ValueError("lower and upper must share a row stride")
    rc = lib().sfa_index_scores_bounded_i8(_p(q_idx), _p(w), _p(q_seq), _p(q_pos), n_q, h_idx,
                                           d_idx, compress_ratio, _p(K8), K8.stride(0),
                                           _p(K8_sr), K8_sr.stride(0), K8.shape[0], n_blk_max,
                                           _p(lower), _p(upper), lower.stride(0),
                                           _p(dev_status), _stream(stream))
    _check("sfa_index_scores_bounded_i8", rc)


def sfa_topk_refine_workspace_bytes(n_q: int, n_blk_max: int) -> int:
    return int(lib().sfa_topk_refine_workspace_bytes(n_q, n_blk_max))


def sfa_topk_blocks_refine(lower, upper, q_idx, w, q_seq, q_pos, Kbar, compress_ratio: int,
                           top_k: int, n_blk_max: int, blk_idx, n_sel, workspace=None,
                           dev_status=None, stream=None):
    """The top_k best blocks by the hi + lo score, from its lower and upper bounds: only the
    blocks the bounds cannot rule out are rescored."""
    n_q, h_idx, d_idx = q_idx.shape
    need = sfa_topk_refine_workspace_bytes(n_q, n_blk_max)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_pos.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().sfa_topk_blocks_refine(_p(lower), _p(upper), lower.stride(0), _p(q_idx), _p(w),
                                      _p(q_seq), _p(q_pos), n_q, h_idx, d_idx, _p(Kbar),
                                      Kbar.stride(0), Kbar.shape[0], compress_ratio, top_k,
                                      n_blk_max, _p(blk_idx), _p(n_sel), _p(workspace),
                                      ws_bytes, _p(dev_status), _stream(stream))
    _check("sfa_topk_blocks_refine", rc)


def sfa_topk_workspace_bytes(n_q: int, n_blk_max: int, top_k: int) -> int:
    return int(lib().sfa_topk_workspace_bytes(n_q, n_blk_max, top_k))


def sfa_topk_blocks(scores, q_pos, compress_ratio: int, top_k: int, n_blk_max: int, blk_idx,
                    n_sel, workspace=None, dev_status=None, stream=None):
    """The top_k best blocks of each query (ascending, -1 padded) and their count.  scores may
    be a view whose rows are apart (score_stride = scores.stride(0)); each row contiguous."""
    if scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be [n_q][>= n_blk_max] with contiguous rows")
    n_q = q_pos.shape[0]
    need = sfa_topk_workspace_bytes(n_q, n_blk_max, top_k)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_pos.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().sfa_topk_blocks(_p(scores, strided=True), scores.stride(0), _p(q_pos), n_q,
                               compress_ratio,
                               top_k, n_blk_max, _p(blk_idx), _p(n_sel), _p(workspace),
                               ws_bytes, _p(dev_status), _stream(stream))
    _check("sfa_topk_blocks", rc)


def sfa_attend_workspace_bytes(n_q: int, h_q: int, h_kv: int, dv: int, n_kv_max: int) -> int:
    return int(lib().sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv_max))


def sfa_attend_plan(dtype_code: int, n_q: int, h_kv: int, dkq: int, has_v: bool, n_kv_max: int,
                    compress_ratio: int, dense: bool = False):
    """(n_split, kernels): CTAs per (query, KV head) list and kernels one attention call
    launches on the current device."""
    ns, nk = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().sfa_attend_plan(dtype_code, n_q, h_kv, dkq, int(has_v), n_kv_max, compress_ratio,
                               int(dense), ctypes.byref(ns), ctypes.byref(nk))
    _check("sfa_attend_plan", rc)
    return ns.value, nk.value


def _check_qkv(Q, K, V):
    if V is not None and K.dtype != V.dtype:
        raise ValueError("K and V must share a dtype")
    if K.dtype == torch.uint8:   # q8_0 cache rows: Q stays bf16
        if Q.dtype != torch.bfloat16:
            raise ValueError("a q8_0 cache takes a bf16 Q")
    elif Q.dtype != K.dtype:
        raise ValueError("Q and K must share a dtype")


def _attn_dims(Q, K, V, O):
    n_q, h_q, dkq = Q.shape
    n_seq, n_tok_cap, h_kv, _ = K.shape
    dv = O.shape[-1]
    _check_qkv(Q, K, V)
    return n_q, h_q, dkq, n_seq, n_tok_cap, h_kv, dv


def sfa_gather_attend(Q, K, V, q_seq, q_pos, blk_idx, n_sel, top_k: int, compress_ratio: int,
                      scale: float, O, lse=None, workspace=None, dev_status=None, stream=None):
    """Attention of each query over its kept blocks plus its tail."""
    n_q, h_q, dkq, n_seq, n_tok_cap, h_kv, dv = _attn_dims(Q, K, V, O)
    n_kv_max = top_k * compress_ratio + compress_ratio - 1
    need = sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv_max)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().sfa_gather_attend(_p(Q), _p(K), _p(V), _dtype_code(K), n_seq, n_tok_cap, n_q, h_q,
                                 h_kv, dkq, dv, float(scale), _p(q_seq), _p(q_pos), _p(blk_idx),
                                 _p(n_sel), top_k, compress_ratio, _p_out(O), _p_out(lse),
                                 _p(workspace), ws_bytes, _p(dev_status), _stream(stream))
    _check("sfa_gather_attend", rc)


def sfa_window_kv_max(top_k: int, compress_ratio: int, window: int, part: int = 0) -> int:
    return int(lib().sfa_window_kv_max(top_k, compress_ratio, window, part))


def sfa_gather_attend_window(Q, K, V, q_seq, q_pos, blk_idx, n_sel, top_k: int,
                             compress_ratio: int, window: int, scale: float, O, lse=None,
                             part: int = SFA_PART_ALL, workspace=None, dev_status=None,
                             stream=None):
    """Attention over the kept blocks, the tail and a dense window of the `window` most recent
    positions (part: the whole set, its kept part before the window, or the window suffix)."""
    n_q, h_q, dkq, n_seq, n_tok_cap, h_kv, dv = _attn_dims(Q, K, V, O)
    n_kv_max = sfa_window_kv_max(top_k, compress_ratio, window, part)
    need = sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv_max)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().sfa_gather_attend_window(_p(Q), _p(K), _p(V), _dtype_code(K), n_seq, n_tok_cap,
                                        n_q, h_q, h_kv, dkq, dv, float(scale), _p(q_seq),
                                        _p(q_pos), _p(blk_idx), _p(n_sel), top_k,
                                        compress_ratio, int(window), int(part), _p_out(O),
                                        _p_out(lse), _p(workspace), ws_bytes, _p(dev_status),
                                        _stream(stream))
    _check("sfa_gather_attend_window", rc)


def sfa_combine_attention(O_a, lse_a, O_b, lse_b, O, lse, stream=None):
    """O, lse = the attention over the union of two disjoint key sets, from each set's (O, lse)
    ([rows][dv] and [rows] fp32; O / lse may be either input)."""
    dv = O.shape[-1]
    n_rows = O.numel() // dv
    for t in (O_a, O_b, O):
        if t.numel() != n_rows * dv or not t.is_contiguous() or t.dtype != torch.float32:
            raise ValueError("O_a, O_b, O must be contiguous fp32 tensors of one shape")
    for t in (lse_a, lse_b, lse):
        if t.numel() != n_rows or not t.is_contiguous() or t.dtype != torch.float32:
            raise ValueError("lse_a, lse_b, lse must be contiguous fp32 tensors of O's rows")
    rc = lib().sfa_combine_attention(_p(O_a), _p(lse_a), _p(O_b), _p(lse_b), n_rows, dv, _p_out(O),
                                     _p_out(lse), _stream(stream))
    _check("sfa_combine_attention", rc)


def sfa_gather_kv_bandwidth(K, V, q_seq, q_pos, blk_idx, n_sel, top_k: int, compress_ratio: int,
                            dkq: int, dv: int, checksum, dev_status=None, stream=None):
    """A measurement: the K/V rows sfa_gather_attend would attend, moved into shared memory
    and nothing else (its time is the attention's data-movement ceiling on these lists)."""
    n_seq, n_tok_cap, h_kv = K.shape[0], K.shape[1], K.shape[2]
    rc = lib().sfa_gather_kv_bandwidth(_p(K), _p(V), n_seq, n_tok_cap, q_seq.numel(), h_kv, dkq,
                                       dv, _p(q_seq), _p(q_pos), _p(blk_idx), _p(n_sel), top_k,
                                       compress_ratio, _p(checksum), _p(dev_status),
                                       _stream(stream))
    _check("sfa_gather_kv_bandwidth", rc)


def sfa_gather_attend_noalloc(Q, K, V, q_seq, q_pos, blk_idx, n_sel, top_k: int,
                              compress_ratio: int, scale: float, O, lse=None, dev_status=None,
                              stream=None):
    """sfa_gather_attend without a workspace: for callers that cannot allocate device memory
    when they call (their split-KV scratch is a fixed 16 MiB array inside libsfa, shared by
    every call on the device; overlapping calls on the GPU race on it)."""
    n_q, h_q, dkq, n_seq, n_tok_cap, h_kv, dv = _attn_dims(Q, K, V, O)
    rc = lib().sfa_gather_attend_noalloc(_p(Q), _p(K), _p(V), _dtype_code(K), n_seq, n_tok_cap,
                                         n_q, h_q, h_kv, dkq, dv, float(scale), _p(q_seq),
                                         _p(q_pos), _p(blk_idx), _p(n_sel), top_k,
                                         compress_ratio, _p_out(O), _p_out(lse), _p(dev_status),
                                         _stream(stream))
    _check("sfa_gather_attend_noalloc", rc)


def sfa_dense_attend(Q, K, V, q_seq, q_pos, n_kv_max: int, scale: float, O, lse=None,
                     workspace=None, dev_status=None, stream=None):
    """Causal attention of each query over all of its sequence's tokens 0..p_i."""
    n_q, h_q, dkq, n_seq, n_tok_cap, h_kv, dv = _attn_dims(Q, K, V, O)
    need = sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv_max)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().sfa_dense_attend(_p(Q), _p(K), _p(V), _dtype_code(K), n_seq, n_tok_cap, n_q, h_q,
                                h_kv, dkq, dv, float(scale), _p(q_seq), _p(q_pos), n_kv_max,
                                _p_out(O), _p_out(lse), _p(workspace), ws_bytes, _p(dev_status),
                                _stream(stream))
    _check("sfa_dense_attend", rc)


def _paged_dims(cell_of, n_cells_of):
    if cell_of.dtype != torch.int32 or cell_of.dim() != 2 or not cell_of.is_contiguous():
        raise ValueError("cell_of must be a contiguous [n_seq][n_pos_cap] int32 tensor")
    return cell_of.shape[0], cell_of.shape[1], n_cells_of


def sfa_pool_index_keys_paged(X, cell_of, compress_ratio: int, blk_begin: int, blk_end: int, Kbar,
                              Kbar_r=None, dev_status=None, stream=None):
    """Paged layout: X [n_cells][d_idx] raw index keys, one cell per row; position t of
    sequence s is in cell cell_of[s][t].  Writes rows [blk_begin, blk_end) of Kbar (and Kbar_r)
    as sfa_pool_index_keys does for the gathered layout."""
    n_cells, d_idx = X.shape
    n_seq, n_pos_cap, _ = _paged_dims(cell_of, n_cells)
    rc = lib().sfa_pool_index_keys_paged(_p(X), _dtype_code(X), n_cells, _p(cell_of), n_pos_cap,
                                         n_seq, d_idx, compress_ratio, blk_begin, blk_end,
                                         _p(Kbar), Kbar.stride(0), _p(Kbar_r),
                                         Kbar_r.stride(0) if Kbar_r is not None else 0,
                                         _p(dev_status), _stream(stream))
    _check("sfa_pool_index_keys_paged", rc)


def _paged_attn_dims(Q, K, V, O, cell_of):
    n_q, h_q, dkq = Q.shape
    n_cells, h_kv, _ = K.shape
    if V is not None and V.shape[0] != n_cells:
        raise ValueError("V must have K's cell count")
    _check_qkv(Q, K, V)
    n_seq, n_pos_cap, _ = _paged_dims(cell_of, n_cells)
    return n_q, h_q, dkq, n_cells, n_seq, n_pos_cap, h_kv, O.shape[-1]


def sfa_gather_attend_paged(Q, K, V, cell_of, q_seq, q_pos, blk_idx, n_sel, top_k: int,
                            compress_ratio: int, scale: float, O, lse=None, workspace=None,
                            dev_status=None, stream=None):
    """sfa_gather_attend on the paged layout: K [n_cells][h_kv][dkq], V [n_cells][h_kv][dv] or
    None, position t of sequence s in cell cell_of[s][t]."""
    n_q, h_q, dkq, n_cells, n_seq, n_pos_cap, h_kv, dv = _paged_attn_dims(Q, K, V, O, cell_of)
    n_kv_max = top_k * compress_ratio + compress_ratio - 1
    need = sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv_max)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().sfa_gather_attend_paged(_p(Q), _p(K), _p(V), _dtype_code(K), n_cells, _p(cell_of),
                                       n_seq, n_pos_cap, n_q, h_q, h_kv, dkq, dv, float(scale),
                                       _p(q_seq), _p(q_pos), _p(blk_idx), _p(n_sel), top_k,
                                       compress_ratio, _p_out(O), _p_out(lse), _p(workspace),
                                       ws_bytes, _p(dev_status), _stream(stream))
    _check("sfa_gather_attend_paged", rc)


def sfa_dense_attend_paged(Q, K, V, cell_of, q_seq, q_pos, n_kv_max: int, scale: float, O,
                           lse=None, workspace=None, dev_status=None, stream=None):
    """sfa_dense_attend on the paged layout (see sfa_gather_attend_paged)."""
    n_q, h_q, dkq, n_cells, n_seq, n_pos_cap, h_kv, dv = _paged_attn_dims(Q, K, V, O, cell_of)
    need = sfa_attend_workspace_bytes(n_q, h_q, h_kv, dv, n_kv_max)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=Q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().sfa_dense_attend_paged(_p(Q), _p(K), _p(V), _dtype_code(K), n_cells, _p(cell_of),
                                      n_seq, n_pos_cap, n_q, h_q, h_kv, dkq, dv, float(scale),
                                      _p(q_seq), _p(q_pos), n_kv_max, _p_out(O), _p_out(lse),
                                      _p(workspace), ws_bytes, _p(dev_status), _stream(stream))
    _check("sfa_dense_attend_paged", rc)


def sfa_q8_0_row_bytes(d: int) -> int:
    """Bytes of one q8_0 cache row of d elements (codes, binary16 scales, padding to 16)."""
    return int(lib().sfa_q8_0_row_bytes(d))


def sfa_quantize_kv_q8_0(X, Y, dev_status=None, stream=None):
    """q8_0 rows of X [n_outer][n_inner][d] (bf16/f32) into Y [n_outer][n_inner][row_bytes(d)]
    uint8; within an outer index the rows of both are contiguous (a cache slice of new tokens of
    every sequence viewed as [n_seq][tokens * h_kv][d])."""
    n_outer, n_inner, d = X.shape
    rb = sfa_q8_0_row_bytes(d)
    if Y.dtype != torch.uint8 or tuple(Y.shape) != (n_outer, n_inner, rb):
        raise ValueError(f"Y must be uint8 [{n_outer}][{n_inner}][{rb}]")
    if (X.stride(2), Y.stride(2)) != (1, 1) or (n_inner > 1 and (X.stride(1), Y.stride(1)) != (d, rb)):
        raise ValueError("rows must be contiguous within an outer index")
    rc = lib().sfa_quantize_kv_q8_0(_p(X, strided=True), _dtype_code(X), n_outer, n_inner, d,
                                    X.stride(0), _p(Y, strided=True), Y.stride(0), _p(dev_status),
                                    _stream(stream))
    _check("sfa_quantize_kv_q8_0", rc)


def _row_copy(dst, src):
    if tuple(dst.shape) != tuple(src.shape) or dst.dtype != src.dtype or dst.dim() < 1:
        raise ValueError("dst and src must have the same shape and dtype")
    for t in (dst, src):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError("sfa_copy_cache_rows takes CUDA or page-locked host tensors")
        if t.shape[0] > 0 and not t[0].is_contiguous():
            raise ValueError("each row must be contiguous")
    es = dst.element_size()
    n = dst.shape[0]
    row = dst[0].numel() * es if n > 0 else 0
    dp = dst.stride(0) * es if n > 1 else max(row, 1)
    sp = src.stride(0) * es if n > 1 else max(row, 1)
    return _RowCopy(dst.data_ptr(), dp, src.data_ptr(), sp, max(row, 1), n if row else 0)


def sfa_copy_cache_rows_multi(pairs, stream=None) -> None:
    """Several (dst, src) row copies as sfa_copy_cache_rows makes them, in one kernel launch."""
    pairs = list(pairs)
    if len(pairs) > SFA_MAX_ROW_COPIES:
        raise ValueError(f"at most {SFA_MAX_ROW_COPIES} copies per call")
    arr = (_RowCopy * max(len(pairs), 1))(*[_row_copy(d, s) for d, s in pairs])
    rc = lib().sfa_copy_cache_rows_multi(len(pairs), ctypes.cast(arr, ctypes.c_void_p),
                                         _stream(stream))
    _check("sfa_copy_cache_rows_multi", rc)


def sfa_copy_cache_rows(dst, src, stream=None) -> None:
    """Copies the rows of src into the rows of dst (the same shape; dim 0 indexes the rows,
    each row contiguous, rows at any stride): one two-dimensional copy, either side on the
    device or in page-locked host memory.  Typically dst = cache[:, p] for a step's new
    position p of every sequence."""
    if tuple(dst.shape) != tuple(src.shape) or dst.dtype != src.dtype or dst.dim() < 1:
        raise ValueError("dst and src must have the same shape and dtype")
    for t in (dst, src):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError("sfa_copy_cache_rows takes CUDA or page-locked host tensors")
        if t.shape[0] > 0 and not t[0].is_contiguous():
            raise ValueError("each row must be contiguous")
    es = dst.element_size()
    row = dst[0].numel() * es if dst.shape[0] > 0 else 0
    n = dst.shape[0]
    dp = dst.stride(0) * es if n > 1 else row
    sp = src.stride(0) * es if n > 1 else row
    if n == 0 or row == 0:
        return
    rc = lib().sfa_copy_cache_rows(ctypes.c_void_p(dst.data_ptr()), dp,
                                   ctypes.c_void_p(src.data_ptr()), sp, row, n, _stream(stream))
    _check("sfa_copy_cache_rows", rc)


def sfa_read_device_status(dev_status, stream=None) -> int:
    out = ctypes.c_int32(0)
    rc = lib().sfa_read_device_status(_p(dev_status), ctypes.byref(out), _stream(stream))
    _check("sfa_read_device_status", rc)
    return int(out.value)
