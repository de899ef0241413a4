"""Thin ctypes binding of libkvc (C ABI in include/kvc.h).

Functions carry the C names and only marshal arguments: torch tensors become
device pointers, the current torch CUDA stream becomes the cudaStream_t, and
a non-zero status becomes a ``KvcError``.  Every step of the path runs in the
library's CUDA kernels; there is no fallback -- importing this module on a
machine without the built library raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvc.so")

KVC_F32, KVC_BF16 = 0, 1
KVC_SEL_GLOBAL_TOPK, KVC_SEL_THRESHOLD, KVC_SEL_PER_HEAD = 0, 1, 2
MODES = {"global": KVC_SEL_GLOBAL_TOPK, "threshold": KVC_SEL_THRESHOLD,
         "per_head": KVC_SEL_PER_HEAD}

KVC_AGG_SUM, KVC_AGG_MAX = 0, 1
AGGREGATIONS = {"sum": KVC_AGG_SUM, "max": KVC_AGG_MAX}

STATUS = {0: "KVC_OK", -1: "KVC_ERR_INVALID", -2: "KVC_ERR_UNSUPPORTED",
          -3: "KVC_ERR_WORKSPACE", -4: "KVC_ERR_CUDA", -5: "KVC_ERR_TIMEOUT",
          -6: "KVC_ERR_RANGE"}

# symbol -> (restype, argtypes)
_P, _I, _I64, _SZ, _D, _F, _U64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                   ctypes.c_size_t, ctypes.c_double, ctypes.c_float,
                                   ctypes.c_uint64)
SIGNATURES = {
    "kvc_version": (_I, []),
    "kvc_status_string": (ctypes.c_char_p, [_I]),
    "kvc_device_status": (_I, [_P]),
    "kvc_score_attn_workspace": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "kvc_score_attn": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P, _P, _SZ, _P]),
    "kvc_score_attn_agg": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _I, _I, _P, _P, _SZ,
                                _P]),
    "kvc_score_linear": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "kvc_select_workspace": (_SZ, [_I, _I, _I, _I]),
    "kvc_select": (_I, [_P, _I, _I, _I, _I, _D, _F, _P, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "kvc_compact": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _I64, _P, _P, _P]),
    "kvc_select_compact_workspace": (_SZ, [_I, _I, _I, _I]),
    "kvc_select_compact": (_I, [_P, _I, _I, _I, _I, _D, _F, _P, _I, _I, _P, _P, _I, _I, _I, _P,
                                _P, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "kvc_decode_workspace": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "kvc_decode_attn": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                             _P, _SZ, _P]),
    "kvc_quantize_rows": (_I, [_P, _I, _I64, _I, _P, _P, _P]),
    "kvc_decode_attn_q8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F,
                                _P, _P, _P, _SZ, _P]),
    "kvc_score_kvzip_plus_workspace": (_SZ, [_I, _I, _I, _I, _I]),
    "kvc_score_kvzip_plus": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P,
                                  _P, _SZ, _P]),
    "kvc_score_mlp_workspace": (_SZ, [_I, _I]),
    "kvc_score_mlp": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "kvc_vector_residual": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _I, _I, _P, _P]),
    "kvc_vector_select": (_I, [_P, _I, _I, _I, _P, _I64, _P, _P, _P, _P]),
    "kvc_vector_compact": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _P, _I64,
                                _P, _I64, _P, _P, _P, _P, _P]),
    "kvc_decode_vector_workspace": (_SZ, [_I, _I, _I, _I, _I]),
    "kvc_decode_attn_vector": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                    _I, _F, _P, _P, _P, _SZ, _P]),
    "kvc_gather_scores": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I64, _P]),
    "kvc_decode_prune": (_I, [ctypes.POINTER(_P), ctypes.POINTER(_I), _I, _P, _P, _P, _P, _I, _I,
                              _I, _F, _I64, _P]),
    "kvc_decode_prune_ring": (_I, [ctypes.POINTER(_P), ctypes.POINTER(_I), _I, _P, _P, _P, _P,
                                   _I64, _P, _I, _I, _I, _F, _I64, _P]),
    "kvc_prune_ring_init": (_I, [_P, _I, _I, _I64, _P, _P]),
    "kvc_decode_noalloc_scratch_bytes": (_SZ, []),
    "kvc_decode_attn_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P,
                                     _P, _P]),
    "kvc_fidelity": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "kvc_selftest_wait_timeout": (_I, [_U64, _P]),
}


class KvcError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


def load(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libkvc.so not built ({path}); run "
                          "`python -m kv_cache_compression_attention_b300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("kvc kernels take CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("kvc kernels take contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _src_ptr(t: torch.Tensor):
    """A source the compaction reads in place: a CUDA tensor, or a host tensor
    (the library accepts pinned host memory the device can read at the same
    address, and refuses any other with KVC_ERR_INVALID before launching)."""
    if not t.is_contiguous():
        raise ValueError("kvc kernels take contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return KVC_F32
    if t.dtype == torch.bfloat16:
        return KVC_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, rc: int):
    if rc != 0:
        raise KvcError(fn, rc)


def _workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


# ----------------------------------------------------------------- entry points
def kvc_score_attn(q_win, k, scores, scale, head_scale=None, causal=True, workspace=None,
                   stream=None, aggregation="sum"):
    """aggregation "sum" (attention mass) calls kvc_score_attn, "max" calls
    kvc_score_attn_agg with KVC_AGG_MAX."""
    U, Hq, W, d = q_win.shape
    _, Hkv, T, _ = k.shape
    dt = _dtype(k)
    need = lib().kvc_score_attn_workspace(U, Hq, Hkv, T, W, d, dt)
    if workspace is None:
        workspace = _workspace(need, k.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if aggregation == "sum":
        rc = lib().kvc_score_attn(_ptr(q_win), _ptr(k), dt, U, Hq, Hkv, T, W, d, float(scale),
                                  _ptr(head_scale), int(bool(causal)), _ptr(scores),
                                  _ptr(workspace), ws_bytes, _stream(stream))
        _check("kvc_score_attn", rc)
    else:
        rc = lib().kvc_score_attn_agg(_ptr(q_win), _ptr(k), dt, U, Hq, Hkv, T, W, d,
                                      float(scale), _ptr(head_scale), int(bool(causal)),
                                      AGGREGATIONS[aggregation], _ptr(scores), _ptr(workspace),
                                      ws_bytes, _stream(stream))
        _check("kvc_score_attn_agg", rc)
    return scores


def kvc_score_linear(hidden, weight, bias, scores, stream=None):
    U, T, Dh = hidden.shape
    Hkv = weight.shape[1]
    rc = lib().kvc_score_linear(_ptr(hidden), _ptr(weight), _ptr(bias), _dtype(hidden), U, T, Dh,
                                Hkv, _ptr(scores), _stream(stream))
    _check("kvc_score_linear", rc)
    return scores


def kvc_score_kvzip_plus(q_win, k, v, gram, hnorm, scores, scale, head_scale=None, causal=True,
                         workspace=None, stream=None):
    """KVzip+ scores [U, Hkv, T] fp32 (q_win, k, v, gram bf16; hnorm [U, W] fp32)."""
    U, Hq, W, d = q_win.shape
    _, Hkv, T, _ = k.shape
    need = lib().kvc_score_kvzip_plus_workspace(U, Hq, Hkv, T, W)
    if workspace is None:
        workspace = _workspace(need, k.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().kvc_score_kvzip_plus(_ptr(q_win), _ptr(k), _ptr(v), _ptr(gram), _ptr(hnorm),
                                    _dtype(k), U, Hq, Hkv, T, W, d, float(scale),
                                    _ptr(head_scale), int(bool(causal)), _ptr(scores),
                                    _ptr(workspace), ws_bytes, _stream(stream))
    _check("kvc_score_kvzip_plus", rc)
    return scores


def kvc_score_mlp(hidden, w1, b1, w2, b2, scores, workspace=None, stream=None):
    """Two-layer surrogate: hidden [U, T, Dh] bf16, w1 [Dh, Dm] bf16, b1 [Dm] fp32,
    w2 [Dm, Hkv] bf16, b2 [Hkv] fp32 -> scores [U, Hkv, T] fp32."""
    U, T, Dh = hidden.shape
    Dm, Hkv = w2.shape
    need = lib().kvc_score_mlp_workspace(Dh, Dm)
    if workspace is None:
        workspace = _workspace(need, hidden.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().kvc_score_mlp(_ptr(hidden), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2),
                             _dtype(hidden), U, T, Dh, Dm, Hkv, _ptr(scores), _ptr(workspace),
                             ws_bytes, _stream(stream))
    _check("kvc_score_mlp", rc)
    return scores


def kvc_select(scores, mode, kept_idx, counts, offsets, keep_ratio=0.0, tau=0.0,
               head_budget=None, n_sink=0, n_recent=0, stream=None):
    U, Hkv, T = scores.shape
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    rc = lib().kvc_select(_ptr(scores), U, Hkv, T, m, float(keep_ratio), float(tau),
                          _ptr(head_budget), int(n_sink), int(n_recent), _ptr(kept_idx),
                          _ptr(counts), _ptr(offsets), None, 0, _stream(stream))
    _check("kvc_select", rc)


def kvc_compact(k, v, kept_idx, counts, offsets, kc, vc, start, length, slack=0, stream=None):
    U, Hkv, T, d = k.shape
    rc = lib().kvc_compact(_src_ptr(k), _src_ptr(v), _dtype(k), U, Hkv, T, d, _ptr(kept_idx),
                           _ptr(counts), _ptr(offsets), int(slack), _ptr(kc), _ptr(vc),
                           kc.shape[0], _ptr(start), _ptr(length), _stream(stream))
    _check("kvc_compact", rc)


def kvc_select_compact(scores, mode, k, v, kept_idx, counts, offsets, kc, vc, start, length,
                       keep_ratio=0.0, tau=0.0, head_budget=None, n_sink=0, n_recent=0, slack=0,
                       workspace=None, stream=None):
    """kvc_select then kvc_compact in one call (see kvc.h); workspace None
    allocates kvc_select_compact_workspace() bytes."""
    U, Hkv, T = scores.shape
    d = k.shape[-1]
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    if workspace is None:
        workspace = _workspace(lib().kvc_select_compact_workspace(U, Hkv, T, m), scores.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().kvc_select_compact(_ptr(scores), U, Hkv, T, m, float(keep_ratio), float(tau),
                                  _ptr(head_budget), int(n_sink), int(n_recent), _src_ptr(k), _src_ptr(v),
                                  _dtype(k), d, int(slack), _ptr(kc), _ptr(vc), kc.shape[0],
                                  _ptr(kept_idx), _ptr(counts), _ptr(offsets), _ptr(start),
                                  _ptr(length), _ptr(workspace) if ws_bytes else None, ws_bytes,
                                  _stream(stream))
    _check("kvc_select_compact", rc)


def kvc_decode_workspace(U, Hq, Hkv, d, max_len, dtype=KVC_BF16) -> int:
    return lib().kvc_decode_workspace(U, Hq, Hkv, d, max_len, dtype)


def kvc_decode_vector_workspace(U, Hq, Hkv, d, max_len) -> int:
    return lib().kvc_decode_vector_workspace(U, Hq, Hkv, d, max_len)


def kvc_decode_attn(q, kc, vc, start, length, out, lse=None, k_new=None, v_new=None,
                    max_len=None, scale=None, workspace=None, stream=None):
    U, Hq, d = q.shape
    Hkv = start.numel() // U
    if max_len is None:
        raise ValueError("max_len is required (upper bound of any head's length)")
    if scale is None:
        scale = d ** -0.5
    dt = _dtype(q)
    need = lib().kvc_decode_workspace(U, Hq, Hkv, d, int(max_len), dt)
    if workspace is None:
        workspace = _workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().kvc_decode_attn(_ptr(q), _ptr(kc), _ptr(vc), _ptr(start), _ptr(length),
                               _ptr(k_new), _ptr(v_new), dt, U, Hq, Hkv, d, int(max_len),
                               float(scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                               _stream(stream))
    _check("kvc_decode_attn", rc)


def kvc_quantize_rows(x, codes, params, stream=None):
    """x [rows, d] bf16 -> codes [rows, d] uint8, params [rows, d / 32, 2] float16 (scale, lo)."""
    rows, d = x.shape
    rc = lib().kvc_quantize_rows(_ptr(x), _dtype(x), int(rows), int(d), _ptr(codes),
                                 _ptr(params), _stream(stream))
    _check("kvc_quantize_rows", rc)


def kvc_decode_attn_q8(q, kq, kp, vq, vp, start, length, out, lse=None, k_new=None, v_new=None,
                       max_len=None, scale=None, workspace=None, stream=None):
    """kvc_decode_attn over a group-quantised pool (codes kq / vq [rows, d] uint8,
    pairs kp / vp [rows, d / 32, 2] float16)."""
    U, Hq, d = q.shape
    Hkv = start.numel() // U
    if max_len is None:
        raise ValueError("max_len is required (upper bound of any head's length)")
    if scale is None:
        scale = d ** -0.5
    dt = _dtype(q)
    need = lib().kvc_decode_workspace(U, Hq, Hkv, d, int(max_len), dt)
    if workspace is None:
        workspace = _workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().kvc_decode_attn_q8(_ptr(q), _ptr(kq), _ptr(kp), _ptr(vq), _ptr(vp), _ptr(start),
                                  _ptr(length), _ptr(k_new), _ptr(v_new), dt, U, Hq, Hkv, d,
                                  int(max_len), float(scale), _ptr(out), _ptr(lse),
                                  _ptr(workspace), ws_bytes, _stream(stream))
    _check("kvc_decode_attn_q8", rc)


def kvc_vector_residual(k, v, W, kept_idx, counts, key, n_sink=0, n_recent=0, stream=None):
    """VECTOR step 2: key[u, g, j] = -||v - W k||^2 of pool position j (NaN if
    protected or empty).  k, v [U, Hkv, T, d] bf16; W [Hkv, d, d] bf16."""
    U, Hkv, T, d = k.shape
    rc = lib().kvc_vector_residual(_ptr(k), _ptr(v), _ptr(W), _dtype(k), U, Hkv, T, d,
                                   _ptr(kept_idx), _ptr(counts), int(n_sink), int(n_recent),
                                   _ptr(key), _stream(stream))
    _check("kvc_vector_residual", rc)


def kvc_vector_select(key, counts, n_approx, approx_pos, approx_counts, approx_offsets,
                      stream=None):
    """VECTOR step 3's choice: per unit, the n_approx highest keys among the
    pool positions j < counts[i] of its heads.  key [U, Hkv, T] fp32."""
    U, Hkv, T = key.shape
    rc = lib().kvc_vector_select(_ptr(key), U, Hkv, T, _ptr(counts), int(n_approx),
                                 _ptr(approx_pos), _ptr(approx_counts), _ptr(approx_offsets),
                                 _stream(stream))
    _check("kvc_vector_select", rc)


def kvc_vector_compact(k, v, kept_idx, counts, offsets, approx_pos, approx_counts,
                       approx_offsets, kc, vc, kstart, klen, vstart, napprox, slack=0,
                       stream=None):
    """VECTOR step 3: K rows of every pool token (approximated first), V rows of
    the exact ones."""
    U, Hkv, T, d = k.shape
    rc = lib().kvc_vector_compact(_ptr(k), _ptr(v), _dtype(k), U, Hkv, T, d, _ptr(kept_idx),
                                  _ptr(counts), _ptr(offsets), _ptr(approx_pos),
                                  _ptr(approx_counts), _ptr(approx_offsets), int(slack),
                                  _ptr(kc), int(kc.shape[0]), _ptr(vc), int(vc.shape[0]),
                                  _ptr(kstart), _ptr(klen), _ptr(vstart), _ptr(napprox),
                                  _stream(stream))
    _check("kvc_vector_compact", rc)


def kvc_decode_attn_vector(q, kc, vc, kstart, klen, vstart, napprox, W, out, lse=None,
                           k_new=None, v_new=None, max_len=None, scale=None, workspace=None,
                           stream=None):
    """One decode step over a VECTOR cache (values of the first napprox rows of
    each head rebuilt as W k)."""
    U, Hq, d = q.shape
    Hkv = kstart.numel() // U
    if max_len is None:
        raise ValueError("max_len is required (upper bound of any head's length)")
    if scale is None:
        scale = d ** -0.5
    need = lib().kvc_decode_vector_workspace(U, Hq, Hkv, d, int(max_len))
    if workspace is None:
        workspace = _workspace(need, q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib().kvc_decode_attn_vector(_ptr(q), _ptr(kc), _ptr(vc), _ptr(kstart), _ptr(klen),
                                      _ptr(vstart), _ptr(napprox), _ptr(W), _ptr(k_new),
                                      _ptr(v_new), _dtype(q), U, Hq, Hkv, d, int(max_len),
                                      float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                      ws_bytes, _stream(stream))
    _check("kvc_decode_attn_vector", rc)


def kvc_gather_scores(scores, kept_idx, counts, start, rscore, stream=None):
    """scores [U, Hkv, T] fp32 -> rscore[start_i + j] = scores of the kept rows."""
    U, Hkv, T = scores.shape
    rc = lib().kvc_gather_scores(_ptr(scores), U, Hkv, T, _ptr(kept_idx), _ptr(counts),
                                 _ptr(start), _ptr(rscore), int(rscore.numel()), _stream(stream))
    _check("kvc_gather_scores", rc)


def kvc_decode_prune(pools, rscore, start, length, s_new, tau, window, n_sink=0, stream=None):
    """Decode-time pruning after an appending decode step.  pools: the row-indexed
    device tensors to move together (e.g. [kc, vc] or [kq, kp, vq, vp]), all with
    rscore.numel() rows."""
    n = len(pools)
    ptrs = (_P * n)(*[_ptr(p) for p in pools])
    rb = (_I * n)(*[int(p.stride(0) * p.element_size()) for p in pools])
    rows = int(rscore.numel())
    for p in pools:
        if p.shape[0] != rows or not p.is_contiguous():
            raise ValueError("every pool needs rscore.numel() contiguous rows")
    rc = lib().kvc_decode_prune(ptrs, rb, n, _ptr(rscore), _ptr(start), _ptr(length),
                                _ptr(s_new), int(length.numel()), int(window), int(n_sink),
                                float(tau), rows, _stream(stream))
    _check("kvc_decode_prune", rc)


def kvc_decode_prune_ring(pools, rscore, start, length, ring, t_new, s_new, tau, window,
                          n_sink=0, stream=None):
    """Decode-time pruning with the window kept as a ring of row indices:
    ring [n_heads, window] int32 (kvc_prune_ring_init), t_new the position of
    the token the step appended."""
    n = len(pools)
    ptrs = (_P * n)(*[_ptr(p) for p in pools])
    rb = (_I * n)(*[int(p.stride(0) * p.element_size()) for p in pools])
    rows = int(rscore.numel())
    for p in pools:
        if p.shape[0] != rows or not p.is_contiguous():
            raise ValueError("every pool needs rscore.numel() contiguous rows")
    rc = lib().kvc_decode_prune_ring(ptrs, rb, n, _ptr(rscore), _ptr(start), _ptr(length),
                                     _ptr(ring), int(t_new), _ptr(s_new), int(length.numel()),
                                     int(window), int(n_sink), float(tau), rows, _stream(stream))
    _check("kvc_decode_prune_ring", rc)


def kvc_prune_ring_init(length, window, t_next, ring, stream=None):
    rc = lib().kvc_prune_ring_init(_ptr(length), int(length.numel()), int(window), int(t_next),
                                   _ptr(ring), _stream(stream))
    _check("kvc_prune_ring_init", rc)


def kvc_decode_attn_noalloc(q, kc, vc, start, length, out, lse=None, k_new=None, v_new=None,
                            max_len=None, scale=None, stream=None):
    """kvc_decode_attn for callers that cannot allocate device memory: the
    split-K scratch is the library's fixed device array, so no workspace is
    allocated here either.  Calls that overlap on the GPU race on that array."""
    U, Hq, d = q.shape
    Hkv = start.numel() // U
    if max_len is None:
        raise ValueError("max_len is required (upper bound of any head's length)")
    if scale is None:
        scale = d ** -0.5
    rc = lib().kvc_decode_attn_noalloc(_ptr(q), _ptr(kc), _ptr(vc), _ptr(start), _ptr(length),
                                       _ptr(k_new), _ptr(v_new), _dtype(q), U, Hq, Hkv, d,
                                       int(max_len), float(scale), _ptr(out), _ptr(lse),
                                       _stream(stream))
    _check("kvc_decode_attn_noalloc", rc)


def kvc_fidelity(out_comp, out_full, lse_comp, lse_full, rel_err, kl, stream=None):
    d = out_comp.shape[-1]
    n = out_comp.numel() // d
    rc = lib().kvc_fidelity(_ptr(out_comp), _ptr(out_full), _ptr(lse_comp), _ptr(lse_full),
                            _dtype(out_comp), n, d, _ptr(rel_err), _ptr(kl), _stream(stream))
    _check("kvc_fidelity", rc)


def kvc_device_status(stream=None) -> int:
    return lib().kvc_device_status(_stream(stream))


def kvc_selftest_wait_timeout(timeout_ns: int, stream=None):
    _check("kvc_selftest_wait_timeout", lib().kvc_selftest_wait_timeout(int(timeout_ns),
                                                                        _stream(stream)))
