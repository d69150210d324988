"""Thin Python binding of the Engram C ABI (include/engram.h).

Argument marshalling only: torch tensors provide device memory and the current
stream; every step of the hot path runs in the CUDA library.  There is no CPU or
PyTorch fallback: if the library is missing, loading fails with an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build

_c = ctypes
_p, _i32, _i64 = _c.c_void_p, _c.c_int32, _c.c_int64

F32, BF16 = 0, 1
_DTYPES = {torch.float32: F32, torch.bfloat16: BF16}

DEVERR_TOKEN_ID = 0x1
DEVERR_COMPRESSED = 0x2
DEVERR_SEQ_OFFSETS = 0x4
DEVERR_TIMEOUT = 0x8


class EngramError(RuntimeError):
    def __init__(self, status: int, where: str, text: str):
        super().__init__(f"{where}: status {status} ({text})")
        self.status = status


class _HashSpec(_c.Structure):
    _fields_ = [("min_order", _i32), ("num_orders", _i32), ("heads", _i32), ("mult_stride", _i32),
                ("multipliers", _p), ("primes", _p)]


class _HashGatherArgs(_c.Structure):
    _fields_ = [("token_ids", _p), ("T", _i64), ("seq_offsets", _p), ("num_seqs", _i32),
                ("compress_map", _p), ("vocab", _i32), ("vocab_c", _i32),
                ("table", _p), ("table_rows", _i64), ("row_dim", _i32), ("dtype", _c.c_int),
                ("out_indices", _p), ("out_rows", _p), ("err_word", _p)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libengram_gb300.so (built in-tree by `build.build()`); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"Engram CUDA library not built ({path}); run __graft_entry__.build() first")
        lib = _c.CDLL(path)
        st = _c.c_int
        sig = {
            "engram_abi_version": (_i32, []),
            "engram_status_string": (_c.c_char_p, [st]),
            "engram_last_error_string": (_c.c_char_p, []),
            "engram_set_validation": (_i32, [_i32]),
            "engram_set_max_ctas": (_i32, [_i32]),
            "engram_set_pdl": (_i32, [_i32]),
            "engram_set_hc_split": (_i32, [_i32]),
            "engram_read_error_word": (st, [_p, _p, _p]),
            "engram_device_status": (st, [_p, _i32]),
            "engram_check_wait_timeout": (st, [_c.c_uint32, _p]),
            "engram_hash_gather": (st, [_p, _p, _p]),
            "engram_hash_gather_host": (st, [_p, _p, _p]),
            "engram_fuse_weight": (st, [_p, _p, _c.c_int, _p, _i32, _p]),
            "engram_gate_fwd": (st, [_p, _p, _p, _c.c_int, _p, _i64, _i32, _c.c_float, _p, _p, _p, _p, _p, _p]),
            "engram_gate_fwd_fold": (st, [_p, _p, _p, _c.c_int, _p, _p, _c.c_int, _i64, _i32, _c.c_float, _p, _p, _p,
                                          _p, _p, _p, _p]),
            "engram_gate_fwd_rms": (st, [_p, _p, _p, _c.c_int, _p, _i64, _i32, _c.c_float, _p, _p, _p, _p, _p, _p,
                                         _c.c_float, _p]),
            "engram_gate_bwd_num_partials": (st, [_i64, _i32, _p]),
            "engram_gate_bwd": (st, [_p, _p, _p, _p, _c.c_int, _p, _p, _p, _p, _p, _i64, _i32, _p, _p, _p, _p,
                                     _i32, _p]),
            "engram_gate_bwd_accumulate": (st, [_p, _p, _p, _p, _c.c_int, _p, _p, _p, _p, _p, _i64, _i32, _p, _p,
                                                _p, _p, _i32, _p]),
            "engram_grad_w_reduce": (st, [_p, _i32, _i32, _p, _p, _p, _p, _p, _p]),
            "engram_gate_hc_fwd": (st, [_p, _p, _c.c_int, _p, _i64, _i32, _i32, _c.c_float, _c.c_float, _p, _p, _p,
                                        _p, _p, _p]),
            "engram_gate_hc_bwd": (st, [_p, _p, _p, _c.c_int, _p, _p, _p, _p, _p, _i64, _i32, _i32, _c.c_float, _p,
                                        _p, _p, _i32, _p]),
            "engram_gate_bwd_reduce_noalloc": (st, [_p, _p, _p, _p, _c.c_int, _p, _p, _p, _p, _p, _i64, _i32, _p, _p,
                                                    _p, _p, _p, _p, _p, _p, _p]),
            "engram_short_conv_fwd": (st, [_p, _p, _c.c_int, _p, _p, _p, _p, _i32, _i64, _i32, _i32, _i32,
                                           _c.c_float, _p, _p, _p]),
            "engram_short_conv_fwd_given_rstd": (st, [_p, _p, _c.c_int, _p, _p, _p, _p, _i32, _i64, _i32, _i32,
                                                      _i32, _p, _p, _p]),
            "engram_short_conv_num_partials": (st, [_i64, _i32, _p]),
            "engram_short_conv_bwd": (st, [_p, _p, _c.c_int, _p, _p, _p, _p, _p, _i32, _i64, _i32, _i32, _i32, _p,
                                           _p, _i32, _p]),
            "engram_short_conv_grad_reduce": (st, [_p, _i32, _i32, _i32, _p, _p, _p, _p]),
            "engram_sinkhorn_momentum_update": (st, [_p, _c.c_int, _p, _p, _i64, _c.c_float, _i32, _p]),
            "engram_sinkhorn_num_partials": (st, [_i64, _i32, _p]),
            "engram_sinkhorn_step": (st, [_p, _p, _p, _i64, _i32, _c.c_float, _p, _p, _i32, _p]),
            "engram_sinkhorn_step_reduce": (st, [_p, _i32, _i32, _p, _p, _c.c_float, _p]),
            "engram_sinkhorn_finalize": (st, [_p, _p, _p, _i64, _i32, _c.c_float, _c.c_float, _p, _p]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype, f.argtypes = res, args
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        lib = load_library()
        raise EngramError(status, where, lib.engram_last_error_string().decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _need(t, name, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def set_validation(level: int) -> int:
    return load_library().engram_set_validation(level)


def set_max_ctas(max_ctas: int) -> int:
    """Cap the CTAs per launch (0 = none); returns the previous cap."""
    return load_library().engram_set_max_ctas(max_ctas)


HC_AUTO, HC_BRANCHES, HC_ROW_SPLIT, HC_ROW_SPLIT4 = 0, 1, 2, 4


def set_hc_split(mode) -> int:
    """The multi-branch gate's form (a test knob): HC_AUTO (0, each call picks), HC_BRANCHES (1 or True,
    branch by branch at every size), HC_ROW_SPLIT / HC_ROW_SPLIT4 (2 / 4, each token shared by a cluster
    of two / four CTAs where their parts fit); returns the previous mode."""
    return int(load_library().engram_set_hc_split(int(mode)))


def set_pdl(on: bool) -> bool:
    """Programmatic dependent launch for the step's kernels (on by default); returns the previous setting."""
    return bool(load_library().engram_set_pdl(int(bool(on))))


def abi_version() -> int:
    return load_library().engram_abi_version()


# ----------------------------------------------------------------------------- B0 / B1


def fuse_weight(w_h, w_k, out=None, stream=None):
    """w_fused = w_h * w_k in fp32 (w_h, w_k fp32 or bf16)."""
    lib = load_library()
    _need(w_h, "w_h")
    _need(w_k, "w_k", w_h.dtype)
    d = w_h.numel()
    out = torch.empty(d, dtype=torch.float32, device=w_h.device) if out is None else _need(out, "out", torch.float32)
    _check(lib.engram_fuse_weight(_ptr(w_h), _ptr(w_k), _DTYPES[w_h.dtype], _ptr(out), d, _stream(stream)),
           "engram_fuse_weight")
    return out


def gate_fwd(h, k, v, w_fused, eps: float = 1e-6, out=None, save_for_backward: bool = True, stats=None,
             stream=None):
    """out = alpha * v with alpha = sigmoid(RMSNorm(h)·RMSNorm(k)/sqrt(d)); returns (out, alpha, rstd_h, rstd_k, dot).

    The statistics are None unless save_for_backward.  `stats` may supply the four [T] fp32 buffers.
    """
    lib = load_library()
    _need(h, "h")
    _need(k, "k", h.dtype)
    _need(v, "v", h.dtype)
    _need(w_fused, "w_fused", torch.float32)
    T, d = h.shape
    out = torch.empty_like(v) if out is None else _need(out, "out", h.dtype)
    if save_for_backward:
        if stats is None:
            stats = tuple(torch.empty(T, dtype=torch.float32, device=h.device) for _ in range(4))
        alpha, rh, rk, dot = (_need(x, "stat", torch.float32) for x in stats)
    else:
        alpha = rh = rk = dot = None
    _check(lib.engram_gate_fwd(_ptr(h), _ptr(k), _ptr(v), _DTYPES[h.dtype], _ptr(w_fused), T, d, float(eps),
                               _ptr(out), _ptr(alpha), _ptr(rh), _ptr(rk), _ptr(dot), _stream(stream)),
           "engram_gate_fwd")
    return out, alpha, rh, rk, dot


def gate_fwd_fold(h, k, v, w_h, w_k, eps: float = 1e-6, out=None, save_for_backward: bool = True, stats=None,
                  w_fused_out=None, stream=None):
    """gate_fwd with the weight fold w_h * w_k done inside the forward (one launch instead of fuse_weight +
    gate_fwd); the fold is written to w_fused_out for the backward.
    Returns (out, alpha, rstd_h, rstd_k, dot, w_fused)."""
    lib = load_library()
    _need(h, "h")
    _need(k, "k", h.dtype)
    _need(v, "v", h.dtype)
    _need(w_h, "w_h")
    _need(w_k, "w_k", w_h.dtype)
    T, d = h.shape
    out = torch.empty_like(v) if out is None else _need(out, "out", h.dtype)
    if save_for_backward:
        if stats is None:
            stats = tuple(torch.empty(T, dtype=torch.float32, device=h.device) for _ in range(4))
        alpha, rh, rk, dot = (_need(x, "stat", torch.float32) for x in stats)
    else:
        alpha = rh = rk = dot = None
    w_fused_out = (torch.empty(d, dtype=torch.float32, device=h.device) if w_fused_out is None
                   else _need(w_fused_out, "w_fused_out", torch.float32))
    _check(lib.engram_gate_fwd_fold(_ptr(h), _ptr(k), _ptr(v), _DTYPES[h.dtype], _ptr(w_h), _ptr(w_k),
                                    _DTYPES[w_h.dtype], T, d, float(eps), _ptr(out), _ptr(alpha), _ptr(rh), _ptr(rk),
                                    _ptr(dot), _ptr(w_fused_out), _stream(stream)),
           "engram_gate_fwd_fold")
    return out, alpha, rh, rk, dot, w_fused_out


def gate_fwd_rms(h, k, v, w_fused, eps: float = 1e-6, out_eps: float = 1e-6, out=None, save_for_backward: bool = True,
                 stats=None, out_rstd=None, stream=None):
    """gate_fwd plus out_rstd [T] = 1/sqrt(mean(out_t^2) + out_eps) of each stored output row, the statistic the
    short convolution's RMSNorm needs (short_conv_fwd(..., given_rstd=out_rstd)).
    Returns (out, alpha, rstd_h, rstd_k, dot, out_rstd)."""
    lib = load_library()
    _need(h, "h")
    _need(k, "k", h.dtype)
    _need(v, "v", h.dtype)
    _need(w_fused, "w_fused", torch.float32)
    T, d = h.shape
    out = torch.empty_like(v) if out is None else _need(out, "out", h.dtype)
    if save_for_backward:
        if stats is None:
            stats = tuple(torch.empty(T, dtype=torch.float32, device=h.device) for _ in range(4))
        alpha, rh, rk, dot = (_need(x, "stat", torch.float32) for x in stats)
    else:
        alpha = rh = rk = dot = None
    out_rstd = (torch.empty(T, dtype=torch.float32, device=h.device) if out_rstd is None
                else _need(out_rstd, "out_rstd", torch.float32))
    _check(lib.engram_gate_fwd_rms(_ptr(h), _ptr(k), _ptr(v), _DTYPES[h.dtype], _ptr(w_fused), T, d, float(eps),
                                   _ptr(out), _ptr(alpha), _ptr(rh), _ptr(rk), _ptr(dot), _ptr(out_rstd),
                                   float(out_eps), _stream(stream)),
           "engram_gate_fwd_rms")
    return out, alpha, rh, rk, dot, out_rstd


# ----------------------------------------------------------------------------- B2 / B3


def gate_bwd_num_partials(T: int, d: int) -> int:
    lib = load_library()
    P = _c.c_int32(0)
    _check(lib.engram_gate_bwd_num_partials(T, d, _c.byref(P)), "engram_gate_bwd_num_partials")
    return P.value


def gate_bwd(dout, h, k, v, w_fused, alpha, rstd_h, rstd_k, dot, P: int | None = None, dh=None, dk=None, dv=None,
             dw_partial=None, accumulate: bool = False, stream=None):
    """Returns (dh, dk, dv, dw_partial [P, d] fp32).  accumulate=True adds each partial's terms onto the
    given dw_partial's rows (engram_gate_bwd_accumulate) instead of overwriting them."""
    lib = load_library()
    for name, t in (("dout", dout), ("h", h), ("k", k), ("v", v)):
        _need(t, name, h.dtype)
    for name, t in (("w_fused", w_fused), ("alpha", alpha), ("rstd_h", rstd_h), ("rstd_k", rstd_k), ("dot", dot)):
        _need(t, name, torch.float32)
    T, d = h.shape
    if P is None:
        P = gate_bwd_num_partials(T, d) if dw_partial is None else dw_partial.shape[0]
    dh = torch.empty_like(h) if dh is None else _need(dh, "dh", h.dtype)
    dk = torch.empty_like(k) if dk is None else _need(dk, "dk", h.dtype)
    dv = torch.empty_like(v) if dv is None else _need(dv, "dv", h.dtype)
    if dw_partial is None:
        if accumulate:
            raise ValueError("accumulate=True needs the dw_partial to add to")
        dw_partial = torch.empty((P, d), dtype=torch.float32, device=h.device)
    else:
        _need(dw_partial, "dw_partial", torch.float32)
    fn = lib.engram_gate_bwd_accumulate if accumulate else lib.engram_gate_bwd
    _check(fn(_ptr(dout), _ptr(h), _ptr(k), _ptr(v), _DTYPES[h.dtype], _ptr(w_fused), _ptr(alpha), _ptr(rstd_h),
              _ptr(rstd_k), _ptr(dot), T, d, _ptr(dh), _ptr(dk), _ptr(dv), _ptr(dw_partial), P, _stream(stream)),
           "engram_gate_bwd_accumulate" if accumulate else "engram_gate_bwd")
    return dh, dk, dv, dw_partial


def grad_w_reduce(dw_partial, dweight_fused=None, w_h=None, w_k=None, grad_w_h=None, grad_w_k=None,
                  want_dweight: bool = True, stream=None):
    """dweight_fused = sum_p dw_partial[p]; with weights, grad_w_h += S*w_k and grad_w_k += S*w_h."""
    lib = load_library()
    _need(dw_partial, "dw_partial", torch.float32)
    P, d = dw_partial.shape
    if dweight_fused is None and want_dweight:
        dweight_fused = torch.empty(d, dtype=torch.float32, device=dw_partial.device)
    for name, t in (("w_h", w_h), ("w_k", w_k), ("grad_w_h", grad_w_h), ("grad_w_k", grad_w_k)):
        if t is not None:
            _need(t, name, torch.float32)
    _check(lib.engram_grad_w_reduce(_ptr(dw_partial), P, d, _ptr(dweight_fused), _ptr(w_h), _ptr(w_k),
                                    _ptr(grad_w_h), _ptr(grad_w_k), _stream(stream)),
           "engram_grad_w_reduce")
    return dweight_fused


def gate_bwd_reduce_noalloc(dout, h, k, v, w_fused, alpha, rstd_h, rstd_k, dot, dh=None, dk=None, dv=None,
                            dweight_fused=None, w_h=None, w_k=None, grad_w_h=None, grad_w_k=None,
                            want_dweight: bool = True, stream=None):
    """Backward + weight-gradient reduction without a caller-provided partials buffer.

    For callers that cannot allocate device memory: the partials live in the library's
    own fixed 16 MiB device array (see include/engram.h).  Returns (dh, dk, dv, dweight_fused).
    """
    lib = load_library()
    for name, t in (("dout", dout), ("h", h), ("k", k), ("v", v)):
        _need(t, name, h.dtype)
    T, d = h.shape
    dh = torch.empty_like(h) if dh is None else _need(dh, "dh", h.dtype)
    dk = torch.empty_like(k) if dk is None else _need(dk, "dk", h.dtype)
    dv = torch.empty_like(v) if dv is None else _need(dv, "dv", h.dtype)
    if dweight_fused is None and want_dweight:
        dweight_fused = torch.empty(d, dtype=torch.float32, device=h.device)
    _check(lib.engram_gate_bwd_reduce_noalloc(_ptr(dout), _ptr(h), _ptr(k), _ptr(v), _DTYPES[h.dtype], _ptr(w_fused),
                                              _ptr(alpha), _ptr(rstd_h), _ptr(rstd_k), _ptr(dot), T, d, _ptr(dh),
                                              _ptr(dk), _ptr(dv), _ptr(dweight_fused), _ptr(w_h), _ptr(w_k),
                                              _ptr(grad_w_h), _ptr(grad_w_k), _stream(stream)),
           "engram_gate_bwd_reduce_noalloc")
    return dh, dk, dv, dweight_fused


def gate_hc_fwd(x, kv, w_fused, eps: float = 1e-6, clamp: float = 1e-6, out=None, save_for_backward: bool = True,
                inplace: bool = False, stats=None, stream=None):
    """Multi-branch gate: x [T, hc, d], kv [T, hc+1, d], w_fused [hc, d] fp32.

    Returns (out, gate, rstd_x, rstd_k, dot); with inplace, out is x itself (and nothing is saved).
    """
    lib = load_library()
    _need(x, "x")
    _need(kv, "kv", x.dtype)
    _need(w_fused, "w_fused", torch.float32)
    T, hc, d = x.shape
    if inplace:
        if save_for_backward:
            raise ValueError("inplace overwrites x, which the backward reads; pass save_for_backward=False")
        out = x
    elif out is None:
        out = torch.empty_like(x)
    if save_for_backward:
        if stats is None:
            stats = tuple(torch.empty((T, hc), dtype=torch.float32, device=x.device) for _ in range(4))
        gate, rx, rk, dot = stats
    else:
        gate = rx = rk = dot = None
    _check(lib.engram_gate_hc_fwd(_ptr(x), _ptr(kv), _DTYPES[x.dtype], _ptr(w_fused), T, hc, d, float(eps),
                                  float(clamp), _ptr(out), _ptr(gate), _ptr(rx), _ptr(rk), _ptr(dot), _stream(stream)),
           "engram_gate_hc_fwd")
    return out, gate, rx, rk, dot


def gate_hc_bwd(dout, x, kv, w_fused, gate, rstd_x, rstd_k, dot, clamp: float = 1e-6, P: int | None = None, dx=None,
                dkv=None, dw_partial=None, stream=None):
    """Returns (dx [T, hc, d], dkv [T, hc+1, d], dw_partial [P, hc, d] fp32)."""
    lib = load_library()
    for name, t in (("dout", dout), ("x", x), ("kv", kv)):
        _need(t, name, x.dtype)
    T, hc, d = x.shape
    if P is None:
        P = gate_bwd_num_partials(T, hc * d) if dw_partial is None else dw_partial.shape[0]
    dx = torch.empty_like(x) if dx is None else _need(dx, "dx", x.dtype)
    dkv = torch.empty_like(kv) if dkv is None else _need(dkv, "dkv", x.dtype)
    if dw_partial is None:
        dw_partial = torch.empty((P, hc, d), dtype=torch.float32, device=x.device)
    _check(lib.engram_gate_hc_bwd(_ptr(dout), _ptr(x), _ptr(kv), _DTYPES[x.dtype], _ptr(w_fused), _ptr(gate),
                                  _ptr(rstd_x), _ptr(rstd_k), _ptr(dot), T, hc, d, float(clamp), _ptr(dx), _ptr(dkv),
                                  _ptr(dw_partial), P, _stream(stream)),
           "engram_gate_hc_bwd")
    return dx, dkv, dw_partial


# ----------------------------------------------------------------------------- the short conv after the gate


def short_conv_fwd(v, norm_w, conv_w, seq_offsets, dilation: int, h=None, bias=None, eps: float = 1e-6, out=None,
                   rstd=None, given_rstd=None, stream=None):
    """out = h + SiLU(causal depthwise conv of RMSNorm(v)) + v, per sequence.  Returns (out, rstd).

    given_rstd: the RMSNorm statistic of v already made (gate_fwd_rms), read instead of computed; it is
    then the returned rstd."""
    lib = load_library()
    _need(v, "v")
    _need(norm_w, "norm_w", torch.float32)
    _need(conv_w, "conv_w", torch.float32)
    _need(seq_offsets, "seq_offsets", torch.int64)
    if h is not None:
        _need(h, "h", v.dtype)
    if bias is not None:
        _need(bias, "bias", torch.float32)
    T, d = v.shape
    width = conv_w.shape[1]
    out = torch.empty_like(v) if out is None else _need(out, "out", v.dtype)
    if given_rstd is not None:
        _need(given_rstd, "given_rstd", torch.float32)
        _check(lib.engram_short_conv_fwd_given_rstd(_ptr(v), _ptr(h), _DTYPES[v.dtype], _ptr(norm_w), _ptr(conv_w),
                                                    _ptr(bias), _ptr(seq_offsets), seq_offsets.numel() - 1, T, d,
                                                    width, int(dilation), _ptr(given_rstd), _ptr(out),
                                                    _stream(stream)),
               "engram_short_conv_fwd_given_rstd")
        return out, given_rstd
    rstd = torch.empty(T, dtype=torch.float32, device=v.device) if rstd is None else _need(rstd, "rstd", torch.float32)
    _check(lib.engram_short_conv_fwd(_ptr(v), _ptr(h), _DTYPES[v.dtype], _ptr(norm_w), _ptr(conv_w), _ptr(bias),
                                     _ptr(seq_offsets), seq_offsets.numel() - 1, T, d, width, int(dilation), float(eps),
                                     _ptr(out), _ptr(rstd), _stream(stream)),
           "engram_short_conv_fwd")
    return out, rstd


def short_conv_num_partials(T: int, dilation: int) -> int:
    lib = load_library()
    P = _c.c_int32(0)
    _check(lib.engram_short_conv_num_partials(T, dilation, _c.byref(P)), "engram_short_conv_num_partials")
    return P.value


def short_conv_bwd(dout, v, norm_w, conv_w, rstd, seq_offsets, dilation: int, bias=None, dv=None, dw_partial=None,
                   stream=None):
    """Returns (dv, dw_partial [P, width + 2, d]); dL/dh is dout itself."""
    lib = load_library()
    _need(dout, "dout", v.dtype)
    _need(v, "v")
    T, d = v.shape
    width = conv_w.shape[1]
    P = short_conv_num_partials(T, dilation)
    dv = torch.empty_like(v) if dv is None else _need(dv, "dv", v.dtype)
    if dw_partial is None:
        dw_partial = torch.empty((P, width + 2, d), dtype=torch.float32, device=v.device)
    _check(lib.engram_short_conv_bwd(_ptr(dout), _ptr(v), _DTYPES[v.dtype], _ptr(norm_w), _ptr(conv_w), _ptr(bias),
                                     _ptr(rstd), _ptr(seq_offsets), seq_offsets.numel() - 1, T, d, width,
                                     int(dilation), _ptr(dv), _ptr(dw_partial), P, _stream(stream)),
           "engram_short_conv_bwd")
    return dv, dw_partial


def short_conv_grad_reduce(dw_partial, width: int, d: int, want_bias: bool = True, out=None, stream=None):
    """Returns (dconv_w [d, width], dbias [d] or None, dnorm_w [d])."""
    lib = load_library()
    P = dw_partial.shape[0] if dw_partial is not None else 0
    dev = dw_partial.device
    dconv_w, dbias, dnorm_w = out if out is not None else (
        torch.empty((d, width), dtype=torch.float32, device=dev),
        torch.empty(d, dtype=torch.float32, device=dev) if want_bias else None,
        torch.empty(d, dtype=torch.float32, device=dev))
    _check(lib.engram_short_conv_grad_reduce(_ptr(dw_partial), P, width, d, _ptr(dconv_w), _ptr(dbias), _ptr(dnorm_w),
                                             _stream(stream)),
           "engram_short_conv_grad_reduce")
    return dconv_w, dbias, dnorm_w


# ----------------------------------------------------------------------------- the Engram Sinkhorn


def sinkhorn_momentum_update(grad, momentum, beta1: float, nesterov: bool, sinkhorn_input=None, stream=None):
    """momentum = beta1 * momentum + grad (in place); returns the fp32 Sinkhorn input."""
    lib = load_library()
    _need(grad, "grad")
    _need(momentum, "momentum", torch.float32)
    if grad.shape != momentum.shape:
        raise ValueError(f"grad {tuple(grad.shape)} and momentum {tuple(momentum.shape)} differ")
    out = torch.empty_like(momentum) if sinkhorn_input is None else _need(sinkhorn_input, "sinkhorn_input",
                                                                         torch.float32)
    _check(lib.engram_sinkhorn_momentum_update(_ptr(grad), _DTYPES[grad.dtype], _ptr(momentum), _ptr(out),
                                               momentum.numel(), float(beta1), int(bool(nesterov)), _stream(stream)),
           "engram_sinkhorn_momentum_update")
    return out


def sinkhorn_num_partials(rows: int, head_dim: int) -> int:
    lib = load_library()
    P = _c.c_int32(0)
    _check(lib.engram_sinkhorn_num_partials(rows, head_dim, _c.byref(P)), "engram_sinkhorn_num_partials")
    return P.value


def sinkhorn_step(matrix, row_scale, col_scale, eps: float = 1e-6, P: int | None = None, row_norm=None,
                  col_sumsq_partial=None, want_row_norm: bool = True, stream=None):
    """Row step (row_scale updated in place).  Returns (row_norm [rows] or None, col_sumsq_partial [P, head_dim])."""
    lib = load_library()
    _need(matrix, "matrix", torch.float32)
    _need(row_scale, "row_scale", torch.float32)
    _need(col_scale, "col_scale", torch.float32)
    rows, D = matrix.shape
    if P is None:
        P = sinkhorn_num_partials(rows, D) if col_sumsq_partial is None else col_sumsq_partial.shape[0]
    if row_norm is None and want_row_norm:
        row_norm = torch.empty(rows, dtype=torch.float32, device=matrix.device)
    if col_sumsq_partial is None:
        col_sumsq_partial = torch.empty((P, D), dtype=torch.float32, device=matrix.device)
    else:
        _need(col_sumsq_partial, "col_sumsq_partial", torch.float32)
    _check(lib.engram_sinkhorn_step(_ptr(matrix), _ptr(row_scale), _ptr(col_scale), rows, D, float(eps),
                                    _ptr(row_norm), _ptr(col_sumsq_partial), P, _stream(stream)),
           "engram_sinkhorn_step")
    return row_norm, col_sumsq_partial


def sinkhorn_step_reduce(col_sumsq_partial, col_sumsq=None, col_scale=None, eps: float = 1e-6,
                         want_col_sumsq: bool = True, stream=None):
    """Ordered reduction of the partials; with col_scale, also col_scale /= sqrt(col_sumsq) + eps in place."""
    lib = load_library()
    _need(col_sumsq_partial, "col_sumsq_partial", torch.float32)
    P, D = col_sumsq_partial.shape
    if col_sumsq is None and want_col_sumsq:
        col_sumsq = torch.empty(D, dtype=torch.float32, device=col_sumsq_partial.device)
    if col_scale is not None:
        _need(col_scale, "col_scale", torch.float32)
    _check(lib.engram_sinkhorn_step_reduce(_ptr(col_sumsq_partial), P, D, _ptr(col_sumsq), _ptr(col_scale), float(eps),
                                           _stream(stream)),
           "engram_sinkhorn_step_reduce")
    return col_sumsq


def sinkhorn_finalize(matrix, row_scale, col_scale, eps: float = 1e-6, alpha: float = 1.0, out=None, stream=None):
    """out = alpha * x / (||x|| + eps) per row, x = row_scale * matrix * col_scale."""
    lib = load_library()
    _need(matrix, "matrix", torch.float32)
    rows, D = matrix.shape
    out = torch.empty_like(matrix) if out is None else _need(out, "out", torch.float32)
    _check(lib.engram_sinkhorn_finalize(_ptr(matrix), _ptr(row_scale), _ptr(col_scale), rows, D, float(eps),
                                        float(alpha), _ptr(out), _stream(stream)),
           "engram_sinkhorn_finalize")
    return out


# ----------------------------------------------------------------------------- A0-A2


class HashSpec:
    """The hash hyper-parameters, kept as host arrays for the C ABI."""

    def __init__(self, min_order: int, num_orders: int, heads: int, multipliers, primes):
        self.min_order, self.num_orders, self.heads = int(min_order), int(num_orders), int(heads)
        self.multipliers = np.ascontiguousarray(multipliers, dtype=np.uint64)
        self.primes = np.ascontiguousarray(primes, dtype=np.uint64)
        self.tables = self.num_orders * self.heads
        if self.multipliers.ndim != 2 or self.multipliers.shape[0] != self.tables or len(self.primes) != self.tables:
            raise ValueError("multipliers must be [tables, stride] and primes [tables]")

    def _c(self):
        return _HashSpec(self.min_order, self.num_orders, self.heads, self.multipliers.shape[1],
                         self.multipliers.ctypes.data, self.primes.ctypes.data)


def hash_gather(spec: HashSpec, token_ids, seq_offsets, table, compress_map=None, vocab: int | None = None,
                vocab_c: int | None = None, want_rows: bool = True, want_indices: bool = False, out_rows=None,
                out_indices=None, err_word=None, stream=None):
    """Returns (rows [T, tables*row_dim] or None, indices [T, tables] int32 or None).

    A table in pinned host memory (a CPU tensor with is_pinned()) is read over the host link
    (engram_hash_gather_host); a CUDA table is read from HBM.
    """
    lib = load_library()
    _need(token_ids, "token_ids", torch.int32)
    _need(seq_offsets, "seq_offsets", torch.int64)
    host_table = not table.is_cuda
    if host_table:
        if not (table.is_pinned() and table.is_contiguous()):
            raise ValueError("a host table must be a contiguous, pinned CPU tensor")
    else:
        _need(table, "table")
    device = token_ids.device
    if compress_map is not None:
        _need(compress_map, "compress_map", torch.int32)
    T = token_ids.numel()
    rows_total, row_dim = table.shape
    if vocab is None:
        vocab = compress_map.numel() if compress_map is not None else (1 << 31) - 1
    if vocab_c is None:
        vocab_c = vocab
    if want_rows and out_rows is None:
        out_rows = torch.empty((T, spec.tables * row_dim), dtype=table.dtype, device=device)
    if want_indices and out_indices is None:
        out_indices = torch.empty((T, spec.tables), dtype=torch.int32, device=device)
    args = _HashGatherArgs(_ptr(token_ids), T, _ptr(seq_offsets), seq_offsets.numel() - 1, _ptr(compress_map),
                           vocab, vocab_c, _ptr(table), rows_total, row_dim, _DTYPES[table.dtype],
                           _ptr(out_indices), _ptr(out_rows), _ptr(err_word))
    cspec = spec._c()
    fn = lib.engram_hash_gather_host if host_table else lib.engram_hash_gather
    _check(fn(_c.byref(cspec), _c.byref(args), _stream(stream)), "engram_hash_gather")
    return out_rows, out_indices


# ----------------------------------------------------------------------------- errors


def read_error_word(err_word, stream=None) -> int:
    """Synchronises the stream and returns the device error word's bits."""
    lib = load_library()
    out = _c.c_uint32(0)
    st = lib.engram_read_error_word(_ptr(err_word), _stream(stream), _c.byref(out))
    if st not in (0, 6):
        _check(st, "engram_read_error_word")
    return out.value


def device_status(clear: bool = False) -> int:
    """Synchronises the device and returns the library's device status bits on the current device."""
    lib = load_library()
    out = _c.c_uint32(0)
    st = lib.engram_device_status(_c.byref(out), 1 if clear else 0)
    if st not in (0, 6):
        _check(st, "engram_device_status")
    return out.value


def check_wait_timeout(limit_us: int = 50000, stream=None):
    """Launch the failure-detection self-check (a bounded wait that must give up); read the result
    with device_status()."""
    _check(load_library().engram_check_wait_timeout(int(limit_us), _stream(stream)), "engram_check_wait_timeout")
