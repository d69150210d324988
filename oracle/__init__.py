"""CPU oracle for the Engram hash-gather and context-aware-gate hot path.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package's smoke check
and by the benchmark's CPU-baseline leg, never by the product path.  The
arithmetic lives in ``engram_oracle.c`` (plain scalar C, fp64 accumulation);
this module only marshals numpy arrays through ctypes.  ctypes releases the GIL
during each call, so callers may split token ranges across Python threads.

Every function is pinned by the CPU test suite against closed forms, torch
library routines, autograd and finite differences (see the header of the C file).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "liboracle_engram.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f64 = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile the oracle library with `make` (gcc, C11) if it is missing or stale."""
    src = os.path.join(_HERE, "engram_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        subprocess.run(["make", "-s", "-C", _HERE], check=True)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            lib.eo_hash_indices.argtypes = [_p, _i64, _p, _i32, _p, _i32, _i32, _i32, _i32, _p, _i32, _p,
                                            _i64, _i64, _p]
            lib.eo_gather_rows.argtypes = [_p, _i64, _i32, _p, _i32, _p, _i64, _p]
            lib.eo_fuse_weight.argtypes = [_p, _p, _i32, _p]
            lib.eo_gate_fwd.argtypes = [_p, _p, _p, ctypes.c_int, _p, _p, _i64, _i32, _f64, _i64, _i64,
                                        _p, _p, _p, _p, _p, _p]
            lib.eo_gate_bwd.argtypes = [_p, _p, _p, _p, ctypes.c_int, _p, _p, _i64, _i32, _f64, _i64, _i64,
                                        _p, _p, _p, _p, _p]
            lib.eo_grad_w_reduce.argtypes = [_p, _i32, _i32, _p, _p, _p, _p, _p]
            lib.eo_gate_hc_fwd.argtypes = [_p, _p, ctypes.c_int, _p, _p, _i64, _i32, _i32, _f64, _f64, _i64, _i64,
                                           _p, _p, _p, _p, _p]
            lib.eo_gate_hc_bwd.argtypes = [_p, _p, _p, ctypes.c_int, _p, _p, _i64, _i32, _i32, _f64, _f64, _i64,
                                           _i64, _p, _p, _p, _p]
            lib.eo_sinkhorn_momentum.argtypes = [_p, ctypes.c_int, _p, _i64, _f64, ctypes.c_int, _p, _p]
            lib.eo_sinkhorn_step.argtypes = [_p, _p, _p, _i64, _i32, _f64, _i64, _i64, _p, _p, _p]
            lib.eo_sinkhorn_col_update.argtypes = [_p, _p, _i32, _f64, _p]
            lib.eo_sinkhorn_finalize.argtypes = [_p, _p, _p, _i64, _i32, _f64, _f64, _p]
            lib.eo_short_conv_fwd.argtypes = [_p, _p, ctypes.c_int, _p, _p, _p, _p, _i32, _i64, _i32, _i32, _i32,
                                              _f64, _i64, _i64, _p, _p, _p]
            lib.eo_short_conv_bwd.argtypes = [_p, _p, ctypes.c_int, _p, _p, _p, _p, _i32, _i64, _i32, _i32, _i32,
                                              _f64, _i64, _i64, _p, _p, _p, _p, _p, _p, _p, _p]
            for f in ("eo_short_conv_fwd", "eo_short_conv_bwd", "eo_sinkhorn_momentum", "eo_sinkhorn_step", "eo_sinkhorn_col_update", "eo_sinkhorn_finalize",
                      "eo_hash_indices", "eo_gather_rows", "eo_fuse_weight", "eo_gate_fwd", "eo_gate_bwd",
                      "eo_grad_w_reduce", "eo_gate_hc_fwd", "eo_gate_hc_bwd"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError("oracle tensors are float32 or raw bfloat16 bits (uint16)")


def hash_indices(token_ids, seq_offsets, compress_map, vocab, min_order, num_orders, heads, multipliers, primes,
                 t_begin: int = 0, t_end: int | None = None) -> np.ndarray:
    """[t_end - t_begin, tables] int64 hash indices (local to each table)."""
    lib = _load()
    ids = np.ascontiguousarray(token_ids, dtype=np.int32)
    offs = np.ascontiguousarray(seq_offsets, dtype=np.int64)
    cmap = None if compress_map is None else np.ascontiguousarray(compress_map, dtype=np.int32)
    mult = np.ascontiguousarray(multipliers, dtype=np.uint64)
    pr = np.ascontiguousarray(primes, dtype=np.uint64)
    T = ids.shape[0]
    t_end = T if t_end is None else t_end
    tables = num_orders * heads
    out = np.zeros((t_end - t_begin, tables), dtype=np.int64)
    rc = lib.eo_hash_indices(_ptr(ids), T, _ptr(offs), len(offs) - 1, _ptr(cmap), vocab, min_order, num_orders,
                             heads, _ptr(mult), mult.shape[1], _ptr(pr), t_begin, t_end, _ptr(out))
    _check(rc, "hash_indices")
    return out


def gather_rows(table: np.ndarray, primes, idx: np.ndarray) -> np.ndarray:
    """[ntok, tables, row] rows of the concatenated table picked by idx [ntok, tables]."""
    lib = _load()
    tab = np.ascontiguousarray(table)
    pr = np.ascontiguousarray(primes, dtype=np.uint64)
    ix = np.ascontiguousarray(idx, dtype=np.int64)
    ntok, tables = ix.shape
    row = tab.shape[1]
    out = np.zeros((ntok, tables, row), dtype=tab.dtype)
    rc = lib.eo_gather_rows(_ptr(tab), tab.shape[0], row * tab.dtype.itemsize, _ptr(pr), tables, _ptr(ix), ntok,
                            _ptr(out))
    _check(rc, "gather_rows")
    return out


def fuse_weight(w_h, w_k) -> np.ndarray:
    lib = _load()
    a = np.ascontiguousarray(w_h, dtype=np.float32)
    b = np.ascontiguousarray(w_k, dtype=np.float32)
    out = np.zeros(a.shape[0], dtype=np.float64)
    _check(lib.eo_fuse_weight(_ptr(a), _ptr(b), a.shape[0], _ptr(out)), "fuse_weight")
    return out


def gate_fwd(h, k, v, w_h, w_k, eps: float, t_begin: int = 0, t_end: int | None = None) -> dict:
    """fp64 out [n, d], alpha, rstd_h, rstd_k, dot, z_fused [n] for tokens [t_begin, t_end)."""
    lib = _load()
    h, k, v = (np.ascontiguousarray(x) for x in (h, k, v))
    dt = _dtype_code(h)
    assert _dtype_code(k) == dt and _dtype_code(v) == dt
    wh = np.ascontiguousarray(w_h, dtype=np.float32)
    wk = np.ascontiguousarray(w_k, dtype=np.float32)
    T, d = h.shape
    t_end = T if t_end is None else t_end
    n = t_end - t_begin
    res = {name: np.zeros(n, dtype=np.float64) for name in ("alpha", "rstd_h", "rstd_k", "dot", "z_fused")}
    res["out"] = np.zeros((n, d), dtype=np.float64)
    rc = lib.eo_gate_fwd(_ptr(h), _ptr(k), _ptr(v), dt, _ptr(wh), _ptr(wk), T, d, float(eps), t_begin, t_end,
                         _ptr(res["out"]), _ptr(res["alpha"]), _ptr(res["rstd_h"]), _ptr(res["rstd_k"]),
                         _ptr(res["dot"]), _ptr(res["z_fused"]))
    _check(rc, "gate_fwd")
    return res


def gate_bwd(dout, h, k, v, w_h, w_k, eps: float, t_begin: int = 0, t_end: int | None = None) -> dict:
    """fp64 dh, dk, dv [n, d], dweight [d] (sum over the token range) and dweight_abs [d] (sum of |terms|)."""
    lib = _load()
    g, h, k, v = (np.ascontiguousarray(x) for x in (dout, h, k, v))
    dt = _dtype_code(h)
    assert all(_dtype_code(x) == dt for x in (g, k, v))
    wh = np.ascontiguousarray(w_h, dtype=np.float32)
    wk = np.ascontiguousarray(w_k, dtype=np.float32)
    T, d = h.shape
    t_end = T if t_end is None else t_end
    n = t_end - t_begin
    res = {name: np.zeros((n, d), dtype=np.float64) for name in ("dh", "dk", "dv")}
    res["dweight"] = np.zeros(d, dtype=np.float64)
    res["dweight_abs"] = np.zeros(d, dtype=np.float64)
    rc = lib.eo_gate_bwd(_ptr(g), _ptr(h), _ptr(k), _ptr(v), dt, _ptr(wh), _ptr(wk), T, d, float(eps), t_begin,
                         t_end, _ptr(res["dh"]), _ptr(res["dk"]), _ptr(res["dv"]), _ptr(res["dweight"]),
                         _ptr(res["dweight_abs"]))
    _check(rc, "gate_bwd")
    return res


def grad_w_reduce(partial, w_h=None, w_k=None) -> dict:
    """S = sum_p partial[p] (fp64) and, with weights, the increments S*w_k (for w_h) and S*w_h (for w_k)."""
    lib = _load()
    part = np.ascontiguousarray(partial, dtype=np.float32)
    P, d = part.shape
    S = np.zeros(d, dtype=np.float64)
    inc_h = np.zeros(d, dtype=np.float64)
    inc_k = np.zeros(d, dtype=np.float64)
    wh = None if w_h is None else np.ascontiguousarray(w_h, dtype=np.float32)
    wk = None if w_k is None else np.ascontiguousarray(w_k, dtype=np.float32)
    rc = lib.eo_grad_w_reduce(_ptr(part), P, d, _ptr(wh), _ptr(wk), _ptr(S), _ptr(inc_h), _ptr(inc_k))
    _check(rc, "grad_w_reduce")
    out = {"S": S}
    if wh is not None:
        out["inc_h"], out["inc_k"] = inc_h, inc_k
    return out


def gate_hc_fwd(x, kv, w_h, w_k, eps: float, clamp: float, t_begin: int = 0, t_end: int | None = None) -> dict:
    """Multi-branch gate: x [T, hc, d], kv [T, hc+1, d], w_h/w_k [hc, d] -> fp64 out [n, hc, d] and
    gate, rstd_x, rstd_k, dot [n, hc]."""
    lib = _load()
    x, kv = np.ascontiguousarray(x), np.ascontiguousarray(kv)
    dt = _dtype_code(x)
    assert _dtype_code(kv) == dt
    T, hc, d = x.shape
    assert kv.shape == (T, hc + 1, d)
    wh = np.ascontiguousarray(w_h, dtype=np.float32).reshape(hc, d)
    wk = np.ascontiguousarray(w_k, dtype=np.float32).reshape(hc, d)
    t_end = T if t_end is None else t_end
    n = t_end - t_begin
    res = {name: np.zeros((n, hc), dtype=np.float64) for name in ("gate", "rstd_x", "rstd_k", "dot")}
    res["out"] = np.zeros((n, hc, d), dtype=np.float64)
    rc = lib.eo_gate_hc_fwd(_ptr(x), _ptr(kv), dt, _ptr(wh), _ptr(wk), T, hc, d, float(eps), float(clamp), t_begin,
                            t_end, _ptr(res["out"]), _ptr(res["gate"]), _ptr(res["rstd_x"]), _ptr(res["rstd_k"]),
                            _ptr(res["dot"]))
    _check(rc, "gate_hc_fwd")
    return res


def gate_hc_bwd(dout, x, kv, w_h, w_k, eps: float, clamp: float, t_begin: int = 0, t_end: int | None = None) -> dict:
    """fp64 dx [n, hc, d], dkv [n, hc+1, d], dweight and dweight_abs [hc, d]."""
    lib = _load()
    g, x, kv = (np.ascontiguousarray(a) for a in (dout, x, kv))
    dt = _dtype_code(x)
    assert _dtype_code(g) == dt and _dtype_code(kv) == dt
    T, hc, d = x.shape
    wh = np.ascontiguousarray(w_h, dtype=np.float32).reshape(hc, d)
    wk = np.ascontiguousarray(w_k, dtype=np.float32).reshape(hc, d)
    t_end = T if t_end is None else t_end
    n = t_end - t_begin
    res = {"dx": np.zeros((n, hc, d), dtype=np.float64), "dkv": np.zeros((n, hc + 1, d), dtype=np.float64),
           "dweight": np.zeros((hc, d), dtype=np.float64), "dweight_abs": np.zeros((hc, d), dtype=np.float64)}
    rc = lib.eo_gate_hc_bwd(_ptr(g), _ptr(x), _ptr(kv), dt, _ptr(wh), _ptr(wk), T, hc, d, float(eps), float(clamp),
                            t_begin, t_end, _ptr(res["dx"]), _ptr(res["dkv"]), _ptr(res["dweight"]),
                            _ptr(res["dweight_abs"]))
    _check(rc, "gate_hc_bwd")
    return res


def sinkhorn_momentum(grad, momentum, beta1: float, nesterov: bool) -> dict:
    """m' = beta1 m + g; input = g + beta1 m' (nesterov) or m' -> fp64 {"momentum", "input"}."""
    lib = _load()
    g = np.ascontiguousarray(grad)
    m = np.ascontiguousarray(momentum, dtype=np.float32)
    n = g.size
    out = {"momentum": np.zeros(n, dtype=np.float64), "input": np.zeros(n, dtype=np.float64)}
    rc = lib.eo_sinkhorn_momentum(_ptr(g), _dtype_code(g), _ptr(m), n, float(beta1), int(bool(nesterov)),
                                  _ptr(out["momentum"]), _ptr(out["input"]))
    _check(rc, "sinkhorn_momentum")
    return {k: v.reshape(g.shape) for k, v in out.items()}


def sinkhorn_step(matrix, row_scale, col_scale, eps: float, r_begin: int = 0, r_end: int | None = None) -> dict:
    """Row step over rows [r_begin, r_end): fp64 row_norm, row_scale [n] and col_sumsq [head_dim]."""
    lib = _load()
    mat = np.ascontiguousarray(matrix, dtype=np.float32)
    rs = np.ascontiguousarray(row_scale, dtype=np.float32)
    cs = np.ascontiguousarray(col_scale, dtype=np.float32)
    R, D = mat.shape
    r_end = R if r_end is None else r_end
    out = {"row_norm": np.zeros(r_end - r_begin), "row_scale": np.zeros(r_end - r_begin), "col_sumsq": np.zeros(D)}
    rc = lib.eo_sinkhorn_step(_ptr(mat), _ptr(rs), _ptr(cs), R, D, float(eps), r_begin, r_end, _ptr(out["row_norm"]),
                              _ptr(out["row_scale"]), _ptr(out["col_sumsq"]))
    _check(rc, "sinkhorn_step")
    return out


def sinkhorn_col_update(col_sumsq, col_scale, eps: float) -> np.ndarray:
    lib = _load()
    s = np.ascontiguousarray(col_sumsq, dtype=np.float64)
    cs = np.ascontiguousarray(col_scale, dtype=np.float32)
    out = np.zeros(cs.size)
    _check(lib.eo_sinkhorn_col_update(_ptr(s), _ptr(cs), cs.size, float(eps), _ptr(out)), "sinkhorn_col_update")
    return out


def sinkhorn_finalize(matrix, row_scale, col_scale, eps: float, alpha: float) -> np.ndarray:
    lib = _load()
    mat = np.ascontiguousarray(matrix, dtype=np.float32)
    rs = np.ascontiguousarray(row_scale, dtype=np.float32)
    cs = np.ascontiguousarray(col_scale, dtype=np.float32)
    R, D = mat.shape
    out = np.zeros((R, D))
    rc = lib.eo_sinkhorn_finalize(_ptr(mat), _ptr(rs), _ptr(cs), R, D, float(eps), float(alpha), _ptr(out))
    _check(rc, "sinkhorn_finalize")
    return out


def _conv_common(v, norm_w, conv_w, bias, seq_offsets):
    v = np.ascontiguousarray(v)
    T, d = v.shape
    nw = np.ascontiguousarray(norm_w, dtype=np.float32).reshape(d)
    cw = np.ascontiguousarray(conv_w, dtype=np.float32)
    assert cw.ndim == 2 and cw.shape[0] == d
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32).reshape(d)
    offs = np.ascontiguousarray(seq_offsets, dtype=np.int64)
    return v, T, d, nw, cw, b, offs


def short_conv_fwd(v, h, norm_w, conv_w, bias, seq_offsets, dilation: int, eps: float, t_begin: int = 0,
                   t_end: int | None = None) -> dict:
    """out = H + SiLU(c) + V~ with c the causal depthwise conv of RMSNorm(V~): fp64 out, c [n, d], rstd [n]."""
    lib = _load()
    v, T, d, nw, cw, b, offs = _conv_common(v, norm_w, conv_w, bias, seq_offsets)
    dt = _dtype_code(v)
    if h is not None:
        h = np.ascontiguousarray(h)
        assert _dtype_code(h) == dt and h.shape == v.shape
    t_end = T if t_end is None else t_end
    n = t_end - t_begin
    res = {"out": np.zeros((n, d)), "c": np.zeros((n, d)), "rstd": np.zeros(n)}
    rc = lib.eo_short_conv_fwd(_ptr(v), _ptr(h), dt, _ptr(nw), _ptr(cw), _ptr(b), _ptr(offs), offs.size - 1, T, d,
                               cw.shape[1], int(dilation), float(eps), t_begin, t_end, _ptr(res["out"]),
                               _ptr(res["c"]), _ptr(res["rstd"]))
    _check(rc, "short_conv_fwd")
    return res


def short_conv_bwd(g, v, norm_w, conv_w, bias, seq_offsets, dilation: int, eps: float, t_begin: int = 0,
                   t_end: int | None = None) -> dict:
    """fp64 dv [n, d], dconv_w [d, w], dbias [d], dnorm_w [d] over tokens [t_begin, t_end), and the
    matching *_abs magnitude sums."""
    lib = _load()
    v, T, d, nw, cw, b, offs = _conv_common(v, norm_w, conv_w, bias, seq_offsets)
    g = np.ascontiguousarray(g)
    dt = _dtype_code(v)
    assert _dtype_code(g) == dt and g.shape == v.shape
    t_end = T if t_end is None else t_end
    n, w = t_end - t_begin, cw.shape[1]
    res = {"dv": np.zeros((n, d)), "dconv_w": np.zeros((d, w)), "dbias": np.zeros(d), "dnorm_w": np.zeros(d),
           "dv_abs": np.zeros((n, d)), "dconv_w_abs": np.zeros((d, w)), "dbias_abs": np.zeros(d),
           "dnorm_w_abs": np.zeros(d)}
    rc = lib.eo_short_conv_bwd(_ptr(g), _ptr(v), dt, _ptr(nw), _ptr(cw), _ptr(b), _ptr(offs), offs.size - 1, T, d,
                               w, int(dilation), float(eps), t_begin, t_end, _ptr(res["dv"]), _ptr(res["dconv_w"]),
                               _ptr(res["dbias"]), _ptr(res["dnorm_w"]), _ptr(res["dv_abs"]),
                               _ptr(res["dconv_w_abs"]), _ptr(res["dbias_abs"]), _ptr(res["dnorm_w_abs"]))
    _check(rc, "short_conv_bwd")
    return res
