"""Shared helpers of the GPU parity tests: host copies, tolerances, threaded oracle calls."""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np
import torch

import oracle

# Tolerances (the gate's output contract):
#   bf16 outputs (out, dh, dk, dv): |gpu - ref| <= 1e-3 + 2e-2 * |ref|
#   fp32 alpha: |gpu - ref| <= 1e-4
#   rstd_h, rstd_k: relative 1e-4
#   dot: |gpu - ref| <= 2e-5 * sum_i |h_i w_i k_i| + 1e-6   (fp32 accumulation of d terms)
#   dweight, grad_w: |gpu - ref| <= 1e-4 * sum_t |c_t h_t,i k_t,i| + 1e-7   (fp32 accumulation over T)
#   fp32 gate outputs (the tiny workload): |gpu - ref| <= 1e-5 * rowmax|ref| + 1e-4 * |ref|
BF16_ATOL, BF16_RTOL = 1e-3, 2e-2
ALPHA_ATOL = 1e-4
RSTD_RTOL = 1e-4


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a CUDA tensor: fp32 as float32, bf16 as raw uint16 bits (the oracle's input form)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close_bf16(got: torch.Tensor, ref: np.ndarray, what: str):
    g = as_f64(got)
    bad = np.abs(g - ref) > BF16_ATOL + BF16_RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst " \
                          f"{np.abs(g - ref)[bad].max():.3g} at {np.argwhere(bad)[0]}"


def assert_close_rows(got: torch.Tensor, ref: np.ndarray, what: str, row_tol=1e-5, rtol=1e-4):
    g = as_f64(got)
    scale = np.abs(ref).max(axis=-1, keepdims=True)
    bad = np.abs(g - ref) > row_tol * scale + rtol * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} outside tolerance; worst {np.abs(g - ref)[bad].max():.3g}"


def check_stats(alpha, rh, rk, dot, f, h, k, w, what=""):
    """alpha/rstd/dot of the GPU against the oracle's fp64 forward (host arrays h, k as oracle inputs)."""
    a = as_f64(alpha)
    assert np.abs(a - f["alpha"]).max() <= ALPHA_ATOL, f"{what} alpha: {np.abs(a - f['alpha']).max()}"
    np.testing.assert_allclose(as_f64(rh), f["rstd_h"], rtol=RSTD_RTOL, err_msg=f"{what} rstd_h")
    np.testing.assert_allclose(as_f64(rk), f["rstd_k"], rtol=RSTD_RTOL, err_msg=f"{what} rstd_k")
    hf, kf = _f64(h), _f64(k)
    scale = np.abs(hf * w[None, :].astype(np.float64) * kf).sum(-1)
    ddot = np.abs(as_f64(dot) - f["dot"])
    assert (ddot <= 2e-5 * scale + 1e-6).all(), f"{what} dot: worst {(ddot / (scale + 1e-30)).max():.3g} rel"


def _f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


def oracle_gate_fwd(h, k, v, w_h, w_k, eps):
    """The oracle's forward over all rows, split across host threads (tokens are independent)."""
    T = h.shape[0]
    n = _threads()
    bounds = [(T * i // n, T * (i + 1) // n) for i in range(n)]
    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(lambda b: oracle.gate_fwd(h[b[0]:b[1]], k[b[0]:b[1]], v[b[0]:b[1]], w_h, w_k, eps),
                            bounds))
    return {key: np.concatenate([p[key] for p in parts]) for key in parts[0]}


def oracle_gate_bwd(g, h, k, v, w_h, w_k, eps):
    """The oracle's backward over all rows, threaded; dweight sums the per-thread ranges in order."""
    T = h.shape[0]
    n = _threads()
    bounds = [(T * i // n, T * (i + 1) // n) for i in range(n)]
    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(lambda b: oracle.gate_bwd(g[b[0]:b[1]], h[b[0]:b[1]], k[b[0]:b[1]], v[b[0]:b[1]],
                                                      w_h, w_k, eps), bounds))
    out = {key: np.concatenate([p[key] for p in parts]) for key in ("dh", "dk", "dv")}
    out["dweight"] = np.sum([p["dweight"] for p in parts], axis=0)
    out["dweight_abs"] = np.sum([p["dweight_abs"] for p in parts], axis=0)
    return out


def _bf16_bad(g: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Elements of a bf16 result (raw bits) outside the bf16 output tolerance of an fp64 reference."""
    return np.abs(_f64(g) - ref) > BF16_ATOL + BF16_RTOL * np.abs(ref)


def check_gate_train_by_partials(t: dict, r: dict, eps: float, what: str, group_tokens: int = 16384):
    """Every element of the gate's forward and backward outputs and every weight-gradient partial of a
    bf16 training step (`r`, on the device, made from the inputs `t`) against the oracle.

    The oracle runs once per partial, over exactly that partial's token range, so each partial is
    compared with the oracle's sum over the same tokens; out, the statistics, dh, dk and dv of those
    tokens are compared element by element.  Host copies are taken a group of partials at a time to
    bound host memory, and the partials of a group run on all host threads.  Finally the reduced
    dweight is compared with the oracle's sum over all partials in order."""
    T, d = t["h"].shape
    P = r["part"].shape[0]
    C = -(-T // P) if T else 1
    w_h, w_k = host_bits(t["w_h"]), host_bits(t["w_k"])
    w = (w_h * w_k).astype(np.float64)
    parts = as_f64(r["part"])
    total, total_abs = np.zeros(d), np.zeros(d)
    per_group = max(1, group_tokens // C)
    n = _threads()
    for g0 in range(0, P, per_group):
        p1 = min(P, g0 + per_group)
        t0, t1 = g0 * C, min(T, p1 * C)
        if t0 >= T:
            assert (parts[g0:] == 0).all(), f"{what}: partials past the last token are not zero"
            break
        x = {k: host_bits(t[k][t0:t1]) for k in ("h", "k", "v", "dout")}
        y = {k: host_bits(r[k][t0:t1]) for k in ("out", "dh", "dk", "dv")}
        s = {k: as_f64(r[k][t0:t1]) for k in ("alpha", "rstd_h", "rstd_k", "dot")}

        def task(p):
            a, b = p * C - t0, min(T, (p + 1) * C) - t0
            if a >= b:
                return p, np.zeros(d), np.zeros(d)
            f = oracle.gate_fwd(x["h"], x["k"], x["v"], w_h, w_k, eps, a, b)
            bw = oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], w_h, w_k, eps, a, b)
            assert np.abs(s["alpha"][a:b] - f["alpha"]).max() <= ALPHA_ATOL, f"{what} alpha, partial {p}"
            for key in ("rstd_h", "rstd_k"):
                assert (np.abs(s[key][a:b] - f[key]) <= RSTD_RTOL * np.abs(f[key])).all(), f"{what} {key}, p {p}"
            scale = np.abs(_f64(x["h"][a:b]) * w[None, :] * _f64(x["k"][a:b])).sum(-1)
            assert (np.abs(s["dot"][a:b] - f["dot"]) <= 2e-5 * scale + 1e-6).all(), f"{what} dot, partial {p}"
            for key, ref in (("out", f["out"]), ("dh", bw["dh"]), ("dk", bw["dk"]), ("dv", bw["dv"])):
                bad = _bf16_bad(y[key][a:b], ref)
                assert not bad.any(), f"{what} {key}: {bad.sum()} of {bad.size} outside tolerance in partial {p}"
            got = parts[p]
            assert (np.abs(got - bw["dweight"]) <= 1e-4 * bw["dweight_abs"] + 1e-7).all(), f"{what} partial {p}"
            return p, bw["dweight"], bw["dweight_abs"]

        with ThreadPoolExecutor(n) as ex:
            for _, dw_p, abs_p in ex.map(task, range(g0, p1)):  # in partial order
                total += dw_p
                total_abs += abs_p
    dw = as_f64(r["dw"])
    assert (np.abs(dw - total) <= 1e-4 * total_abs + 1e-7).all(), f"{what}: reduced dweight"
