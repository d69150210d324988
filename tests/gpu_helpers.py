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
