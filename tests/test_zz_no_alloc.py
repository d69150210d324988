"""The allocation-free backward + reduction entry point, engram_gate_bwd_reduce_noalloc.

It serves callers that cannot allocate device memory: their device memory already
belongs to a framework allocator or to an arena reserved at start-up, or their
serving loop forbids allocation (cudaMalloc and cudaFree can synchronise the device).
Instead of a caller buffer it keeps the weight-gradient partials in a fixed device
array of the library.  These checks call it through the C ABI (ctypes, no binding
code) and compare it, bit for bit, with the existing pair engram_gate_bwd +
engram_grad_w_reduce on consecutive calls, so that anything a call leaves in the
shared array would show up in the next; one call is also checked against the
oracle.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import engram_conditional_memory_gb300 as ecm
from synth import device as SD
from synth import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ERR_SHAPE = 2


def _c_entry(lib):
    f = lib.engram_gate_bwd_reduce_noalloc
    f.restype = ctypes.c_int
    p = ctypes.c_void_p
    f.argtypes = [p, p, p, p, ctypes.c_int, p, p, p, p, p, ctypes.c_int64, ctypes.c_int32, p, p, p, p, p, p, p, p,
                  p]
    return f


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _inputs(seed, T, d, dtype="bf16"):
    wl = W.GateWorkload(name="noalloc", T=T, d=d, dtype=dtype, seed=seed)
    t = SD.gate_device_inputs(wl, DEV)
    t["w_fused"] = ecm.fuse_weight(t["w_h"], t["w_k"])
    _, *st = ecm.gate_fwd(t["h"], t["k"], t["v"], t["w_fused"], wl.eps)
    t["stats"] = st
    t["eps"] = wl.eps
    return t


def _existing(t, gh0, gk0):
    dh, dk, dv, part = ecm.gate_bwd(t["dout"], t["h"], t["k"], t["v"], t["w_fused"], *t["stats"])
    gh, gk = gh0.clone(), gk0.clone()
    dw = ecm.grad_w_reduce(part, w_h=t["w_h"], w_k=t["w_k"], grad_w_h=gh, grad_w_k=gk)
    return dh, dk, dv, dw, gh, gk


def _noalloc(entry, t, gh0, gk0):
    T, d = t["h"].shape
    dh, dk, dv = (torch.empty_like(t["h"]) for _ in range(3))
    dw = torch.empty(d, dtype=torch.float32, device=DEV)
    gh, gk = gh0.clone(), gk0.clone()
    a, rh, rk, dot = t["stats"]
    dt = 1 if t["h"].dtype == torch.bfloat16 else 0
    st = entry(_ptr(t["dout"]), _ptr(t["h"]), _ptr(t["k"]), _ptr(t["v"]), dt, _ptr(t["w_fused"]), _ptr(a), _ptr(rh),
               _ptr(rk), _ptr(dot), T, d, _ptr(dh), _ptr(dk), _ptr(dv), _ptr(dw), _ptr(t["w_h"]), _ptr(t["w_k"]),
               _ptr(gh), _ptr(gk), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, ecm.load_library().engram_last_error_string()
    return dh, dk, dv, dw, gh, gk


NAMES = ("dh", "dk", "dv", "dweight_fused", "grad_w_h", "grad_w_k")


def test_matches_existing_entry_points_on_two_calls_in_a_row(cuda_lib):
    """Bitwise equal to engram_gate_bwd + engram_grad_w_reduce (the same kernels, the same P and the
    same ordered reduction), call after call: a partial row left stale in the shared array by the
    first call, which has more tokens and so more partial rows, would change the second call's sums.
    The second call is also compared with the oracle."""
    lib = ecm.load_library()
    entry = _c_entry(lib)
    d = 4096
    gh0 = torch.linspace(-1, 1, d, device=DEV)
    gk0 = torch.linspace(2, -2, d, device=DEV)
    for seed, T in ((11, 9000), (12, 3001)):
        t = _inputs(seed, T, d)
        ref = _existing(t, gh0, gk0)
        got = _noalloc(entry, t, gh0, gk0)
        torch.cuda.synchronize()
        for name, g_, r_ in zip(NAMES, got, ref):
            assert torch.equal(g_, r_), f"T = {T}: {name} differs from the caller-buffer path"
    # the second call against the oracle, within the gate's tolerances
    x = {n: H.host_bits(t[n]) for n in ("dout", "h", "k", "v", "w_h", "w_k")}
    b = H.oracle_gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], t["eps"])
    for name, g_ in zip(("dh", "dk", "dv"), got[:3]):
        H.assert_close_bf16(g_, b[name], name)
    dw = H.as_f64(got[3])
    assert (np.abs(dw - b["dweight"]) <= 1e-4 * b["dweight_abs"] + 1e-7).all(), "dweight_fused vs the oracle"
    assert ecm.device_status() == 0


def test_empty_batch_and_fp32_match_existing_entry_points(cuda_lib):
    """An empty bf16 batch (partials all zero: dweight_fused = 0, the accumulated gradients kept) and
    an fp32 batch, each bitwise equal to the caller-buffer path, again on consecutive calls."""
    entry = _c_entry(ecm.load_library())
    for seed, T, d, dtype in ((13, 0, 1024, "bf16"), (14, 777, 1024, "f32"), (15, 0, 1024, "bf16")):
        gh0 = torch.linspace(-1, 1, d, device=DEV)
        gk0 = torch.linspace(3, -1, d, device=DEV)
        t = _inputs(seed, T, d, dtype)
        ref = _existing(t, gh0, gk0)
        got = _noalloc(entry, t, gh0, gk0)
        torch.cuda.synchronize()
        for name, g_, r_ in zip(NAMES, got, ref):
            assert torch.equal(g_, r_), f"T = {T} {dtype}: {name} differs from the caller-buffer path"
        if T == 0:
            assert (got[3] == 0).all() and torch.equal(got[4], gh0) and torch.equal(got[5], gk0)
    assert ecm.device_status() == 0


def test_rejects_sizes_beyond_its_scratch(cuda_lib):
    entry = _c_entry(ecm.load_library())
    small = torch.zeros((4, 8192), dtype=torch.bfloat16, device=DEV)
    stat = torch.zeros(4, dtype=torch.float32, device=DEV)
    w = torch.zeros(8192, dtype=torch.float32, device=DEV)
    # T = 16384, d = 8192 needs 1024 x 8192 x 4 B = 32 MiB of partials: refused on the host, nothing launched
    st = entry(*(_ptr(small) for _ in range(4)), 1, _ptr(w), *(_ptr(stat) for _ in range(4)), 16384, 8192,
               *(_ptr(small) for _ in range(3)), _ptr(w), None, None, None, None, None)
    assert st == ERR_SHAPE
    assert b"bytes this entry point holds" in ecm.load_library().engram_last_error_string()
