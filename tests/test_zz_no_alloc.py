"""The allocation-free backward + reduction entry point, engram_gate_bwd_reduce_noalloc.

It serves callers that cannot allocate device memory: their device memory already
belongs to a framework allocator or to an arena reserved at start-up, or their
serving loop forbids allocation (cudaMalloc and cudaFree can synchronise the device).
Instead of a caller buffer it keeps the weight-gradient partials in a fixed device
array of the library.  These checks call it through the C ABI (ctypes, no binding
code) and compare it with the existing pair engram_gate_bwd + engram_grad_w_reduce
on two calls in a row, so that anything a first call leaves in the shared array
would show up in the second.  This file is collected last on purpose.
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


def _inputs(seed, T, d):
    wl = W.GateWorkload(name="noalloc", T=T, d=d, dtype="bf16", seed=seed)
    t = SD.gate_device_inputs(wl, DEV)
    t["w_fused"] = ecm.fuse_weight(t["w_h"], t["w_k"])
    _, *st = ecm.gate_fwd(t["h"], t["k"], t["v"], t["w_fused"], wl.eps)
    t["stats"] = st
    return t


def _existing(t, gh0, gk0):
    dh, dk, dv, part = ecm.gate_bwd(t["dout"], t["h"], t["k"], t["v"], t["w_fused"], *t["stats"])
    gh, gk = gh0.clone(), gk0.clone()
    dw = ecm.grad_w_reduce(part, w_h=t["w_h"], w_k=t["w_k"], grad_w_h=gh, grad_w_k=gk)
    scale = part.double().abs().sum(0)  # magnitude of the summed terms, for the fp32 tolerance
    return dh, dk, dv, dw, gh, gk, scale


def _noalloc(entry, t, gh0, gk0):
    T, d = t["h"].shape
    dh, dk, dv = (torch.empty_like(t["h"]) for _ in range(3))
    dw = torch.empty(d, dtype=torch.float32, device=DEV)
    gh, gk = gh0.clone(), gk0.clone()
    a, rh, rk, dot = t["stats"]
    st = entry(_ptr(t["dout"]), _ptr(t["h"]), _ptr(t["k"]), _ptr(t["v"]), 1, _ptr(t["w_fused"]), _ptr(a), _ptr(rh),
               _ptr(rk), _ptr(dot), T, d, _ptr(dh), _ptr(dk), _ptr(dv), _ptr(dw), _ptr(t["w_h"]), _ptr(t["w_k"]),
               _ptr(gh), _ptr(gk), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, ecm.load_library().engram_last_error_string()
    return dh, dk, dv, dw, gh, gk


def _close(got, ref, scale, what):
    g, r, s = got.double().cpu().numpy(), ref.double().cpu().numpy(), scale.cpu().numpy()
    bad = np.abs(g - r) > 1e-4 * s + 1e-7
    assert not bad.any(), f"{what}: {bad.sum()} values outside tolerance"


def test_matches_existing_entry_points_on_two_calls_in_a_row(cuda_lib):
    lib = ecm.load_library()
    entry = _c_entry(lib)
    d = 4096
    gh0 = torch.linspace(-1, 1, d, device=DEV)
    gk0 = torch.linspace(2, -2, d, device=DEV)
    # the second call has fewer tokens, hence fewer partial rows, than the first
    for seed, T in ((11, 9000), (12, 3001)):
        t = _inputs(seed, T, d)
        ref = _existing(t, gh0, gk0)
        got = _noalloc(entry, t, gh0, gk0)
        torch.cuda.synchronize()
        for name, g_, r_ in zip(("dh", "dk", "dv"), got[:3], ref[:3]):
            H.assert_close_bf16(g_, H.as_f64(r_), name)
        scale = ref[6]
        _close(got[3], ref[3], scale, "dweight_fused")
        w_abs_k, w_abs_h = t["w_k"].double().abs(), t["w_h"].double().abs()
        _close(got[4], ref[4], scale * w_abs_k + gh0.double().abs() * 1e-3, "grad_w_h")
        _close(got[5], ref[5], scale * w_abs_h + gk0.double().abs() * 1e-3, "grad_w_k")
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
