"""Device-side seeded draws of the large synthetic tensors (activations, embedding tables).

Drawing multi-GB tensors on the host would dominate test and benchmark time, so
they are drawn on the GPU with torch's seeded generator.  Whatever a check
needs from them is copied back to the host and handed to the oracle as input.
"""
from __future__ import annotations

import numpy as np
import torch

from .workloads import GateWorkload, HashGatherWorkload

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def normal_tensor(shape, seed: int, mean: float, std: float, dtype: str, device, chunk_rows: int = 1 << 20):
    """A [rows, cols] tensor of N(mean, std) draws in `dtype`, drawn chunk by chunk (bounded fp32 scratch)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & ((1 << 63) - 1))
    rows, cols = shape
    out = torch.empty((rows, cols), dtype=_DT[dtype], device=device)
    step = max(1, min(rows, chunk_rows * 64 // max(cols, 1)))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = torch.randn((r1 - r0, cols), generator=g, device=device, dtype=torch.float32)
        out[r0:r1] = (x * std + mean).to(out.dtype)
    return out


def gate_device_inputs(w: GateWorkload, device, with_dout: bool = True):
    """h, k, v (and dout) [T, d] N(0, 1) in the workload dtype; w_h, w_k [d] N(1, 0.1) fp32."""
    out = {}
    names = ("h", "k", "v", "dout") if with_dout else ("h", "k", "v")
    for i, name in enumerate(names):
        out[name] = normal_tensor((w.T, w.d), w.seed + 1000 * (i + 1), 0.0, 1.0, w.dtype, device)
    out["w_h"] = normal_tensor((1, w.d), w.seed + 7001, 1.0, 0.1, "f32", device).reshape(w.d)
    out["w_k"] = normal_tensor((1, w.d), w.seed + 7002, 1.0, 0.1, "f32", device).reshape(w.d)
    return out


def gate_inputs_to_device(host: dict, dtype: str, device):
    """Copy host draws (see `workloads.gate_host_inputs`) to the device as torch tensors."""
    out = {}
    for name, arr in host.items():
        if arr.dtype == np.uint16:
            t = torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(arr))
        out[name] = t.to(device)
    return out


def hash_table(w: HashGatherWorkload, device):
    """The concatenated [sum(primes), row_dim] table, on the device."""
    if w.table_host is not None:
        return torch.from_numpy(np.ascontiguousarray(w.table_host)).to(device)
    return normal_tensor((w.spec.total_rows, w.row_dim), w.table_seed, 0.0, w.table_std, w.dtype, device)
