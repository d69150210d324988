"""GPU parity of the gate path (fold, forward, backward, weight-gradient reduction) against the CPU oracle.

Every comparison goes through the C ABI (via the thin binding).  Sizes: the tiny
fp32 workload; the T = 8192, d = 2048 and T = 16384, d = 4096 bf16 workloads in
full; the d = 7168 sweep (T = 4096, 32768, 131072 and a ragged 64-sequence pack)
element by element, each weight-gradient partial against the oracle over its own
token range, plus properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import engram_conditional_memory_gb300 as ecm
import oracle
from synth import device as SD
from synth import generators as G
from synth import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _status_clean(cuda_lib):
    ecm.device_status(clear=True)
    yield
    assert ecm.device_status() == 0, "a kernel reported a device-side error"


def _train_step(t, eps, P=None):
    wf = ecm.fuse_weight(t["w_h"], t["w_k"])
    out, a, rh, rk, dot = ecm.gate_fwd(t["h"], t["k"], t["v"], wf, eps)
    dh, dk, dv, part = ecm.gate_bwd(t["dout"], t["h"], t["k"], t["v"], wf, a, rh, rk, dot, P=P)
    dw = ecm.grad_w_reduce(part)
    return dict(wf=wf, out=out, alpha=a, rstd_h=rh, rstd_k=rk, dot=dot, dh=dh, dk=dk, dv=dv, part=part, dw=dw)


def _host(t):
    return {n: H.host_bits(x) for n, x in t.items()}


def test_fuse_weight_matches_fp32_product():
    w_h = torch.from_numpy(G.normal(1, 1000, 1, 0.1).astype(np.float32)).to(DEV)
    w_k = torch.from_numpy(G.normal(2, 1000, 1, 0.1).astype(np.float32)).to(DEV)
    got = ecm.fuse_weight(w_h, w_k).cpu().numpy()
    ref = oracle.fuse_weight(w_h.cpu().numpy(), w_k.cpu().numpy())
    # the fp32 product is the correctly rounded fp64 product
    assert np.array_equal(got, ref.astype(np.float32))
    wb_h, wb_k = w_h.bfloat16(), w_k.bfloat16()
    got_b = ecm.fuse_weight(wb_h, wb_k).cpu().numpy()
    assert np.array_equal(got_b, oracle.fuse_weight(wb_h.float().cpu().numpy(), wb_k.float().cpu().numpy())
                          .astype(np.float32))


def test_tiny_fp32_workload():
    g = W.tiny_gate()
    x = W.gate_host_inputs(g)
    t = SD.gate_inputs_to_device(x, g.dtype, DEV)
    r = _train_step(t, g.eps)
    f = oracle.gate_fwd(x["h"], x["k"], x["v"], x["w_h"], x["w_k"], g.eps)
    b = oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], g.eps)
    H.check_stats(r["alpha"], r["rstd_h"], r["rstd_k"], r["dot"], f, x["h"], x["k"], x["w_h"] * x["w_k"], "tiny")
    H.assert_close_rows(r["out"], f["out"], "out")
    for name in ("dh", "dk", "dv"):
        H.assert_close_rows(r[name], b[name], name)
    dw = H.as_f64(r["dw"])
    assert (np.abs(dw - b["dweight"]) <= 1e-4 * b["dweight_abs"] + 1e-7).all()


@pytest.mark.parametrize("wl", [W.gate_fwd_2k(), W.gate_train_4k()], ids=lambda w: w.name)
def test_full_size_bf16_workloads(wl):
    t = SD.gate_device_inputs(wl, DEV)
    r = _train_step(t, wl.eps)
    x = _host(t)
    f = H.oracle_gate_fwd(x["h"], x["k"], x["v"], x["w_h"], x["w_k"], wl.eps)
    H.check_stats(r["alpha"], r["rstd_h"], r["rstd_k"], r["dot"], f, x["h"], x["k"], x["w_h"] * x["w_k"], wl.name)
    H.assert_close_bf16(r["out"], f["out"], "out")
    b = H.oracle_gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], wl.eps)
    for name in ("dh", "dk", "dv"):
        H.assert_close_bf16(r[name], b[name], name)
    dw = H.as_f64(r["dw"])
    assert (np.abs(dw - b["dweight"]) <= 1e-4 * b["dweight_abs"] + 1e-7).all()


SWEEP = [W.gate_sweep_7k(4096), W.gate_sweep_7k(32768), W.gate_sweep_7k(131072), W.gate_ragged_7k()]


@pytest.mark.parametrize("wl", SWEEP, ids=lambda w: w.name)
def test_large_hidden_sweep_every_element(wl):
    t = SD.gate_device_inputs(wl, DEV)
    r = _train_step(t, wl.eps)
    torch.cuda.synchronize()
    H.check_gate_train_by_partials(t, r, wl.eps, wl.name)
    # the reduction is the sum of the partials (a property that holds at any size)
    S = r["part"].double().sum(0).cpu().numpy()
    A = r["part"].double().abs().sum(0).cpu().numpy()
    assert (np.abs(H.as_f64(r["dw"]) - S) <= 1e-5 * A + 1e-7).all()


@pytest.mark.parametrize("dtype,d,T", [("bf16", 8, 37), ("f32", 4, 5), ("bf16", 8192, 40), ("f32", 4096, 33),
                                       ("bf16", 1000, 100), ("bf16", 7168, 1), ("f32", 100, 257),
                                       ("bf16", 2048, 3)])
def test_edge_shapes(dtype, d, T):
    wl = W.GateWorkload(name="edge", T=T, d=d, dtype=dtype, seed=1234 + d + T)
    x = W.gate_host_inputs(wl)
    t = SD.gate_inputs_to_device(x, dtype, DEV)
    r = _train_step(t, wl.eps)
    f = oracle.gate_fwd(x["h"], x["k"], x["v"], x["w_h"], x["w_k"], wl.eps)
    b = oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], wl.eps)
    H.check_stats(r["alpha"], r["rstd_h"], r["rstd_k"], r["dot"], f, x["h"], x["k"], x["w_h"] * x["w_k"], "edge")
    check = H.assert_close_bf16 if dtype == "bf16" else H.assert_close_rows
    check(r["out"], f["out"], "out")
    for name in ("dh", "dk", "dv"):
        check(r[name], b[name], name)
    assert (np.abs(H.as_f64(r["dw"]) - b["dweight"]) <= 1e-4 * b["dweight_abs"] + 1e-7).all()


def test_empty_batch_writes_nothing_and_zero_partials():
    d = 64
    h = torch.empty((0, d), dtype=torch.bfloat16, device=DEV)
    wf = torch.ones(d, dtype=torch.float32, device=DEV)
    out, a, rh, rk, dot = ecm.gate_fwd(h, h, h, wf)
    assert out.shape == (0, d)
    part = torch.full((3, d), 7.0, dtype=torch.float32, device=DEV)
    ecm.gate_bwd(h, h, h, h, wf, a, rh, rk, dot, dw_partial=part, accumulate=True)
    assert (part == 7.0).all()  # accumulating no token keeps every row
    ecm.gate_bwd(h, h, h, h, wf, a, rh, rk, dot, dw_partial=part)
    assert (part == 0).all()
    with pytest.raises(ValueError):  # nothing to add to
        ecm.gate_bwd(h, h, h, h, wf, a, rh, rk, dot, P=3, accumulate=True)


def test_zero_key_gives_half_and_stats_are_optional():
    wl = W.GateWorkload(name="k0", T=300, d=512, dtype="bf16", seed=99)
    t = SD.gate_device_inputs(wl, DEV)
    wf = ecm.fuse_weight(t["w_h"], t["w_k"])
    k0 = torch.zeros_like(t["k"])
    out, a, rh, rk, dot = ecm.gate_fwd(t["h"], k0, t["v"], wf)
    assert (a == 0.5).all() and (dot == 0).all()
    assert torch.equal(out, (t["v"].float() * 0.5).bfloat16())
    out2, *_ = ecm.gate_fwd(t["h"], t["k"], t["v"], wf, save_for_backward=False)
    out3, *_ = ecm.gate_fwd(t["h"], t["k"], t["v"], wf)
    assert torch.equal(out2, out3)


def test_bitwise_determinism_across_runs_and_grids():
    wl = W.GateWorkload(name="det", T=5000, d=4096, dtype="bf16", seed=5)
    t = SD.gate_device_inputs(wl, DEV)
    base = _train_step(t, wl.eps)
    try:
        for cap in (1, 7, 151, 0):
            ecm.set_max_ctas(cap)
            r = _train_step(t, wl.eps)
            for name in ("out", "alpha", "dot", "dh", "dk", "dv", "part", "dw"):
                assert torch.equal(r[name], base[name]), (cap, name)
    finally:
        ecm.set_max_ctas(0)


@pytest.mark.parametrize("P", [1, 2, 333, 5000, 6000])
def test_partition_counts(P):
    wl = W.GateWorkload(name="parts", T=5000, d=256, dtype="bf16", seed=8)
    x = W.gate_host_inputs(wl)
    t = SD.gate_inputs_to_device(x, "bf16", DEV)
    r = _train_step(t, wl.eps, P=P)
    chunk = -(-wl.T // P)
    b = oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], wl.eps)
    assert (np.abs(H.as_f64(r["dw"]) - b["dweight"]) <= 1e-4 * b["dweight_abs"] + 1e-7).all()
    for p in (0, P - 1):
        t0, t1 = p * chunk, min(wl.T, (p + 1) * chunk)
        if t0 >= wl.T:
            assert (r["part"][p] == 0).all()
            continue
        ob = oracle.gate_bwd(x["dout"][t0:t1], x["h"][t0:t1], x["k"][t0:t1], x["v"][t0:t1], x["w_h"], x["w_k"],
                             wl.eps)
        assert (np.abs(H.as_f64(r["part"][p]) - ob["dweight"]) <= 1e-4 * ob["dweight_abs"] + 1e-7).all()


@pytest.mark.parametrize("P,d", [(1, 4), (7, 64), (1024, 4096), (3000, 4100), (0, 8)])
def test_grad_w_reduce_and_accumulate(P, d):
    part_h = G.normal(P * 1000 + d, P * d).astype(np.float32).reshape(P, d)
    w_h = G.normal(3, d, 1, 0.1).astype(np.float32)
    w_k = G.normal(4, d, 1, 0.1).astype(np.float32)
    gh0 = G.normal(5, d).astype(np.float32)
    gk0 = G.normal(6, d).astype(np.float32)
    part = torch.from_numpy(part_h).to(DEV)
    wh, wk = torch.from_numpy(w_h).to(DEV), torch.from_numpy(w_k).to(DEV)
    gh, gk = torch.from_numpy(gh0).to(DEV), torch.from_numpy(gk0).to(DEV)
    S = ecm.grad_w_reduce(part, w_h=wh, w_k=wk, grad_w_h=gh, grad_w_k=gk)
    ref = oracle.grad_w_reduce(part_h, w_h, w_k)
    scale = np.abs(part_h).sum(0) if P else np.zeros(d)
    assert (np.abs(H.as_f64(S) - ref["S"]) <= 1e-6 * scale + 1e-7).all()
    ecm.grad_w_reduce(part, want_dweight=False, w_h=wh, w_k=wk, grad_w_h=gh, grad_w_k=gk)
    tol = 1e-6 * (scale * 2.2) + 1e-6 * (np.abs(gh0) + 1)
    assert (np.abs(H.as_f64(gh) - (gh0 + 2 * ref["inc_h"])) <= tol).all()
    assert (np.abs(H.as_f64(gk) - (gk0 + 2 * ref["inc_k"])) <= tol).all()
    # bitwise reproducible
    S2 = ecm.grad_w_reduce(part)
    assert torch.equal(S, S2)


@pytest.mark.parametrize("P", [333, 6000])
def test_backward_accumulates_partials_over_micro_batches(P):
    """engram_gate_bwd then engram_gate_bwd_accumulate on one partial array: dh, dk, dv bitwise those of
    the plain call; each partial equals the oracle's sum over its token range in both micro-batches;
    partials with no token keep their rows; accumulating onto zeros is bitwise the plain call; and
    the result does not depend on the grid."""
    wa = W.GateWorkload(name="acc_a", T=5000, d=256, dtype="bf16", seed=21)
    wb = W.GateWorkload(name="acc_b", T=5000, d=256, dtype="bf16", seed=22)
    xa, xb = W.gate_host_inputs(wa), W.gate_host_inputs(wb)
    xb["w_h"], xb["w_k"] = xa["w_h"], xa["w_k"]  # one set of weights across the micro-batches
    ta, tb = (SD.gate_inputs_to_device(x, "bf16", DEV) for x in (xa, xb))
    wf = ecm.fuse_weight(ta["w_h"], ta["w_k"])

    def run(cap=0):
        ecm.set_max_ctas(cap)
        try:
            part = torch.empty((P, 256), dtype=torch.float32, device=DEV)
            outs = []
            for i, t in enumerate((ta, tb)):
                _, *st = ecm.gate_fwd(t["h"], t["k"], t["v"], wf, wa.eps)
                outs.append(ecm.gate_bwd(t["dout"], t["h"], t["k"], t["v"], wf, *st, P=P, dw_partial=part,
                                         accumulate=i > 0)[:3])
            return part, outs
        finally:
            ecm.set_max_ctas(0)

    part, outs = run()
    # the accumulating call writes dh, dk, dv exactly as the plain call does
    _, *st = ecm.gate_fwd(tb["h"], tb["k"], tb["v"], wf, wa.eps)
    plain = ecm.gate_bwd(tb["dout"], tb["h"], tb["k"], tb["v"], wf, *st, P=P)
    for got, ref in zip(outs[1], plain[:3]):
        assert torch.equal(got, ref)
    # onto zeros, the accumulating call is bitwise the plain call
    z = torch.zeros((P, 256), dtype=torch.float32, device=DEV)
    ecm.gate_bwd(tb["dout"], tb["h"], tb["k"], tb["v"], wf, *st, P=P, dw_partial=z, accumulate=True)
    assert torch.equal(z, plain[3])
    # each partial against the oracle over its token range in both micro-batches
    chunk = -(-5000 // P)
    got = H.as_f64(part)
    for p in sorted({0, 1, P // 2, P - 1}):
        t0, t1 = p * chunk, min(5000, (p + 1) * chunk)
        if t0 >= 5000:
            assert (part[p] == 0).all()  # written as zeros by the first call, kept by the second
            continue
        ref, mag = np.zeros(256), np.zeros(256)
        for x in (xa, xb):
            ob = oracle.gate_bwd(*(x[n][t0:t1] for n in ("dout", "h", "k", "v")), xa["w_h"], xa["w_k"], wa.eps)
            ref += ob["dweight"]
            mag += ob["dweight_abs"]
        assert (np.abs(got[p] - ref) <= 1e-4 * mag + 1e-7).all(), f"partial {p}"
    # grid independence, bitwise
    for cap in (1, 7, 151):
        part2, _ = run(cap)
        assert torch.equal(part2, part), cap


@pytest.mark.parametrize("dtype,wdtype,d,T", [("bf16", "f32", 4096, 3001), ("bf16", "bf16", 2048, 700),
                                              ("f32", "f32", 100, 257), ("bf16", "f32", 8192, 40),
                                              ("bf16", "f32", 512, 0)])
def test_forward_with_the_fold_inside_matches_fold_then_forward(dtype, wdtype, d, T):
    """engram_gate_fwd_fold: every output, and the fold it writes for the backward, bitwise those of
    engram_fuse_weight followed by engram_gate_fwd (an empty batch writes only the fold)."""
    wl = W.GateWorkload(name="fold", T=T, d=d, dtype=dtype, seed=77 + d + T)
    t = SD.gate_device_inputs(wl, DEV, with_dout=False)
    w_h, w_k = (t[n] if wdtype == "f32" else t[n].bfloat16() for n in ("w_h", "w_k"))
    wf = ecm.fuse_weight(w_h, w_k)
    ref = ecm.gate_fwd(t["h"], t["k"], t["v"], wf, wl.eps)
    got = ecm.gate_fwd_fold(t["h"], t["k"], t["v"], w_h, w_k, wl.eps)
    assert torch.equal(got[5], wf)
    for name, g_, r_ in zip(("out", "alpha", "rstd_h", "rstd_k", "dot"), got[:5], ref):
        assert torch.equal(g_, r_), name
