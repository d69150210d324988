"""GPU parity of the Engram Sinkhorn (momentum, row step, ordered reduction, finalize) against the
CPU oracle, through the C ABI.

Sizes: small matrices that span several partials and CTAs with ragged tails, head_dim from 4 to the
largest supported 8192, more partials than rows (empty partials), no row at all; the full
16384 x 5120 workload element by element; the printed 3 x 4 walk-through iterated to its fixed
point; bitwise reruns on different grids.

Tolerances are derived from the fp32 arithmetic of the kernels (u = 2^-24, all sums are of positive
terms, so a chain of n roundings costs at most about n u relative):
  * the row's sum of squares: per thread VPT float4 vectors (VPT = ceil(head_dim / 512)), each a
    3-rounding tree, added in order; 5 shuffle levels; 4 warp partials in order; each term x^2 with
    x = row_scale * m * col_scale two roundings off -> at most (4 VPT + 20) u; row_norm = sqrt:
    ss_rel / 2 + u;
  * row_scale / (row_norm + eps): + 3 u;  y = x / (row_norm + eps) and y^2, the partial's rows in
    two interleaved ascending chains added at the end: 2 (nrm_rel + 5 u) + (C + 1) u;  the
    reduction adds (ceil(P / 128) + 16 + 8) u;
  * finalize: alpha x / (||x|| + eps): nrm_rel + 5 u;
  * momentum: one fused multiply-add, correctly rounded: |gpu - ref| <= u |ref| (plus u beta |m'|
    for the Nesterov look-ahead, which reads the rounded m').
Each bound is doubled in the checks.  A dropped row or column term moves a value by ~1/rows or
~1/head_dim relative, far above these.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import engram_conditional_memory_gb300 as ecm
import oracle
from synth import generators as G
from synth import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
U = 2.0 ** -24


@pytest.fixture(autouse=True)
def _status_clean(cuda_lib):
    ecm.device_status(clear=True)
    yield
    assert ecm.device_status() == 0, "a kernel reported a device-side error"


def _vpt(D):
    return -(-D // 512)


def _nrm_rel(D):
    return (4 * _vpt(D) + 20) * U / 2 + U


def _rel_ok(got, ref, rel, what):
    got = np.asarray(got, dtype=np.float64)
    bad = np.abs(got - ref) > 2 * rel * np.abs(ref) + 1e-300
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside {2 * rel:.3g} relative; first at " \
                          f"{np.argwhere(bad)[0].tolist()}: {got[bad][0]!r} vs {ref[bad][0]!r}"


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _f64(t):
    return t.detach().cpu().numpy().astype(np.float64)


def _check_step(m, rs, cs, eps, P, row_norm, rs_new, part):
    """row_norm, the updated row_scale and every partial row against the oracle over its rows."""
    R, D = m.shape
    C = 1 if R == 0 else -(-R // P)
    ref = oracle.sinkhorn_step(m, rs, cs, eps)
    nrel = _nrm_rel(D)
    if R:
        _rel_ok(_f64(row_norm), ref["row_norm"], nrel, "row_norm")
        _rel_ok(_f64(rs_new), ref["row_scale"], nrel + 3 * U, "row_scale")
    part = _f64(part)
    for p in range(P):
        a, b = min(R, p * C), min(R, (p + 1) * C)
        if a == b:
            assert (part[p] == 0).all(), f"partial {p} has no row but is not 0"
            continue
        r = oracle.sinkhorn_step(m, rs, cs, eps, a, b)
        _rel_ok(part[p], r["col_sumsq"], 2 * (nrel + 5 * U) + (C + 1) * U, f"partial {p}")
    return ref


@pytest.mark.parametrize("R,D,P", [(37, 64, None), (300, 1024, 7), (1000, 5120, None), (17, 8192, 3),
                                   (5, 4, 8), (100, 132, 100), (1, 256, 1), (2000, 1028, 152), (333, 2052, 40)])
def test_step_reduce_finalize_small(R, D, P):
    w = W.SinkhornWorkload(name="t", rows=R, head_dim=D, grad_dtype="f32", seed=900 + R + D)
    x = W.sinkhorn_host_inputs(w)
    m, rs, cs = x["grad"], x["row_scale"], x["col_scale"]
    tm, trs, tcs = _t(m), _t(rs), _t(cs)
    P = P or ecm.sinkhorn_num_partials(R, D)
    row_norm, part = ecm.sinkhorn_step(tm, trs, tcs, w.eps, P=P)
    torch.cuda.synchronize()
    ref = _check_step(m, rs, cs, w.eps, P, row_norm, trs, part)
    # the ordered reduction and the column step, in place on col_scale
    C = -(-R // P)
    col_rel = 2 * (_nrm_rel(D) + 5 * U) + (C + 1) * U + (-(-P // 128) + 24) * U
    tcs2 = tcs.clone()
    col_sumsq = ecm.sinkhorn_step_reduce(part, col_scale=tcs2, eps=w.eps)
    torch.cuda.synchronize()
    _rel_ok(_f64(col_sumsq), ref["col_sumsq"], col_rel, "col_sumsq")
    _rel_ok(_f64(tcs2), oracle.sinkhorn_col_update(ref["col_sumsq"], cs, w.eps), col_rel / 2 + 3 * U, "col_scale")
    # finalize with the original scales
    out = ecm.sinkhorn_finalize(tm, _t(rs), tcs, w.eps, alpha=math.sqrt(D))
    torch.cuda.synchronize()
    _rel_ok(_f64(out), oracle.sinkhorn_finalize(m, rs, cs, w.eps, math.sqrt(D)), _nrm_rel(D) + 5 * U, "finalize")


def test_no_rows():
    tm = torch.empty((0, 64), dtype=torch.float32, device=DEV)
    trs = torch.empty(0, dtype=torch.float32, device=DEV)
    tcs = torch.ones(64, dtype=torch.float32, device=DEV)
    part = torch.full((3, 64), 7.0, device=DEV)
    ecm.sinkhorn_step(tm, trs, tcs, P=3, col_sumsq_partial=part)
    assert (part == 0).all()
    assert ecm.sinkhorn_finalize(tm, trs, tcs).shape == (0, 64)


@pytest.mark.parametrize("dtype,n,nesterov,beta", [("f32", 1001, True, 0.9), ("bf16", 4096 + 7, True, 0.95),
                                                   ("bf16", 3, False, 0.9), ("f32", 1 << 20, False, 0.5)])
def test_momentum(dtype, n, nesterov, beta):
    beta = float(np.float32(beta))  # the kernel's beta1 is fp32
    g = G.normal(950 + n, n)
    g = g.astype(np.float32) if dtype == "f32" else G.to_bf16_bits(g)
    m0 = G.normal(951 + n, n, 0.0, 0.5).astype(np.float32)
    tg = _t(g) if dtype == "f32" else _t(g.view(np.int16)).view(torch.bfloat16)
    tm = _t(m0)
    inp = ecm.sinkhorn_momentum_update(tg, tm, beta, nesterov)
    torch.cuda.synchronize()
    ref = oracle.sinkhorn_momentum(g, m0, beta, nesterov)
    gm, gi = _f64(tm), _f64(inp)
    assert (np.abs(gm - ref["momentum"]) <= U * np.abs(ref["momentum"]) * 1.0001).all()
    bound = U * (np.abs(ref["input"]) + (beta * np.abs(ref["momentum"]) if nesterov else 0)) * 1.0001
    assert (np.abs(gi - ref["input"]) <= bound + 1e-300).all()


def test_full_size_every_element():
    """The 16384 x 5120 workload: momentum (bf16 gradient) -> row step -> reduction + column step ->
    finalize, every output element against the oracle run on its own chain of results."""
    w = W.sinkhorn_16k_x_5120()
    x = W.sinkhorn_host_inputs(w)
    R, D = w.rows, w.head_dim
    beta = float(np.float32(w.beta1))
    tg = _t(x["grad"].view(np.int16)).view(torch.bfloat16)
    tm, trs, tcs = _t(x["momentum"]), _t(x["row_scale"]), _t(x["col_scale"])
    inp = ecm.sinkhorn_momentum_update(tg, tm, beta, w.nesterov)
    P = ecm.sinkhorn_num_partials(R, D)
    row_norm, part = ecm.sinkhorn_step(inp, trs, tcs, w.eps, P=P)
    part_host = part.clone()
    tcs_new = tcs.clone()
    col_sumsq = ecm.sinkhorn_step_reduce(part, col_scale=tcs_new, eps=w.eps)
    out = ecm.sinkhorn_finalize(inp, trs, tcs_new, w.eps, alpha=math.sqrt(D))
    torch.cuda.synchronize()

    mom = oracle.sinkhorn_momentum(x["grad"], x["momentum"], beta, w.nesterov)
    gi = _f64(inp)
    assert (np.abs(gi - mom["input"]) <= U * (np.abs(mom["input"]) + beta * np.abs(mom["momentum"])) * 1.0001).all()
    m32 = mom["input"].astype(np.float32)  # the oracle's own chain: its input rounded to the fp32 interface
    # Where the momentum step cancels (g + beta m' near 0) the GPU's fp32 input is off from the
    # oracle's by up to dm = u (|input| + beta |m'|) absolute (plus the oracle's own rounding to
    # fp32), not relative.  Every later value is smooth in each input element, so that difference
    # enters each check below as an absolute term through the element's sensitivity.
    dm = U * (1.5 * np.abs(mom["input"]) + beta * np.abs(mom["momentum"]))
    rs0, cs0 = x["row_scale"], x["col_scale"]
    ref = oracle.sinkhorn_step(m32, rs0, cs0, w.eps)
    a0 = np.abs(rs0)[:, None].astype(np.float64) * np.abs(cs0)[None, :]    # d x / d m
    x0 = a0 * np.abs(m32)
    inv0 = 1.0 / (ref["row_norm"] + w.eps)
    d_norm = (x0 * a0 * dm).sum(axis=1) * inv0                                # d ||x|| <= sum |x| a dm / ||x||
    nrel = _nrm_rel(D)
    bad = np.abs(_f64(row_norm) - ref["row_norm"]) > 2 * nrel * ref["row_norm"] + 2 * d_norm
    assert not bad.any(), "row_norm"
    d_rs = ref["row_scale"] * d_norm * inv0
    bad = np.abs(_f64(trs) - ref["row_scale"]) > 2 * (nrel + 3 * U) * ref["row_scale"] + 2 * d_rs
    assert not bad.any(), "row_scale"
    # d (y^2) with y = x / (||x|| + eps): 2 |y| (a dm + |x| d||x|| / ||x||) / ||x||
    y0 = x0 * inv0[:, None]
    d_y2 = 2 * y0 * (a0 * dm + x0 * (d_norm * inv0)[:, None]) * inv0[:, None]
    C = -(-R // P)
    parts = _f64(part_host)
    part_rel = 2 * (nrel + 5 * U) + (C + 1) * U
    d_col = np.zeros(D)
    for p in range(P):
        lo, hi = p * C, min(R, (p + 1) * C)
        r = oracle.sinkhorn_step(m32, rs0, cs0, w.eps, lo, hi)
        d_part = d_y2[lo:hi].sum(axis=0)
        d_col += d_part
        bad = np.abs(parts[p] - r["col_sumsq"]) > 2 * part_rel * r["col_sumsq"] + 2 * d_part
        assert not bad.any(), f"partial {p}: {np.argwhere(bad)[:3].tolist()}"
    col_rel = part_rel + (-(-P // 128) + 24) * U
    bad = np.abs(_f64(col_sumsq) - ref["col_sumsq"]) > 2 * col_rel * ref["col_sumsq"] + 2 * d_col
    assert not bad.any(), "col_sumsq"
    cs1 = oracle.sinkhorn_col_update(ref["col_sumsq"], cs0, w.eps)
    cs_rel = col_rel / 2 + 3 * U + d_col / ref["col_sumsq"] / 2
    bad = np.abs(_f64(tcs_new) - cs1) > 2 * cs_rel * cs1
    assert not bad.any(), "col_scale"
    # finalize on the oracle's chain (its row_scale and col_scale rounded to fp32).  out is
    # alpha x / ||x||: row_scale cancels; a column scale off by cs_rel moves its element and, less,
    # the norm; the input difference reaches out scaled by alpha rs cs / ||x||
    rs1, cs1 = ref["row_scale"].astype(np.float32), cs1.astype(np.float32)
    fin = oracle.sinkhorn_finalize(m32, rs1, cs1, w.eps, math.sqrt(D))
    x1 = rs1[:, None].astype(np.float64) * m32 * cs1[None, :].astype(np.float64)
    k = math.sqrt(D) * np.abs(rs1)[:, None] * np.abs(cs1)[None, :] / (np.linalg.norm(x1, axis=1)[:, None] + w.eps)
    rel = _nrm_rel(D) + 5 * U + U + 2 * (cs_rel.max() + U)
    bad = np.abs(_f64(out) - fin) > 2 * rel * np.abs(fin) + 2 * k * dm
    assert not bad.any(), f"finalize: {bad.sum()} outside tolerance; first at {np.argwhere(bad)[0].tolist()}"


def test_printed_walkthrough_fixed_point_on_gpu():
    """The 3 x 4 walk-through: 60 alternating row / column steps on the GPU reach the fixed point the
    pages print (column norms sqrt(3/4) before the column step, row norms sqrt(4/3) before finalize)
    and finalize with alpha = 2 gives rows of norm 2."""
    with open(os.path.join(os.path.dirname(__file__), "golden", "sinkhorn_demo.json")) as f:
        demo = json.load(f)
    R, D, alpha = demo["rows"], demo["head_dim"], demo["alpha"]
    m = np.abs(G.normal(602, R * D)).astype(np.float32).reshape(R, D) + 0.1
    tm = _t(m)
    trs = torch.ones(R, dtype=torch.float32, device=DEV)
    tcs = torch.ones(D, dtype=torch.float32, device=DEV)
    for _ in range(60):
        _, part = ecm.sinkhorn_step(tm, trs, tcs, 1e-6)
        col_sumsq = ecm.sinkhorn_step_reduce(part, col_scale=tcs, eps=1e-6)
    fp = demo["fixed_point"]
    np.testing.assert_allclose(np.sqrt(_f64(col_sumsq)), fp["col_l2_before_col_step"], rtol=1e-5)
    it = _f64(trs)[:, None] * m * _f64(tcs)[None, :]
    np.testing.assert_allclose(np.linalg.norm(it, axis=1), fp["row_l2_before_finalize"], rtol=1e-5)
    out = ecm.sinkhorn_finalize(tm, trs, tcs, 1e-6, alpha)
    np.testing.assert_allclose(np.linalg.norm(_f64(out), axis=1), demo["printed"]["row_l2_after_finalize"], rtol=1e-5)


def test_bitwise_reproducible_across_grids():
    w = W.SinkhornWorkload(name="g", rows=5000, head_dim=2048, grad_dtype="f32", seed=77)
    x = W.sinkhorn_host_inputs(w)
    tm, tcs = _t(x["grad"]), _t(x["col_scale"])
    P = ecm.sinkhorn_num_partials(w.rows, w.head_dim)

    def run():
        trs = _t(x["row_scale"])
        nrm, part = ecm.sinkhorn_step(tm, trs, tcs, w.eps, P=P)
        cs = tcs.clone()
        s = ecm.sinkhorn_step_reduce(part, col_scale=cs, eps=w.eps)
        out = ecm.sinkhorn_finalize(tm, trs, cs, w.eps, 3.0)
        return nrm, trs, part, s, cs, out

    base = run()
    try:
        for cap in (1, 3, 0):
            ecm.set_max_ctas(cap)
            again = run()
            for a, b in zip(base, again):
                assert torch.equal(a, b)
    finally:
        ecm.set_max_ctas(0)


def test_reduction_order_is_the_documented_one():
    """engram_sinkhorn_step_reduce sums 128 groups of ceil(P / 128) consecutive partials in
    ascending order, then runs of 16 consecutive group sums in ascending order, then the 8 run sums
    in ascending order: an fp32 emulation of that order on host-drawn partials matches bit for bit
    (another order would differ in the last bits)."""
    for P, D in ((1000, 256), (64, 8), (3, 4), (1024, 5120)):
        part = G.normal(960 + P, P * D).astype(np.float32).reshape(P, D) ** 2
        got = ecm.sinkhorn_step_reduce(_t(part)).cpu().numpy()
        per = -(-P // 128)
        groups = np.zeros((128, D), dtype=np.float32)
        for g in range(128):
            for q in range(g * per, min(P, (g + 1) * per)):
                groups[g] = groups[g] + part[q]
        runs = []
        for u in range(8):
            run = groups[16 * u].copy()
            for q in range(1, 16):
                run = run + groups[16 * u + q]
            runs.append(run)
        want = runs[0].copy()
        for u in range(1, 8):
            want = want + runs[u]
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (P, D)
