"""GPU parity of the multi-branch gate (x [T, hc, d], kv [T, hc+1, d]) against the CPU oracle.

Sizes: small fp32/bf16 cases for hc = 1, 2, 4; the production shape T = 8192, hc = 4, d = 4096
(bf16) element by element; edge cases: the clamp branch (k = 0), in-place writing (forward and
backward, in both forms), an empty batch, and bitwise reruns.  The fused weight is [hc, d] (engram_fuse_weight over hc*d) and the
partials reduce with engram_grad_w_reduce over hc*d columns.
"""
import math

import numpy as np
import pytest
import torch

import engram_conditional_memory_gb300 as ecm
import oracle
from synth import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _status_clean(cuda_lib):
    ecm.device_status(clear=True)
    yield
    assert ecm.device_status() == 0, "a kernel reported a device-side error"


def _dev(x):
    out = {}
    for n, a in x.items():
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 else torch.from_numpy(a)
        out[n] = t.to(DEV)
    return out


def _run(t, wl, P=None):
    T, hc, d = t["x"].shape
    wf = ecm.fuse_weight(t["w_h"].reshape(-1), t["w_k"].reshape(-1)).reshape(hc, d)
    out, gate, rx, rk, dot = ecm.gate_hc_fwd(t["x"], t["kv"], wf, wl.eps, wl.clamp)
    dx, dkv, part = ecm.gate_hc_bwd(t["dout"], t["x"], t["kv"], wf, gate, rx, rk, dot, wl.clamp, P=P)
    dw = ecm.grad_w_reduce(part.reshape(part.shape[0], hc * d)).reshape(hc, d)
    return dict(wf=wf, out=out, gate=gate, rstd_x=rx, rstd_k=rk, dot=dot, dx=dx, dkv=dkv, part=part, dw=dw)


def _check(r, x, wl, f=None, b=None):
    """Element-wise parity with the oracle.

    Tolerances: those of the single-branch gate, plus, for everything downstream of the
    activation's slope, the error that the fp32 dot product carries into it.  The signed square
    root has slope 1/(2 sqrt|z|) (up to 1/(2 sqrt(clamp)) = 500), so a dot-product error dz
    becomes a relative error dz / (2 |z|) of c = dL/d dot; dx, dk and the weight gradient inherit
    it in proportion to the c-weighted terms.  dz is the dot tolerance mapped to z.
    """
    f = f or oracle.gate_hc_fwd(x["x"], x["kv"], x["w_h"], x["w_k"], wl.eps, wl.clamp)
    b = b or oracle.gate_hc_bwd(x["dout"], x["x"], x["kv"], x["w_h"], x["w_k"], wl.eps, wl.clamp)
    check_plain = H.assert_close_bf16 if wl.dtype == "bf16" else H.assert_close_rows
    assert np.abs(H.as_f64(r["gate"]) - f["gate"]).max() <= H.ALPHA_ATOL
    np.testing.assert_allclose(H.as_f64(r["rstd_x"]), f["rstd_x"], rtol=H.RSTD_RTOL)
    np.testing.assert_allclose(H.as_f64(r["rstd_k"]), f["rstd_k"], rtol=H.RSTD_RTOL)
    xf, kvf, gf = H._f64(x["x"]), H._f64(x["kv"]), H._f64(x["dout"])
    kf, vf = kvf[:, :wl.hc], kvf[:, wl.hc]
    w = (x["w_h"] * x["w_k"]).astype(np.float64)[None]
    dot_scale = np.abs(xf * w * kf).sum(-1)
    dot_tol = 2e-5 * dot_scale + 1e-6
    assert (np.abs(H.as_f64(r["dot"]) - f["dot"]) <= dot_tol).all()
    check_plain(r["out"], f["out"], "out")
    # c = dL/d dot (fp64, from the oracle's statistics) and its relative sensitivity to dz
    sc = f["rstd_x"] * f["rstd_k"] / math.sqrt(wl.d)
    z = f["dot"] * sc
    dgate = (gf * vf[:, None, :]).sum(-1)
    live = ~(np.abs(z) < wl.clamp)
    c = np.where(live, dgate * f["gate"] * (1 - f["gate"]) / (2 * np.sqrt(np.maximum(np.abs(z), wl.clamp))) * sc, 0.0)
    rel_c = np.where(live, dot_tol * sc / (2 * np.maximum(np.abs(z), wl.clamp)), 0.0)
    extra = (rel_c * np.abs(c))[..., None]
    base = (lambda ref: H.BF16_ATOL + H.BF16_RTOL * np.abs(ref)) if wl.dtype == "bf16" else \
        (lambda ref: 1e-5 * np.abs(ref).max(axis=-1, keepdims=True) + 1e-4 * np.abs(ref))
    dotx = (f["dot"] * f["rstd_x"] ** 2 / wl.d)[..., None]
    dotk = (f["dot"] * f["rstd_k"] ** 2 / wl.d)[..., None]
    dx, dk = H.as_f64(r["dx"]), H.as_f64(r["dkv"])[:, :wl.hc]
    tol_dx = base(b["dx"]) + extra * (np.abs(w * kf) + np.abs(xf * dotx))
    tol_dk = base(b["dkv"][:, :wl.hc]) + extra * (np.abs(w * xf) + np.abs(kf * dotk))
    bad = np.abs(dx - b["dx"]) > tol_dx
    assert not bad.any(), f"dx: {bad.sum()} outside tolerance at {np.argwhere(bad)[:3].tolist()}"
    bad = np.abs(dk - b["dkv"][:, :wl.hc]) > tol_dk
    assert not bad.any(), f"dk: {bad.sum()} outside tolerance at {np.argwhere(bad)[:3].tolist()}"
    bad = np.abs(H.as_f64(r["dkv"])[:, wl.hc] - b["dkv"][:, wl.hc]) > base(b["dkv"][:, wl.hc])
    assert not bad.any(), f"dv: {bad.sum()} outside tolerance"
    dw_extra = np.einsum("th,thi->hi", rel_c * np.abs(c), np.abs(xf * kf))
    assert (np.abs(H.as_f64(r["dw"]) - b["dweight"]) <= 1e-4 * b["dweight_abs"] + dw_extra + 1e-7).all()
    return f, b


@pytest.mark.parametrize("dtype,hc,d,T", [("f32", 4, 64, 37), ("bf16", 4, 128, 50), ("bf16", 4, 4096, 40),
                                          ("f32", 4, 2048, 9), ("bf16", 2, 1000, 33), ("f32", 1, 96, 70),
                                          ("bf16", 1, 7168, 21), ("bf16", 2, 8192, 5)])
def test_small_cases(dtype, hc, d, T):
    wl = W.GateHcWorkload(name="t", T=T, hc=hc, d=d, dtype=dtype, seed=700 + hc * d + T)
    x = W.gate_hc_host_inputs(wl)
    r = _run(_dev(x), wl)
    torch.cuda.synchronize()
    _check(r, x, wl)


@pytest.mark.parametrize("dtype,hc,d,T", [("bf16", 4, 7168, 41), ("bf16", 4, 8192, 9), ("f32", 4, 3072, 17),
                                          ("f32", 2, 4096, 13)])
def test_rows_too_large_for_a_whole_token(dtype, hc, d, T):
    """Rows whose token does not fit twice in one CTA's shared memory (d = 7168 at hc = 4, the largest
    rows, fp32 past its whole-token limit) run on clusters of two CTAs that each hold half of every
    row and exchange their halves' sums: every output against the oracle."""
    wl = W.GateHcWorkload(name="t", T=T, hc=hc, d=d, dtype=dtype, seed=760 + hc * d + T)
    x = W.gate_hc_host_inputs(wl)
    r = _run(_dev(x), wl)
    torch.cuda.synchronize()
    _check(r, x, wl)


@pytest.mark.parametrize("dtype,hc,d,T", [("bf16", 4, 7168, 41), ("bf16", 4, 8192, 9)])
def test_large_rows_in_clusters_of_four(dtype, hc, d, T):
    """The row split over clusters of four CTAs (two per SM) forced at the large rows: every output
    against the oracle."""
    wl = W.GateHcWorkload(name="t4", T=T, hc=hc, d=d, dtype=dtype, seed=770 + hc * d + T)
    x = W.gate_hc_host_inputs(wl)
    prev = ecm.set_hc_split(ecm.HC_ROW_SPLIT4)
    try:
        r = _run(_dev(x), wl)
        torch.cuda.synchronize()
    finally:
        ecm.set_hc_split(prev)
    _check(r, x, wl)


@pytest.mark.parametrize("dtype,hc,d,T", [("bf16", 4, 1024, 300), ("f32", 2, 96, 77), ("bf16", 4, 4096, 40)])
@pytest.mark.parametrize("mode", [ecm.HC_BRANCHES, ecm.HC_ROW_SPLIT, ecm.HC_ROW_SPLIT4],
                         ids=["branch_by_branch", "row_split", "row_split4"])
def test_other_forms_at_whole_token_sizes(dtype, hc, d, T, mode):
    """The branch-by-branch form and the two-CTA row split forced where the whole-token kernels also
    run: each against the oracle, and in-place writing (out = x) kept."""
    wl = W.GateHcWorkload(name="t", T=T, hc=hc, d=d, dtype=dtype, seed=780 + hc * d + T)
    x = W.gate_hc_host_inputs(wl)
    prev = ecm.set_hc_split(mode)
    try:
        t = _dev(x)
        r = _run(t, wl)
        torch.cuda.synchronize()
        _check(r, x, wl)
        xi = t["x"].clone()
        ecm.gate_hc_fwd(xi, t["kv"], r["wf"], wl.eps, wl.clamp, inplace=True, save_for_backward=False)
        assert torch.equal(xi, r["out"])
    finally:
        ecm.set_hc_split(prev)


@pytest.mark.parametrize("wl", [W.gate_hc_4x4k(),
                                W.GateHcWorkload(name="gate_hc4_T2048_d7168", T=2048, hc=4, d=7168, dtype="bf16",
                                                 seed=6 * 101 + 31)], ids=lambda w: w.name)
def test_production_shape_every_element(wl):
    """The release's shape, hc = 4 at d = 4096 (whole token per CTA) and at its width d = 7168 (a token
    shared by clusters of two CTAs forward and four backward): every element against the oracle."""
    x = W.gate_hc_host_inputs(wl)
    r = _run(_dev(x), wl)
    torch.cuda.synchronize()
    n = 16
    bounds = [(wl.T * i // n, wl.T * (i + 1) // n) for i in range(n)]
    from concurrent.futures import ThreadPoolExecutor

    def part(bnd):
        a, b = bnd
        return (oracle.gate_hc_fwd(x["x"], x["kv"], x["w_h"], x["w_k"], wl.eps, wl.clamp, a, b),
                oracle.gate_hc_bwd(x["dout"], x["x"], x["kv"], x["w_h"], x["w_k"], wl.eps, wl.clamp, a, b))

    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(part, bounds))
    f = {k: np.concatenate([p[0][k] for p in parts]) for k in parts[0][0]}
    b = {k: np.concatenate([p[1][k] for p in parts]) for k in ("dx", "dkv")}
    b["dweight"] = np.sum([p[1]["dweight"] for p in parts], axis=0)
    b["dweight_abs"] = np.sum([p[1]["dweight_abs"] for p in parts], axis=0)
    _check(r, x, wl, f, b)


def test_zero_keys_hit_the_clamp():
    wl = W.GateHcWorkload(name="k0", T=64, hc=4, d=512, dtype="bf16", seed=41)
    x = W.gate_hc_host_inputs(wl)
    x["kv"][:, :4] = 0  # bf16 +0
    t = _dev(x)
    r = _run(t, wl)
    g0 = 1.0 / (1.0 + math.exp(-0.001))
    assert np.abs(H.as_f64(r["gate"]) - g0).max() <= 1e-6
    assert torch.equal(r["dx"], t["dout"])  # no gradient through the clamped gate
    assert (r["dkv"][:, :4] == 0).all() and (r["part"] == 0).all()
    _check(r, x, wl)


def test_in_place_forward_matches_and_refuses_saving():
    wl = W.GateHcWorkload(name="ip", T=300, hc=4, d=1024, dtype="bf16", seed=42)
    x = W.gate_hc_host_inputs(wl)
    t = _dev(x)
    wf = ecm.fuse_weight(t["w_h"].reshape(-1), t["w_k"].reshape(-1)).reshape(4, 1024)
    ref, *_ = ecm.gate_hc_fwd(t["x"], t["kv"], wf, save_for_backward=False)
    xin = t["x"].clone()
    out, *_ = ecm.gate_hc_fwd(xin, t["kv"], wf, save_for_backward=False, inplace=True)
    assert out.data_ptr() == xin.data_ptr() and torch.equal(xin, ref)
    stats = tuple(torch.empty((300, 4), dtype=torch.float32, device=DEV) for _ in range(4))
    # out == x with a statistic requested: refused on the host (a backward would read the overwritten x)
    lib = ecm.load_library()
    st = lib.engram_gate_hc_fwd(xin.data_ptr(), t["kv"].data_ptr(), 1, wf.data_ptr(), 300, 4, 1024, 1e-6, 1e-6,
                                xin.data_ptr(), stats[0].data_ptr(), None, None, None,
                                torch.cuda.current_stream().cuda_stream)
    assert st == 2 and torch.equal(xin, ref)
    with pytest.raises(ValueError):
        ecm.gate_hc_fwd(xin, t["kv"], wf, inplace=True)


def test_empty_batch_and_bitwise_reruns():
    wl = W.GateHcWorkload(name="e", T=0, hc=4, d=256, dtype="bf16", seed=1)
    x = W.gate_hc_host_inputs(wl)
    t = _dev(x)
    r = _run(t, wl, P=3)
    assert r["out"].shape == (0, 4, 256) and (r["part"] == 0).all()
    wl = W.GateHcWorkload(name="d", T=3000, hc=4, d=4096, dtype="bf16", seed=2)
    t = _dev(W.gate_hc_host_inputs(wl))
    a, b = _run(t, wl), _run(t, wl)
    for k in ("out", "gate", "dx", "dkv", "part", "dw"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("mode", [ecm.HC_AUTO, ecm.HC_BRANCHES, ecm.HC_ROW_SPLIT, ecm.HC_ROW_SPLIT4],
                         ids=["whole_token", "branch_by_branch", "row_split", "row_split4"])
def test_in_place_backward(mode):
    """dx written over dout, and dkv over kv, give bitwise the out-of-place results in every form.
    The pair together is served by the whole-token and row-split forms and refused, before anything
    is written, in the branch-by-branch form (the value row's gradient reads dout, the branch
    kernels read the value row).  Other overlaps of an output with an input are refused."""
    wl = W.GateHcWorkload(name="ipb", T=300, hc=4, d=1024, dtype="bf16", seed=43)
    t = _dev(W.gate_hc_host_inputs(wl))
    split = mode == ecm.HC_BRANCHES
    prev = ecm.set_hc_split(mode)
    try:
        r = _run(t, wl)
        st = (r["gate"], r["rstd_x"], r["rstd_k"], r["dot"])
        P = r["part"].shape[0]

        def bwd(dout, kv, **kw):
            return ecm.gate_hc_bwd(dout, t["x"], kv, r["wf"], *st, wl.clamp, P=P, **kw)

        g = t["dout"].clone()
        dx, dkv, part = bwd(g, t["kv"], dx=g)
        assert dx.data_ptr() == g.data_ptr()
        assert torch.equal(g, r["dx"]) and torch.equal(dkv, r["dkv"]) and torch.equal(part, r["part"])
        kv = t["kv"].clone()
        dx, _, part = bwd(t["dout"], kv, dkv=kv)
        assert torch.equal(dx, r["dx"]) and torch.equal(kv, r["dkv"]) and torch.equal(part, r["part"])
        g, kv = t["dout"].clone(), t["kv"].clone()
        if split:
            with pytest.raises(ecm.EngramError) as e:
                bwd(g, kv, dx=g, dkv=kv)
            assert e.value.status == 2
            torch.cuda.synchronize()
            assert torch.equal(g, t["dout"]) and torch.equal(kv, t["kv"])
        else:
            bwd(g, kv, dx=g, dkv=kv)
            assert torch.equal(g, r["dx"]) and torch.equal(kv, r["dkv"])
        # an output shifted by one token against its input, and dx over the keys: refused
        big = torch.cat([t["dout"], t["dout"][:1]]).contiguous()
        with pytest.raises(ecm.EngramError):
            bwd(big[1:], t["kv"], dx=big[:-1])
        with pytest.raises(ecm.EngramError):
            bwd(t["dout"], t["kv"], dx=t["kv"].view(-1)[: 300 * 4 * 1024].view(300, 4, 1024))
    finally:
        ecm.set_hc_split(prev)


@pytest.mark.parametrize("dtype,hc,d,T", [("bf16", 4, 4160, 37), ("bf16", 4, 6144, 3), ("f32", 4, 2080, 11),
                                          ("bf16", 4, 4104, 5), ("bf16", 4, 7168, 1), ("bf16", 4, 4112, 19)])
def test_forms_chosen_at_unusual_widths(dtype, hc, d, T):
    """Widths between the forms' limits, each run in the form the library picks: d = 4160 and 6144 bf16
    and 2080 fp32 on clusters of 2 (forward) and 4 (backward); d = 4112, whose quarter rows are not a
    multiple of 16 bytes, on pairs in both directions; d = 4104, whose half rows are not either,
    branch by branch; and a single token.  Every output against the oracle."""
    wl = W.GateHcWorkload(name="u", T=T, hc=hc, d=d, dtype=dtype, seed=990 + d + T)
    x = W.gate_hc_host_inputs(wl)
    r = _run(_dev(x), wl)
    torch.cuda.synchronize()
    _check(r, x, wl)


@pytest.mark.parametrize("mode", [ecm.HC_ROW_SPLIT, ecm.HC_ROW_SPLIT4], ids=["row_split", "row_split4"])
def test_cluster_forms_bitwise_across_grids(mode):
    """The cluster forms give bitwise the same outputs, statistics and partials whatever the grid:
    capped at 1 CTA (one cluster walks every token and partial), at 7 and 151 CTAs, and uncapped."""
    wl = W.GateHcWorkload(name="g", T=700, hc=4, d=2048, dtype="bf16", seed=55)
    t = _dev(W.gate_hc_host_inputs(wl))
    prev = ecm.set_hc_split(mode)
    try:
        base = _run(t, wl)
        for cap in (1, 7, 151, 0):
            ecm.set_max_ctas(cap)
            try:
                r = _run(t, wl)
            finally:
                ecm.set_max_ctas(0)
            for k in ("out", "gate", "rstd_x", "rstd_k", "dot", "dx", "dkv", "part", "dw"):
                assert torch.equal(r[k], base[k]), (cap, k)
    finally:
        ecm.set_hc_split(prev)
