"""GPU parity of the short convolution after the gate (forward, backward, weight-gradient reduction)
against the CPU oracle, through the C ABI.

Sizes: small packed batches (ragged and empty sequences, several time chunks, channel blocks with a
ragged last block, widths 1 to 4, dilations 1 to 5 and 40, with and without H and bias, both dtypes, d up to
the largest supported 8192); the 4 x 4096-token, d = 4096 bf16 workload element by element; edge
cases (no token, in-place output) and bitwise reruns.

Tolerances come from the fp32 arithmetic (u = 2^-24):
  * rstd: a lane sums d/32 squares in order, then 5 shuffle levels, then rsqrtf (2 ulp):
    r_rel = (d/32 + 5)/2 u + 4 u;
  * conv: four products of u = V~ rstd norm_w (2 roundings + r_rel) and the taps, plus 4 adds:
    |dc| <= (r_rel + 8u) (|bias| + sum |w u|); SiLU (expf, 2 ulp; a division) adds 4u |SiLU|
    and |SiLU'| <= 1.1 times the conv error; the two residual adds 2u of the magnitudes; the output
    rounding half an ulp of |out| (an ulp for bf16, whose rounding the fp32 error can tip);
  * backward: dv = dout + rstd norm_w du - rstd^3 V~ s/d, with du from 4 products of the taps and
    dc, s a sum over d of 4 per thread (two pairs), a warp's 32 lanes in 5 shuffle levels, a
    CTA's 4 warps in 2 levels and up to 16 cluster blocks in order (26 levels; 29u is kept, the
    bound of the earlier order, a thread's 4 lanes in order before the shuffles):
    rel_b = 3 r_rel + 16u + 29u, times the oracle's magnitude sum
    |dout| + |rstd norm_w du| +
    |rstd^3 V~| sum|norm_w du V~|/d; and the conv's absolute error, carried into dc through SiLU''
    (at most 1/2 in size) and from there through the taps into du, dv and the weight gradients;
  * weight gradients: each term 2 r_rel + 12u, summed over a work item's tokens (at most
    L/dilation, L = max(256, T/256)) and by the reduction (P/128 + 16 + 8): times the magnitude sums.
Each bound is doubled in the checks.
"""
import math
from concurrent.futures import ThreadPoolExecutor

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


def _t(a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(DEV)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _h64(a):
    if a is None:
        return None
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64) if a.dtype == np.uint16 else \
        a.astype(np.float64)


def _r_rel(d):
    return (d / 32 + 5) / 2 * U + 4 * U


def _run(x, wl, out=None):
    t = {k: _t(v) for k, v in x.items()}
    o, rstd = ecm.short_conv_fwd(t["v"], t["norm_w"], t["conv_w"], t["seq_offsets"], wl.dilation, h=t["h"],
                                 bias=t["bias"], eps=wl.eps, out=out)
    dv, part = ecm.short_conv_bwd(t["dout"], t["v"], t["norm_w"], t["conv_w"], rstd, t["seq_offsets"], wl.dilation,
                                  bias=t["bias"])
    dcw, dbias, dnw = ecm.short_conv_grad_reduce(part, wl.width, wl.d, want_bias=wl.bias)
    torch.cuda.synchronize()
    return dict(out=o, rstd=rstd, dv=dv, part=part, dconv_w=dcw, dbias=dbias, dnorm_w=dnw)


def _oracle(x, wl, threads=1):
    T = wl.T
    bounds = [(T * i // threads, T * (i + 1) // threads) for i in range(threads)]

    def part(b):
        a, e = b
        f = oracle.short_conv_fwd(x["v"], x["h"], x["norm_w"], x["conv_w"], x["bias"], x["seq_offsets"], wl.dilation,
                                  wl.eps, a, e)
        g = oracle.short_conv_bwd(x["dout"], x["v"], x["norm_w"], x["conv_w"], x["bias"], x["seq_offsets"],
                                  wl.dilation, wl.eps, a, e)
        return f, g

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(part, bounds))
    f = {k: np.concatenate([p[0][k] for p in parts]) for k in ("out", "c", "rstd")}
    b = {k: np.concatenate([p[1][k] for p in parts]) for k in ("dv", "dv_abs")}
    for k in ("dconv_w", "dbias", "dnorm_w", "dconv_w_abs", "dbias_abs", "dnorm_w_abs"):
        b[k] = np.sum([p[1][k] for p in parts], axis=0)
    return f, b


def _shift(a, back, seq_start, seq_end):
    """a[t - back] within t's sequence (0 outside it); back < 0 looks ahead."""
    T = a.shape[0]
    idx = np.arange(T) - back
    ok = (idx >= seq_start) & (idx < seq_end)
    out = np.zeros_like(a)
    out[ok] = a[idx[ok]]
    return out


def _check_fwd(r, x, wl, f):
    """rstd and out against the oracle's forward; returns the conv's error bound for the backward."""
    d = wl.d
    rr = _r_rel(d)
    bf16 = wl.dtype == "bf16"
    np.testing.assert_allclose(_f64(r["rstd"]), f["rstd"], rtol=2 * rr)
    # forward: the conv's magnitude from the oracle's own rstd
    v, h, g = _h64(x["v"]), _h64(x["h"]), _h64(x["dout"])
    u = v * f["rstd"][:, None] * x["norm_w"].astype(np.float64)
    offs = x["seq_offsets"]
    seq_start = np.repeat(offs[:-1], np.diff(offs))
    seq_end = np.repeat(offs[1:], np.diff(offs))
    cw = np.abs(x["conv_w"].astype(np.float64))
    conv_abs = np.abs(x["bias"]).astype(np.float64)[None, :] if x["bias"] is not None else np.zeros((1, d))
    for i in range(wl.width):
        conv_abs = conv_abs + cw[:, i][None, :] * np.abs(_shift(u, (wl.width - 1 - i) * wl.dilation, seq_start,
                                                               seq_end))
    silu = f["out"] - (h if h is not None else 0) - v
    err_c = (rr + 8 * U) * conv_abs
    mag = np.abs(v) + np.abs(silu) + (np.abs(h) if h is not None else 0)
    round_out = (2.0 ** -8 if bf16 else U) * np.abs(f["out"])
    tol = round_out + 1.1 * err_c + 4 * U * np.abs(silu) + 2 * U * mag
    bad = np.abs(_f64(r["out"]) - f["out"]) > 2 * tol + 1e-30
    assert not bad.any(), f"out: {bad.sum()} of {bad.size}; first {np.argwhere(bad)[0].tolist()}"
    return err_c, u, seq_start, seq_end, cw


def _check(r, x, wl, f, b):
    d, T = wl.d, wl.T
    rr = _r_rel(d)
    bf16 = wl.dtype == "bf16"
    err_c, u, seq_start, seq_end, cw = _check_fwd(r, x, wl, f)
    v, g = _h64(x["v"]), _h64(x["dout"])
    # backward.  Besides the relative error of its own arithmetic, each dc = dout SiLU'(c) carries
    # the conv's absolute error through SiLU'' (|SiLU''| <= 1/2): dc_err = |dout| (err_c / 2 + 4.4 u);
    # du gathers it through the taps, dv through rstd norm_w and the row dot s.
    dc_err = np.abs(g) * (0.5 * err_c + 4.4 * U)
    du_err = np.zeros_like(dc_err)
    for i in range(wl.width):
        du_err += cw[:, i][None, :] * _shift(dc_err, -(wl.width - 1 - i) * wl.dilation, seq_start, seq_end)
    rs = f["rstd"][:, None]
    nw = np.abs(x["norm_w"].astype(np.float64))[None, :]
    dv_err = rs * nw * du_err + rs ** 3 * np.abs(v) / d * (nw * np.abs(v) * du_err).sum(axis=1, keepdims=True)
    rel_b = 3 * rr + 16 * U + 29 * U
    round_dv = (2.0 ** -8 if bf16 else U) * np.abs(b["dv"])
    bad = np.abs(_f64(r["dv"]) - b["dv"]) > 2 * (round_dv + rel_b * b["dv_abs"] + dv_err) + 1e-30
    assert not bad.any(), f"dv: {bad.sum()} of {bad.size}; first {np.argwhere(bad)[0].tolist()}"
    L = max(256, -(-T // 256))
    P = r["part"].shape[0]
    rel_w = 2 * rr + 12 * U + (L / wl.dilation + P / 128 + 24) * U
    extra = {"dbias": dc_err.sum(axis=0), "dnorm_w": (np.abs(v) * rs * du_err).sum(axis=0),
             "dconv_w": np.stack([(np.abs(_shift(u, (wl.width - 1 - i) * wl.dilation, seq_start, seq_end)) *
                                   dc_err).sum(axis=0) for i in range(wl.width)], axis=1)}
    for k in ("dconv_w", "dnorm_w") + (("dbias",) if wl.bias else ()):
        got = _f64(r[k])
        bad = np.abs(got - b[k]) > 2 * (rel_w * b[k + "_abs"] + extra[k]) + 1e-30
        assert not bad.any(), f"{k}: {bad.sum()} of {bad.size}; first {np.argwhere(bad)[0].tolist()}"


@pytest.mark.parametrize("lengths,d,width,dil,dtype,bias,with_h", [
    ([300, 0, 700], 256, 4, 3, "bf16", True, True),
    ([1000], 128, 4, 3, "f32", True, True),
    ([17] * 10, 1024, 4, 3, "bf16", False, True),
    ([513, 1, 2, 400], 4096, 4, 3, "bf16", True, True),
    ([64], 8, 2, 1, "bf16", True, False),
    ([2000], 136, 3, 5, "f32", True, True),
    ([5, 2], 8192, 4, 3, "bf16", True, True),
    ([300, 77], 512, 1, 3, "bf16", True, True),
    ([600], 1000, 4, 2, "bf16", True, False),
    ([500, 1, 300], 64, 4, 40, "bf16", True, True),
])
def test_small_cases(lengths, d, width, dil, dtype, bias, with_h):
    wl = W.ShortConvWorkload(name="t", lengths=lengths, d=d, width=width, dilation=dil, dtype=dtype,
                             seed=800 + d + len(lengths) + width, bias=bias, with_h=with_h)
    x = W.short_conv_host_inputs(wl)
    r = _run(x, wl)
    f, b = _oracle(x, wl, threads=8)
    _check(r, x, wl, f, b)


def test_long_sequences_larger_chunks():
    """T above 65,536: the backward's chunks grow beyond 256 tokens (L = ceil(T / 256)), 256 of them."""
    wl = W.ShortConvWorkload(name="long", lengths=[40000, 3, 30001], d=64, width=4, dilation=3, dtype="bf16",
                             seed=97, bias=True, with_h=True)
    x = W.short_conv_host_inputs(wl)
    r = _run(x, wl)
    assert r["part"].shape[0] == 256 * 3
    f, b = _oracle(x, wl, threads=16)
    _check(r, x, wl, f, b)


def test_full_workload_every_element():
    wl = W.short_conv_4x4k()
    x = W.short_conv_host_inputs(wl)
    r = _run(x, wl)
    f, b = _oracle(x, wl, threads=16)
    _check(r, x, wl, f, b)


def test_in_place_output_and_bitwise_reruns():
    wl = W.ShortConvWorkload(name="ip", lengths=[700, 300, 1], d=512, width=4, dilation=3, dtype="bf16", seed=81)
    x = W.short_conv_host_inputs(wl)
    a = _run(x, wl)
    b = _run(x, wl)
    for k in ("out", "rstd", "dv", "part", "dconv_w", "dbias", "dnorm_w"):
        assert torch.equal(a[k], b[k]), k
    h = _t(x["h"])
    t = {k: _t(v) for k, v in x.items()}
    o, _ = ecm.short_conv_fwd(t["v"], t["norm_w"], t["conv_w"], t["seq_offsets"], 3, h=h, bias=t["bias"], out=h)
    assert o.data_ptr() == h.data_ptr() and torch.equal(h, a["out"])
    # the weight-gradient reduction on 1 or 5 CTAs: each walks a larger share of the columns
    try:
        for cap in (1, 5):
            ecm.set_max_ctas(cap)
            dcw, dbias, dnw = ecm.short_conv_grad_reduce(a["part"], wl.width, wl.d, want_bias=wl.bias)
            assert torch.equal(dcw, a["dconv_w"]) and torch.equal(dbias, a["dbias"]) and torch.equal(dnw, a["dnorm_w"])
    finally:
        ecm.set_max_ctas(0)


@pytest.mark.parametrize("lengths,dil", [([3000, 1, 1500, 700], 3), ([513], 3), ([300, 213], 40)],
                         ids=["ragged", "empty_items", "empty_items_dil40"])
def test_backward_bitwise_across_grids(lengths, dil):
    """The backward's clusters take contiguous ranges of work items in class order, so the grid decides
    where one cluster's sweep stops and the next one's starts; outputs and partials must not depend on
    it.  On 1, 2, 3 and 7 clusters of 2 CTAs against the uncapped grid, bit for bit: 63 work items of
    ragged sequences; and last time chunks shorter than the dilation (513 tokens: chunk 2 holds token
    512 alone, so 2 of 3 classes, or at dilation 40 with a sequence boundary at 300, 39 of 40, have
    no token there), whose empty items then sit inside one cluster's range and still get zero rows.
    The partials are filled with NaN before each capped run, so a row left unwritten would show."""
    wl = W.ShortConvWorkload(name="grids", lengths=lengths, d=1024, width=4, dilation=dil, dtype="bf16",
                             seed=83 + dil, bias=True, with_h=False)
    x = W.short_conv_host_inputs(wl)
    t = {k: _t(v) for k, v in x.items() if v is not None}
    a = _run(x, wl)
    assert not torch.isnan(a["part"]).any()
    try:
        for ncl in (1, 2, 3, 7):
            ecm.set_max_ctas(2 * ncl)
            part = torch.full_like(a["part"], float("nan"))
            dv, part = ecm.short_conv_bwd(t["dout"], t["v"], t["norm_w"], t["conv_w"], a["rstd"], t["seq_offsets"],
                                          wl.dilation, bias=t.get("bias"), dw_partial=part)
            torch.cuda.synchronize()
            assert torch.equal(dv, a["dv"]), f"dv on {ncl} clusters"
            assert torch.equal(part, a["part"]), f"partials on {ncl} clusters"
    finally:
        ecm.set_max_ctas(0)
    assert ecm.device_status() == 0


@pytest.mark.parametrize("lengths,d,dtype", [([700, 0, 300, 1], 4096, "bf16"), ([500], 136, "f32"),
                                             ([64, 64], 8192, "bf16"), ([1], 8, "bf16")])
def test_gate_statistic_feeds_the_conv(lengths, d, dtype):
    """The gate writes V~ with its RMS statistic (gate_fwd_rms), and the conv takes that statistic
    instead of its own pass: the gate's other outputs are those of gate_fwd bit for bit, the
    statistic matches the oracle's rstd of the stored V~, and the conv's output the oracle's conv of
    that V~, within the forward's bounds."""
    wl = W.ShortConvWorkload(name="g", lengths=lengths, d=d, width=4, dilation=3, dtype=dtype, seed=900 + d)
    x = W.short_conv_host_inputs(wl)
    T = wl.T
    cv = (lambda a: a.astype(np.float32)) if dtype == "f32" else G.to_bf16_bits
    hg, kg, vg = (_t(cv(G.normal(930 + i, T * d).reshape(T, d))) for i in range(3))
    wf = ecm.fuse_weight(_t(G.normal(934, d, 1.0, 0.1).astype(np.float32)),
                         _t(G.normal(935, d, 1.0, 0.1).astype(np.float32)))
    ref = ecm.gate_fwd(hg, kg, vg, wf, 1e-6)
    got = ecm.gate_fwd_rms(hg, kg, vg, wf, 1e-6, out_eps=wl.eps)
    for a, b in zip(ref, got[:5]):
        assert torch.equal(a, b)
    vt, out_rstd = got[0], got[5]
    # the conv over V~ = the gate's output as stored, with the statistic given
    x["v"] = vt.cpu().view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else vt.cpu().numpy()
    t = {k: _t(v) for k, v in x.items()}
    o, r_std = ecm.short_conv_fwd(vt, t["norm_w"], t["conv_w"], t["seq_offsets"], wl.dilation, h=t["h"],
                                  bias=t["bias"], given_rstd=out_rstd)
    assert r_std.data_ptr() == out_rstd.data_ptr()
    f = oracle.short_conv_fwd(x["v"], x["h"], x["norm_w"], x["conv_w"], x["bias"], x["seq_offsets"], wl.dilation,
                              wl.eps, 0, T)
    _check_fwd({"out": o, "rstd": out_rstd}, x, wl, f)
    # with the conv's own statistic given back, its output is the ordinary forward's bit for bit
    o2, r2 = ecm.short_conv_fwd(vt, t["norm_w"], t["conv_w"], t["seq_offsets"], wl.dilation, h=t["h"],
                                bias=t["bias"])
    o3, _ = ecm.short_conv_fwd(vt, t["norm_w"], t["conv_w"], t["seq_offsets"], wl.dilation, h=t["h"],
                               bias=t["bias"], given_rstd=r2)
    assert torch.equal(o2, o3)


def test_gate_statistic_empty_batch():
    h = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    wf = torch.ones(64, dtype=torch.float32, device=DEV)
    out, *_, ostd = ecm.gate_fwd_rms(h, h, h, wf)
    assert out.shape == (0, 64) and ostd.shape == (0,)
    v = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    offs = torch.zeros(2, dtype=torch.int64, device=DEV)
    o, _ = ecm.short_conv_fwd(v, wf, torch.ones((64, 4), dtype=torch.float32, device=DEV), offs, 3, given_rstd=ostd)
    assert o.shape == (0, 64)


def test_no_token():
    wl = W.ShortConvWorkload(name="e", lengths=[0], d=64, width=4, dilation=3, dtype="bf16", seed=5)
    x = W.short_conv_host_inputs(wl)
    r = _run(x, wl)
    assert r["out"].shape == (0, 64) and r["part"].shape[0] == 0
    assert (r["dconv_w"] == 0).all() and (r["dnorm_w"] == 0).all() and (r["dbias"] == 0).all()
