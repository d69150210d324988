"""Pins of the CPU oracle against things other than itself (CPU only).

* hash: hand-derived closed forms (tests/golden/hash_closed_forms.json),
  brute-force invariants over every pair of tokens, range, determinism, the
  O(1) rows-per-token property, and bucket occupancy close to the uniform-hash
  expectation;
* gather: a table whose rows encode their own index;
* gate forward: torch's fp64 rms_norm + sigmoid (a library routine), the k = 0
  and h = +-k closed forms, the fused/unfused identity, scale invariance;
* gate backward: torch fp64 autograd, central finite differences of the oracle's
  own forward, and the near scale-invariance identities;
* grad_w reduce: constant partials with closed-form sums.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from synth import generators as G
from synth import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hash_closed_forms.json")


# ----------------------------------------------------------------------------- hash

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hash_closed_forms(case):
    got = oracle.hash_indices(
        np.array(case["token_ids"]), np.array(case["seq_offsets"]),
        None if case["compress_map"] is None else np.array(case["compress_map"]),
        case["vocab"], case["min_order"], case["num_orders"], case["heads"],
        np.array(case["multipliers"], dtype=np.uint64), np.array(case["primes"], dtype=np.uint64))
    assert got.tolist() == case["expected"]


def _windows(ids_c, offsets, t, n):
    start = max(s for s in offsets[:-1] if s <= t)
    return tuple(int(ids_c[t - j]) if t - j >= start else 0 for j in range(n))


def test_hash_equal_windows_equal_indices_and_range():
    w = W.tiny_hash(seed=3)
    # a longer pack with repeats so that equal windows occur across sequences
    ids = np.concatenate([w.token_ids[:20] % 7, w.token_ids[:20] % 7, w.token_ids[:24] % 5]).astype(np.int32)
    offs = np.array([0, 20, 40, 64], dtype=np.int64)
    s = w.spec
    idx = oracle.hash_indices(ids, offs, w.compress_map, w.vocab, s.min_order, s.num_orders, s.heads,
                              s.multipliers, s.primes)
    assert idx.shape == (64, s.tables)
    assert (idx >= 0).all() and (idx < s.primes.astype(np.int64)[None, :]).all()
    ids_c = w.compress_map[ids]
    seen = {}
    for t in range(64):
        for ni in range(s.num_orders):
            n = s.min_order + ni
            key_w = _windows(ids_c, offs, t, n)
            for k in range(s.heads):
                tb = ni * s.heads + k
                key = (tb, key_w)
                if key in seen:
                    assert seen[key] == idx[t, tb]
                seen[key] = idx[t, tb]
    # determinism: a second call gives identical indices
    idx2 = oracle.hash_indices(ids, offs, w.compress_map, w.vocab, s.min_order, s.num_orders, s.heads,
                               s.multipliers, s.primes)
    assert np.array_equal(idx, idx2)


def test_rows_per_token_do_not_depend_on_table_size():
    w = W.tiny_hash()
    s = w.spec
    for anchor in (1009, 258_000, 10_000_000):
        primes = G.consecutive_primes(anchor, s.tables)
        idx = oracle.hash_indices(w.token_ids, w.seq_offsets, w.compress_map, w.vocab, s.min_order,
                                  s.num_orders, s.heads, s.multipliers, primes)
        assert idx.shape == (w.T, (s.min_order + s.num_orders - 1 - 1) * s.heads)
        assert (idx < primes.astype(np.int64)).all()


def test_hash_bucket_occupancy_matches_uniform_expectation():
    # 3000 distinct bigrams hashed into p = 1009 buckets: a uniform hash fills
    # p * (1 - exp(-N/p)) buckets on average (about 957, sd about 5).
    n = 3000
    rng_ids = G.uniform_int(99, 2 * n, 0, 1 << 20).reshape(n, 2)
    ids = rng_ids.reshape(-1).astype(np.int32)
    offs = np.arange(0, 2 * n + 1, 2, dtype=np.int64)
    mult = G.odd_multipliers(1234, 1, 2)
    p = np.array([1009], dtype=np.uint64)
    idx = oracle.hash_indices(ids, offs, None, 1 << 20, 2, 1, 1, mult, p)[1::2, 0]
    occupied = len(np.unique(idx))
    expect = 1009 * (1 - math.exp(-n / 1009))
    assert abs(occupied - expect) < 40


# ----------------------------------------------------------------------------- gather

def test_gather_returns_the_addressed_rows():
    w = W.tiny_hash(seed=2)
    s = w.spec
    rows, r = s.total_rows, 16
    table = (np.arange(rows * r, dtype=np.float64)).astype(np.float32).reshape(rows, r)  # row q holds q*r + c
    idx = oracle.hash_indices(w.token_ids, w.seq_offsets, w.compress_map, w.vocab, s.min_order, s.num_orders,
                              s.heads, s.multipliers, s.primes)
    out = oracle.gather_rows(table, s.primes, idx)
    offsets = np.concatenate([[0], np.cumsum(s.primes.astype(np.int64))[:-1]])
    q = offsets[None, :] + idx
    assert np.array_equal(out[:, :, 0].astype(np.int64), q * r)
    assert np.array_equal(out - out[:, :, :1], np.broadcast_to(np.arange(r, dtype=np.float32), out.shape))


def test_gather_rejects_out_of_range_index():
    p = np.array([5, 7], dtype=np.uint64)
    table = np.zeros((12, 4), dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.gather_rows(table, p, np.array([[5, 0]]))


# ----------------------------------------------------------------------------- gate forward

def _torch_gate(h, k, v, w_h, w_k, eps):
    d = h.shape[-1]
    nh = F.rms_norm(h, (d,), w_h, eps)
    nk = F.rms_norm(k, (d,), w_k, eps)
    a = torch.sigmoid((nh * nk).sum(-1) / math.sqrt(d))
    return a[:, None] * v, a


def _f64(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 256), ("f32", 1000)])
def test_gate_fwd_matches_torch_rms_norm(dtype, d):
    wl = W.GateWorkload(name="pin", T=24, d=d, dtype=dtype, seed=77 + d)
    x = W.gate_host_inputs(wl)
    res = oracle.gate_fwd(x["h"], x["k"], x["v"], x["w_h"], x["w_k"], 1e-6)
    th = {n: torch.from_numpy(_f64(x[n])) for n in ("h", "k", "v")}
    out, a = _torch_gate(th["h"], th["k"], th["v"], torch.from_numpy(x["w_h"].astype(np.float64)),
                         torch.from_numpy(x["w_k"].astype(np.float64)), 1e-6)
    np.testing.assert_allclose(res["alpha"], a.numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(res["out"], out.numpy(), rtol=1e-12, atol=1e-13)
    rh = 1.0 / np.sqrt((th["h"].numpy() ** 2).mean(-1) + 1e-6)
    np.testing.assert_allclose(res["rstd_h"], rh, rtol=1e-13)
    # the fused-weight form gives the same z (the pages print 1.2e-7 for this identity in fp32)
    z = np.log(res["alpha"] / (1 - res["alpha"]))
    np.testing.assert_allclose(res["z_fused"], z, rtol=1e-9, atol=1e-12)
    assert ((res["alpha"] > 0) & (res["alpha"] < 1)).all()


def test_gate_zero_key_gives_half():
    wl = W.tiny_gate()
    x = W.gate_host_inputs(wl)
    k0 = np.zeros_like(x["k"])
    res = oracle.gate_fwd(x["h"], k0, x["v"], x["w_h"], x["w_k"], 1e-6)
    assert (res["alpha"] == 0.5).all() and (res["dot"] == 0.0).all()
    np.testing.assert_array_equal(res["out"], 0.5 * x["v"].astype(np.float64))


def test_gate_closed_form_for_equal_and_opposite_vectors():
    wl = W.tiny_gate(seed=5)
    x = W.gate_host_inputs(wl)
    d, eps = wl.d, 1e-6
    ones = np.ones(d, dtype=np.float32)
    h = x["h"]
    plus = oracle.gate_fwd(h, h, x["v"], ones, ones, eps)
    minus = oracle.gate_fwd(h, -h, x["v"], ones, ones, eps)
    m = (h.astype(np.float64) ** 2).mean(-1)
    z = math.sqrt(d) * m / (m + eps)
    np.testing.assert_allclose(plus["alpha"], 1 / (1 + np.exp(-z)), rtol=1e-14)
    np.testing.assert_allclose(minus["alpha"], 1 / (1 + np.exp(z)), rtol=1e-13)


def test_gate_is_scale_invariant_without_eps():
    wl = W.tiny_gate(seed=6)
    x = W.gate_host_inputs(wl)
    a = oracle.gate_fwd(x["h"], x["k"], x["v"], x["w_h"], x["w_k"], 0.0)["alpha"]
    b = oracle.gate_fwd((4.0 * x["h"]).astype(np.float32), (0.25 * x["k"]).astype(np.float32), x["v"],
                        x["w_h"], x["w_k"], 0.0)["alpha"]
    np.testing.assert_allclose(a, b, rtol=1e-13)


# ----------------------------------------------------------------------------- gate backward

@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_gate_bwd_matches_torch_autograd(dtype, d):
    wl = W.GateWorkload(name="pin", T=16, d=d, dtype=dtype, seed=300 + d)
    x = W.gate_host_inputs(wl)
    eps = 1e-6
    th = {n: torch.from_numpy(_f64(x[n])).requires_grad_() for n in ("h", "k", "v")}
    wh = torch.from_numpy(x["w_h"].astype(np.float64)).requires_grad_()
    wk = torch.from_numpy(x["w_k"].astype(np.float64)).requires_grad_()
    out, _ = _torch_gate(th["h"], th["k"], th["v"], wh, wk, eps)
    g = torch.from_numpy(_f64(x["dout"]))
    (out * g).sum().backward()
    res = oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], eps)
    for name in ("h", "k", "v"):
        np.testing.assert_allclose(res["d" + name], th[name].grad.numpy(), rtol=1e-10, atol=1e-13)
    # grad of w_h and w_k through the fold w = w_h * w_k
    np.testing.assert_allclose(res["dweight"] * x["w_k"], wh.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(res["dweight"] * x["w_h"], wk.grad.numpy(), rtol=1e-10, atol=1e-13)


def _loss(x, eps):
    r = oracle.gate_fwd(x["h"], x["k"], x["v"], x["w_h"], x["w_k"], eps)
    return float((r["out"] * x["dout"].astype(np.float64)).sum())


def test_gate_bwd_matches_central_finite_differences():
    wl = W.tiny_gate(seed=9)
    x = W.gate_host_inputs(wl)
    eps = 1e-6
    res = oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], eps)
    grads = {"h": res["dh"], "k": res["dk"], "v": res["dv"]}
    delta = 2.0 ** -12
    checked = 0
    for name in ("h", "k", "v"):
        for t, i in [(0, 0), (3, 17), (40, 63), (63, 31)]:
            base = x[name][t, i]
            plus, minus = np.float32(base + delta), np.float32(base - delta)
            if float(plus) - float(base) != delta or float(base) - float(minus) != delta:
                continue  # the perturbation must be exact in fp32
            xp = dict(x); xp[name] = x[name].copy(); xp[name][t, i] = plus
            xm = dict(x); xm[name] = x[name].copy(); xm[name][t, i] = minus
            fd = (_loss(xp, eps) - _loss(xm, eps)) / (2 * delta)
            assert abs(fd - grads[name][t, i]) <= 1e-6 * max(1.0, abs(fd)), (name, t, i)
            checked += 1
    assert checked >= 8
    # the weight gradient: d/dw_h,i = dweight_i * w_k,i
    for i in (0, 5, 33):
        base = x["w_h"][i]
        xp = dict(x); xp["w_h"] = x["w_h"].copy(); xp["w_h"][i] = np.float32(base + delta)
        xm = dict(x); xm["w_h"] = x["w_h"].copy(); xm["w_h"][i] = np.float32(base - delta)
        step = float(xp["w_h"][i]) - float(xm["w_h"][i])
        fd = (_loss(xp, eps) - _loss(xm, eps)) / step
        assert abs(fd - res["dweight"][i] * x["w_k"][i]) <= 1e-6 * max(1.0, abs(fd))


def test_gate_bwd_identities():
    wl = W.tiny_gate(seed=11)
    x = W.gate_host_inputs(wl)
    eps, d = 1e-3, wl.d
    f = oracle.gate_fwd(x["h"], x["k"], x["v"], x["w_h"], x["w_k"], eps)
    b = oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], eps)
    h, k, v, g = (x[n].astype(np.float64) for n in ("h", "k", "v", "dout"))
    a = f["alpha"]
    np.testing.assert_array_equal(b["dv"], a[:, None] * g)
    c = (g * v).sum(-1) * a * (1 - a) * f["rstd_h"] * f["rstd_k"] / math.sqrt(d)
    # h . dh = c * dot * eps * rstd_h^2 (RMSNorm is scale invariant up to eps); same for k
    np.testing.assert_allclose((h * b["dh"]).sum(-1), c * f["dot"] * eps * f["rstd_h"] ** 2, rtol=1e-8, atol=1e-12)
    np.testing.assert_allclose((k * b["dk"]).sum(-1), c * f["dot"] * eps * f["rstd_k"] ** 2, rtol=1e-8, atol=1e-12)
    w = oracle.fuse_weight(x["w_h"], x["w_k"])
    np.testing.assert_allclose((w * b["dweight"]).sum(), (c * f["dot"]).sum(), rtol=1e-10)


def test_gate_bwd_token_ranges_add_up():
    wl = W.tiny_gate(seed=12)
    x = W.gate_host_inputs(wl)
    full = oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], 1e-6)
    a = oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], 1e-6, 0, 20)
    b = oracle.gate_bwd(x["dout"], x["h"], x["k"], x["v"], x["w_h"], x["w_k"], 1e-6, 20, 64)
    np.testing.assert_allclose(a["dweight"] + b["dweight"], full["dweight"], rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(np.concatenate([a["dh"], b["dh"]]), full["dh"])


# ----------------------------------------------------------------------------- fold + reduce

def test_fuse_weight_is_the_elementwise_product():
    a = np.array([1.5, -2.0, 0.25, 3.0], dtype=np.float32)
    b = np.array([2.0, 0.5, -4.0, 1.0 / 3.0], dtype=np.float32)
    np.testing.assert_array_equal(oracle.fuse_weight(a, b), [3.0, -1.0, -1.0, 3.0 * float(np.float32(1.0 / 3.0))])


def test_grad_w_reduce_closed_forms():
    P, d = 37, 12
    ones = np.ones((P, d), dtype=np.float32)
    assert (oracle.grad_w_reduce(ones)["S"] == P).all()
    rows = np.repeat(np.arange(P, dtype=np.float32)[:, None], d, axis=1)
    assert (oracle.grad_w_reduce(rows)["S"] == P * (P - 1) / 2).all()
    cols = np.repeat(np.arange(d, dtype=np.float32)[None, :], P, axis=0)
    wh = np.linspace(0.5, 1.5, d).astype(np.float32)
    wk = np.linspace(2.0, -1.0, d).astype(np.float32)
    r = oracle.grad_w_reduce(cols, wh, wk)
    np.testing.assert_array_equal(r["S"], P * np.arange(d))
    np.testing.assert_array_equal(r["inc_h"], P * np.arange(d) * wk.astype(np.float64))
    np.testing.assert_array_equal(r["inc_k"], P * np.arange(d) * wh.astype(np.float64))
    assert (oracle.grad_w_reduce(np.zeros((0, d), dtype=np.float32))["S"] == 0).all()


# ----------------------------------------------------------------------------- the multi-branch gate

def _torch_gate_hc(x, kv, wh, wk, eps, clamp):
    T, hc, d = x.shape
    k, v = kv[:, :hc], kv[:, hc]
    nx = F.rms_norm(x, (d,), None, eps) * wh
    nk = F.rms_norm(k, (d,), None, eps) * wk
    z = (nx * nk).sum(-1) / math.sqrt(d)
    s = torch.copysign(torch.sqrt(torch.clamp(z.abs(), min=clamp)), z)
    gate = torch.sigmoid(s)
    return x + gate[..., None] * v[:, None, :], gate


@pytest.mark.parametrize("dtype,hc,d", [("f32", 4, 64), ("bf16", 4, 128), ("f32", 1, 96), ("bf16", 2, 256)])
def test_gate_hc_matches_torch_forward_and_autograd(dtype, hc, d):
    wl = W.GateHcWorkload(name="pin", T=12, hc=hc, d=d, dtype=dtype, seed=500 + hc * d)
    x = W.gate_hc_host_inputs(wl)
    t = {n: torch.from_numpy(_f64(x[n])).requires_grad_() for n in ("x", "kv")}
    wh = torch.from_numpy(x["w_h"].astype(np.float64)).requires_grad_()
    wk = torch.from_numpy(x["w_k"].astype(np.float64)).requires_grad_()
    out, gate = _torch_gate_hc(t["x"], t["kv"], wh, wk, wl.eps, wl.clamp)
    f = oracle.gate_hc_fwd(x["x"], x["kv"], x["w_h"], x["w_k"], wl.eps, wl.clamp)
    np.testing.assert_allclose(f["gate"], gate.detach().numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(f["out"], out.detach().numpy(), rtol=1e-12, atol=1e-13)
    g = torch.from_numpy(_f64(x["dout"]))
    (out * g).sum().backward()
    b = oracle.gate_hc_bwd(x["dout"], x["x"], x["kv"], x["w_h"], x["w_k"], wl.eps, wl.clamp)
    np.testing.assert_allclose(b["dx"], t["x"].grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(b["dkv"], t["kv"].grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(b["dweight"] * x["w_k"], wh.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(b["dweight"] * x["w_h"], wk.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_gate_hc_zero_key_hits_the_clamp():
    # k = 0 gives z = 0, held at the clamp: gate = sigmoid(+sqrt(1e-6)) = sigmoid(0.001), and no gradient
    # reaches x or k through the gate (dx = dout exactly, dk = 0); dv = sum_h gate * dout_h.
    wl = W.GateHcWorkload(name="pin", T=6, hc=4, d=32, dtype="f32", seed=77)
    x = W.gate_hc_host_inputs(wl)
    kv = x["kv"].copy()
    kv[:, :4] = 0.0
    f = oracle.gate_hc_fwd(x["x"], kv, x["w_h"], x["w_k"], wl.eps, wl.clamp)
    g0 = 1.0 / (1.0 + math.exp(-0.001))
    assert np.allclose(f["gate"], g0, rtol=0, atol=1e-16)
    np.testing.assert_allclose(f["out"], x["x"] + g0 * kv[:, 4][:, None, :].astype(np.float64), rtol=1e-15)
    b = oracle.gate_hc_bwd(x["dout"], x["x"], kv, x["w_h"], x["w_k"], wl.eps, wl.clamp)
    np.testing.assert_array_equal(b["dx"], x["dout"].astype(np.float64))
    assert (b["dkv"][:, :4] == 0).all() and (b["dweight"] == 0).all()
    np.testing.assert_allclose(b["dkv"][:, 4], g0 * x["dout"].astype(np.float64).sum(1), rtol=1e-14)


def test_gate_hc_finite_differences():
    wl = W.GateHcWorkload(name="pin", T=5, hc=4, d=48, dtype="f32", seed=91)
    x = W.gate_hc_host_inputs(wl)
    b = oracle.gate_hc_bwd(x["dout"], x["x"], x["kv"], x["w_h"], x["w_k"], wl.eps, wl.clamp)

    def loss(xx):
        f = oracle.gate_hc_fwd(xx["x"], xx["kv"], xx["w_h"], xx["w_k"], wl.eps, wl.clamp)
        return float((f["out"] * x["dout"].astype(np.float64)).sum())

    delta = 2.0 ** -12
    checked = 0
    for name, grad, idx in (("x", b["dx"], [(0, 0, 0), (3, 2, 17), (4, 3, 47)]),
                            ("kv", b["dkv"], [(1, 0, 5), (2, 3, 30), (0, 4, 7), (4, 4, 40)])):
        for ix in idx:
            base = x[name][ix]
            plus, minus = np.float32(base + delta), np.float32(base - delta)
            if float(plus) - float(base) != delta or float(base) - float(minus) != delta:
                continue
            xp = dict(x); xp[name] = x[name].copy(); xp[name][ix] = plus
            xm = dict(x); xm[name] = x[name].copy(); xm[name][ix] = minus
            fd = (loss(xp) - loss(xm)) / (2 * delta)
            assert abs(fd - grad[ix]) <= 1e-6 * max(1.0, abs(fd)), (name, ix)
            checked += 1
    assert checked >= 5


# ----------------------------------------------------------------------------- the Engram Sinkhorn

def test_sinkhorn_row_step_against_numpy_norms():
    R, D, eps = 37, 50, 1e-6
    m = G.normal(601, R * D).astype(np.float32).reshape(R, D)
    ones_r, ones_c = np.ones(R, dtype=np.float32), np.ones(D, dtype=np.float32)
    r = oracle.sinkhorn_step(m, ones_r, ones_c, eps)
    norms = np.linalg.norm(m.astype(np.float64), axis=1)
    np.testing.assert_allclose(r["row_norm"], norms, rtol=1e-13)
    np.testing.assert_allclose(r["row_scale"], 1.0 / (norms + eps), rtol=1e-13)
    unit = m.astype(np.float64) / (norms + eps)[:, None]
    np.testing.assert_allclose(r["col_sumsq"], np.linalg.norm(unit, axis=0) ** 2, rtol=1e-12)
    # scales enter as row_scale * m * col_scale: scaling m by 3 and row_scale by 1/3 changes nothing
    rs = np.full(R, 1.0 / 3.0, dtype=np.float32)
    r3 = oracle.sinkhorn_step((3 * m).astype(np.float32), rs, ones_c, eps)
    np.testing.assert_allclose(r3["row_norm"], norms, rtol=1e-6)
    # row ranges partition the column sums
    a = oracle.sinkhorn_step(m, ones_r, ones_c, eps, 0, 20)
    b = oracle.sinkhorn_step(m, ones_r, ones_c, eps, 20, R)
    np.testing.assert_allclose(a["col_sumsq"] + b["col_sumsq"], r["col_sumsq"], rtol=1e-13)


def _sinkhorn_iterate(m, steps, eps=1e-6):
    R, D = m.shape
    rs, cs = np.ones(R, dtype=np.float32), np.ones(D, dtype=np.float32)
    col_l2 = None
    for _ in range(steps):
        st = oracle.sinkhorn_step(m, rs, cs, eps)
        rs = st["row_scale"].astype(np.float32)
        col_l2 = np.sqrt(st["col_sumsq"])                 # column norms seen before the column step
        cs = oracle.sinkhorn_col_update(st["col_sumsq"], cs, eps).astype(np.float32)
    it = rs[:, None].astype(np.float64) * m * cs[None, :]
    return rs, cs, col_l2, np.linalg.norm(it, axis=1)     # row norms seen before finalize


def test_sinkhorn_fixed_point_matches_the_printed_walkthrough():
    with open(os.path.join(os.path.dirname(__file__), "golden", "sinkhorn_demo.json")) as f:
        demo = json.load(f)
    R, D, alpha = demo["rows"], demo["head_dim"], demo["alpha"]
    m = np.abs(G.normal(602, R * D)).astype(np.float32).reshape(R, D) + 0.1
    rs, cs, col_l2, row_l2 = _sinkhorn_iterate(m, 60)
    fp = demo["fixed_point"]
    np.testing.assert_allclose(col_l2, fp["col_l2_before_col_step"], rtol=1e-5)
    np.testing.assert_allclose(row_l2, fp["row_l2_before_finalize"], rtol=1e-5)
    # the pages' printed values lie next to the same fixed point (their run stopped at step 7)
    assert np.allclose(demo["printed"]["col_l2_before_col_step_step7"], fp["col_l2_before_col_step"], atol=1e-3)
    assert np.allclose(demo["printed"]["row_l2_before_finalize"], fp["row_l2_before_finalize"], atol=1e-3)
    out = oracle.sinkhorn_finalize(m, rs, cs, 1e-6, alpha)
    np.testing.assert_allclose(np.linalg.norm(out, axis=1), demo["printed"]["row_l2_after_finalize"], rtol=1e-5)
    # after a row step every row of the iterate is a unit vector (up to eps)
    st = oracle.sinkhorn_step(m, rs, cs, 1e-6)
    it = st["row_scale"][:, None] * m * cs[None, :]
    assert np.abs(np.linalg.norm(it, axis=1) - 1).max() < 1e-5


def test_sinkhorn_momentum_closed_forms():
    g = G.normal(603, 64).astype(np.float32)
    m0 = np.zeros(64, dtype=np.float32)
    plain = oracle.sinkhorn_momentum(g, m0, 0.9, False)
    nest = oracle.sinkhorn_momentum(g, m0, 0.9, True)
    np.testing.assert_array_equal(plain["momentum"], g.astype(np.float64))
    np.testing.assert_array_equal(plain["input"], g.astype(np.float64))
    np.testing.assert_allclose(nest["input"], 1.9 * g.astype(np.float64), rtol=1e-15)
    m1 = plain["momentum"].astype(np.float32)
    second = oracle.sinkhorn_momentum(g, m1, 0.5, False)
    np.testing.assert_allclose(second["momentum"], 1.5 * g.astype(np.float64), rtol=1e-7)
    zero_beta = oracle.sinkhorn_momentum(g, m1, 0.0, True)
    np.testing.assert_array_equal(zero_beta["input"], g.astype(np.float64))


def test_sinkhorn_nesterov_with_prior_momentum():
    # m' = beta m0 + g and input = g + beta m' = (1 + beta) g + beta^2 m0: with m0 != 0 this tells the
    # Nesterov look-ahead apart from m' + beta g, which agrees with it only when m0 = 0.
    g = G.normal(604, 32).astype(np.float32)
    m0 = G.normal(605, 32).astype(np.float32)
    beta = 0.75
    r = oracle.sinkhorn_momentum(g, m0, beta, True)
    expect = (1 + beta) * g.astype(np.float64) + beta ** 2 * m0.astype(np.float64)
    np.testing.assert_allclose(r["input"], expect, rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------------------------- the short conv after the gate

def _conv_case(lengths, d, w, dil, seed, dtype="f32", bias=True):
    T = int(sum(lengths))
    v = G.normal(seed, T * d).reshape(T, d)
    h = G.normal(seed + 1, T * d).reshape(T, d)
    g = G.normal(seed + 2, T * d).reshape(T, d)
    conv = lambda a: a.astype(np.float32) if dtype == "f32" else G.to_bf16_bits(a)
    return dict(v=conv(v), h=conv(h), g=conv(g), norm_w=G.normal(seed + 3, d, 1.0, 0.1).astype(np.float32),
                conv_w=G.normal(seed + 4, d * w, 0.0, 0.5).astype(np.float32).reshape(d, w),
                bias=G.normal(seed + 5, d, 0.0, 0.1).astype(np.float32) if bias else None,
                offs=G.offsets_from_lengths(lengths), dil=dil, T=T, d=d, w=w)


def _as64(a):
    return torch.from_numpy((a.astype(np.uint32) << 16).view(np.float32).astype(np.float64) if a.dtype == np.uint16
                            else a.astype(np.float64))


def _torch_short_conv(c, eps, v=None, norm_w=None, conv_w=None, bias=None):
    """torch's rms_norm + depthwise conv1d (dilation, left padding, per sequence) + silu, fp64."""
    v = _as64(c["v"]) if v is None else v
    nw = torch.from_numpy(c["norm_w"].astype(np.float64)) if norm_w is None else norm_w
    cw = torch.from_numpy(c["conv_w"].astype(np.float64)) if conv_w is None else conv_w
    b = (None if c["bias"] is None else torch.from_numpy(c["bias"].astype(np.float64))) if bias is None else bias
    u = torch.nn.functional.rms_norm(v, (c["d"],), nw, eps)
    pad = (c["w"] - 1) * c["dil"]
    outs = []
    for s in range(len(c["offs"]) - 1):
        a, e = int(c["offs"][s]), int(c["offs"][s + 1])
        if a == e:
            continue
        x = u[a:e].T.unsqueeze(0)
        y = torch.nn.functional.conv1d(x, cw.unsqueeze(1), b, padding=pad, dilation=c["dil"], groups=c["d"])
        outs.append(y[0, :, : e - a].T)
    conv = torch.cat(outs)
    return conv, _as64(c["h"]) + torch.nn.functional.silu(conv) + v


@pytest.mark.parametrize("lengths,d,w,dil,dtype", [([13, 9], 6, 4, 3, "f32"), ([20], 5, 4, 1, "bf16"),
                                                    ([4, 0, 11, 2], 3, 3, 2, "f32"), ([7], 4, 1, 3, "f32")])
def test_short_conv_against_torch_conv1d(lengths, d, w, dil, dtype):
    c = _conv_case(lengths, d, w, dil, 610 + d, dtype)
    eps = 1e-6
    r = oracle.short_conv_fwd(c["v"], c["h"], c["norm_w"], c["conv_w"], c["bias"], c["offs"], dil, eps)
    conv, out = _torch_short_conv(c, eps)
    np.testing.assert_allclose(r["c"], conv.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["out"], out.numpy(), rtol=1e-12, atol=1e-13)
    vv = _as64(c["v"]).numpy()
    np.testing.assert_allclose(r["rstd"], 1 / np.sqrt((vv ** 2).mean(axis=1) + eps), rtol=1e-14)


def test_short_conv_backward_against_autograd():
    c = _conv_case([13, 1, 9], 6, 4, 3, 620, "f32")
    eps = 1e-6
    v = _as64(c["v"]).requires_grad_()
    nw = torch.from_numpy(c["norm_w"].astype(np.float64)).requires_grad_()
    cw = torch.from_numpy(c["conv_w"].astype(np.float64)).requires_grad_()
    b = torch.from_numpy(c["bias"].astype(np.float64)).requires_grad_()
    _, out = _torch_short_conv(c, eps, v, nw, cw, b)
    (out * _as64(c["g"])).sum().backward()
    r = oracle.short_conv_bwd(c["g"], c["v"], c["norm_w"], c["conv_w"], c["bias"], c["offs"], 3, eps)
    np.testing.assert_allclose(r["dv"], v.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r["dconv_w"], cw.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r["dbias"], b.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r["dnorm_w"], nw.grad.numpy(), rtol=1e-10, atol=1e-12)
    # token ranges partition the weight gradients and give the same per-token rows
    a = oracle.short_conv_bwd(c["g"], c["v"], c["norm_w"], c["conv_w"], c["bias"], c["offs"], 3, eps, 0, 10)
    z = oracle.short_conv_bwd(c["g"], c["v"], c["norm_w"], c["conv_w"], c["bias"], c["offs"], 3, eps, 10, c["T"])
    for k in ("dconv_w", "dbias", "dnorm_w"):
        np.testing.assert_allclose(a[k] + z[k], r[k], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(np.concatenate([a["dv"], z["dv"]]), r["dv"], rtol=1e-13, atol=1e-15)


def test_short_conv_closed_forms():
    c = _conv_case([10, 7], 4, 4, 3, 630, "f32", bias=False)
    eps = 1e-6
    vv, hh = _as64(c["v"]).numpy(), _as64(c["h"]).numpy()
    u = vv / np.sqrt((vv ** 2).mean(axis=1, keepdims=True) + eps) * c["norm_w"].astype(np.float64)
    silu = lambda x: x / (1 + np.exp(-x))
    # the current-token tap alone: c = u
    delta = np.zeros((4, 4), dtype=np.float32)
    delta[:, 3] = 1
    r = oracle.short_conv_fwd(c["v"], c["h"], c["norm_w"], delta, None, c["offs"], 3, eps)
    np.testing.assert_allclose(r["c"], u, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r["out"], hh + silu(u) + vv, rtol=1e-13)
    # the oldest tap alone: c[t] = u[t - 9] inside a sequence, 0 for its first 9 tokens (SiLU(0) = 0)
    old = np.zeros((4, 4), dtype=np.float32)
    old[:, 0] = 1
    r = oracle.short_conv_fwd(c["v"], None, c["norm_w"], old, None, c["offs"], 3, eps)
    for s0, s1 in ((0, 10), (10, 17)):
        np.testing.assert_array_equal(r["c"][s0:min(s1, s0 + 9)], 0)
        np.testing.assert_array_equal(r["out"][s0:min(s1, s0 + 9)], vv[s0:min(s1, s0 + 9)])
        for t in range(s0 + 9, s1):
            np.testing.assert_allclose(r["c"][t], u[t - 9], rtol=1e-14)
    # SiLU'(0) = 1/2: with every tap 0 and bias 0, dv = g and the weight gradients follow from dc = g / 2
    zero = np.zeros((4, 4), dtype=np.float32)
    b = oracle.short_conv_bwd(c["g"], c["v"], c["norm_w"], zero, None, c["offs"], 3, eps)
    np.testing.assert_allclose(b["dv"], _as64(c["g"]).numpy(), rtol=1e-15)
    np.testing.assert_allclose(b["dbias"], _as64(c["g"]).numpy().sum(0) / 2, rtol=1e-13)
    np.testing.assert_array_equal(b["dnorm_w"], 0)
