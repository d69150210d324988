"""The C-ABI library on a machine without a GPU: it builds, loads, exports every
symbol include/engram.h declares, and rejects bad arguments on the host before
touching the device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "engram.h")


@pytest.fixture(scope="module")
def lib():
    from engram_conditional_memory_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(engram_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    # the hot path's entry points and the error reader, under the names the scope table gives them
    for required in ("engram_hash_gather", "engram_fuse_weight", "engram_gate_fwd", "engram_gate_bwd",
                     "engram_gate_bwd_num_partials", "engram_grad_w_reduce", "engram_get_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_side_rejections(lib):
    st = ctypes.c_int
    lib.engram_gate_fwd.restype = st
    lib.engram_gate_fwd.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                                            ctypes.c_float] + [ctypes.c_void_p] * 6
    lib.engram_gate_fwd.argtypes[3] = ctypes.c_int
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: each call below fails before any CUDA call
    odd = ctypes.c_void_p(0x10008)
    # NULL input
    assert lib.engram_gate_fwd(None, fake, fake, 1, fake, 8, 64, 1e-6, fake, None, None, None, None, None) == 1
    # unknown dtype
    assert lib.engram_gate_fwd(fake, fake, fake, 7, fake, 8, 64, 1e-6, fake, None, None, None, None, None) == 3
    # negative T, and a row that is not a multiple of 16 bytes (d = 4 bf16)
    assert lib.engram_gate_fwd(fake, fake, fake, 1, fake, -1, 64, 1e-6, fake, None, None, None, None, None) == 2
    assert lib.engram_gate_fwd(fake, fake, fake, 1, fake, 8, 4, 1e-6, fake, None, None, None, None, None) == 4
    # row too long (8200 bf16 > 16 KB) and a misaligned tensor
    assert lib.engram_gate_fwd(fake, fake, fake, 1, fake, 8, 8200, 1e-6, fake, None, None, None, None, None) == 2
    assert lib.engram_gate_fwd(odd, fake, fake, 1, fake, 8, 64, 1e-6, fake, None, None, None, None, None) == 4
    lib.engram_last_error_string.restype = ctypes.c_char_p
    assert b"aligned" in lib.engram_last_error_string()

    lib.engram_grad_w_reduce.restype = st
    lib.engram_grad_w_reduce.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32] + [ctypes.c_void_p] * 6
    assert lib.engram_grad_w_reduce(None, 4, 64, fake, None, None, None, None, None) == 1
    assert lib.engram_grad_w_reduce(fake, 4, 64, None, None, None, None, None, None) == 1  # no output
    assert lib.engram_grad_w_reduce(fake, 4, 64, fake, fake, None, None, None, None) == 1  # weights not all given
    assert lib.engram_grad_w_reduce(fake, 4, 66, fake, None, None, None, None, None) == 4
    assert lib.engram_grad_w_reduce(fake, -1, 64, fake, None, None, None, None, None) == 2


def test_newer_entry_points_reject_on_the_host(lib):
    """The gate with its output statistic, the conv taking it, the conv's reduction and the
    multi-branch gate's knob: argument errors come back before any CUDA call."""
    st, vp, i32, i64, f32 = ctypes.c_int, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    fake = vp(0x10000)
    g = lib.engram_gate_fwd_rms
    g.restype = st
    g.argtypes = [vp, vp, vp, ctypes.c_int, vp, i64, i32, f32, vp, vp, vp, vp, vp, vp, f32, vp]
    assert g(fake, fake, fake, 1, fake, 8, 64, 1e-6, fake, None, None, None, None, None, 1e-6, None) == 1  # no out_rstd
    assert g(None, fake, fake, 1, fake, 8, 64, 1e-6, fake, None, None, None, None, fake, 1e-6, None) == 1
    assert g(fake, fake, fake, 7, fake, 8, 64, 1e-6, fake, None, None, None, None, fake, 1e-6, None) == 3
    c = lib.engram_short_conv_fwd_given_rstd
    c.restype = st
    c.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, vp, vp]
    assert c(fake, None, 1, fake, fake, None, fake, 1, 8, 64, 4, 3, None, fake, None) == 1  # no rstd
    assert c(fake, None, 1, fake, fake, None, fake, 1, 8, 64, 5, 3, fake, fake, None) == 2  # width 5
    assert c(fake, None, 1, fake, fake, None, fake, 1, 8, 64, 4, 0, fake, fake, None) == 2  # dilation 0
    r = lib.engram_short_conv_grad_reduce
    r.restype = st
    r.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
    assert r(fake, 4, 4, 6, fake, None, fake, None) == 4  # d not a multiple of 4
    assert r(None, 4, 4, 64, fake, None, fake, None) == 1
    k = lib.engram_set_hc_split
    k.restype, k.argtypes = i32, [i32]
    assert k(1) == 0 and k(0) == 1 and k(0) == 0
    assert k(2) == 0 and k(4) == 2 and k(7) == 4 and k(0) == 0  # modes 0, 1, 2, 4; any other value is 0


def test_partition_rule(lib):
    lib.engram_gate_bwd_num_partials.restype = ctypes.c_int
    lib.engram_gate_bwd_num_partials.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
    P = ctypes.c_int32()

    def parts(T, d=4096):
        assert lib.engram_gate_bwd_num_partials(T, d, ctypes.byref(P)) == 0
        return P.value

    assert parts(0) == 1 and parts(1) == 1 and parts(16) == 1 and parts(17) == 2
    assert parts(4096) == 256 and parts(16384) == 1024 and parts(131072) == 1024
    for T in (1, 100, 4096, 16384, 32768, 131072, 139_000):
        p = parts(T)
        chunk = -(-T // p)
        assert 1 <= p <= 1024 and chunk >= min(T, 15) and (p - 1) * chunk < T <= p * chunk
    assert lib.engram_gate_bwd_num_partials(-1, 64, ctypes.byref(P)) == 2


def test_hash_gather_host_rejections(lib):
    import numpy as np

    from engram_conditional_memory_gb300.binding import _HashGatherArgs, _HashSpec

    lib.engram_hash_gather.restype = ctypes.c_int
    lib.engram_hash_gather.argtypes = [ctypes.c_void_p] * 3
    mult = np.ones((4, 3), dtype=np.uint64)
    primes = np.array([5, 7, 11, 13], dtype=np.uint64)
    spec = _HashSpec(2, 2, 2, 3, mult.ctypes.data, primes.ctypes.data)
    fake = 0x10000
    args = _HashGatherArgs(fake, 10, fake, 1, None, 100, 100, fake, 36, 8, 1, None, fake, None)
    # too few table rows for sum(primes) = 36 - 1
    args.table_rows = 35
    assert lib.engram_hash_gather(ctypes.byref(spec), ctypes.byref(args), None) == 2
    args.table_rows = 36
    args.row_dim = 4  # 8-byte rows
    assert lib.engram_hash_gather(ctypes.byref(spec), ctypes.byref(args), None) == 4
    args.row_dim = 16384  # 4 tables x 32 KB rows = a 128 KB e_t row, over the 64 KB the kernel takes
    args.table_rows = 1 << 20
    assert lib.engram_hash_gather(ctypes.byref(spec), ctypes.byref(args), None) == 2
    args.row_dim = 8
    args.table_rows = 36
    bad = _HashSpec(2, 2, 2, 2, mult.ctypes.data, primes.ctypes.data)  # stride 2 < max order 3
    assert lib.engram_hash_gather(ctypes.byref(bad), ctypes.byref(args), None) == 2
    many = _HashSpec(2, 2, 17, 3, mult.ctypes.data, primes.ctypes.data)  # 34 tables > 32
    assert lib.engram_hash_gather(ctypes.byref(many), ctypes.byref(args), None) == 2
    zero = np.array([5, 0, 11, 13], dtype=np.uint64)
    zspec = _HashSpec(2, 2, 2, 3, mult.ctypes.data, zero.ctypes.data)
    assert lib.engram_hash_gather(ctypes.byref(zspec), ctypes.byref(args), None) == 2
    args.out_rows = None
    assert lib.engram_hash_gather(ctypes.byref(spec), ctypes.byref(args), None) == 1  # no output at all
    args.token_ids = None
    args.out_rows = fake
    assert lib.engram_hash_gather(ctypes.byref(spec), ctypes.byref(args), None) == 1  # NULL ids with T > 0


def test_sinkhorn_host_side_rejections(lib):
    """Argument errors of the Sinkhorn calls are caught on the host, before any CUDA call."""
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.engram_sinkhorn_step.restype = ctypes.c_int
    lib.engram_sinkhorn_step.argtypes = [vp, vp, vp, i64, i32, f32, vp, vp, i32, vp]
    lib.engram_sinkhorn_step_reduce.restype = ctypes.c_int
    lib.engram_sinkhorn_step_reduce.argtypes = [vp, i32, i32, vp, vp, f32, vp]
    lib.engram_sinkhorn_finalize.restype = ctypes.c_int
    lib.engram_sinkhorn_finalize.argtypes = [vp, vp, vp, i64, i32, f32, f32, vp, vp]
    lib.engram_sinkhorn_momentum_update.restype = ctypes.c_int
    lib.engram_sinkhorn_momentum_update.argtypes = [vp, ctypes.c_int, vp, vp, i64, f32, i32, vp]
    fake, odd = vp(0x10000), vp(0x10008)
    step = lib.engram_sinkhorn_step
    assert step(fake, fake, fake, 64, 130, 1e-6, None, fake, 4, None) == 4       # head_dim not a multiple of 4
    assert step(fake, fake, fake, 64, 8196, 1e-6, None, fake, 4, None) == 2      # head_dim above 8192
    assert step(fake, fake, fake, -1, 64, 1e-6, None, fake, 4, None) == 2
    assert step(fake, fake, fake, 64, 64, 1e-6, None, fake, 0, None) == 2        # P = 0
    assert step(None, fake, fake, 64, 64, 1e-6, None, fake, 4, None) == 1
    assert step(fake, fake, fake, 64, 64, 1e-6, None, None, 4, None) == 1        # no partials
    assert step(odd, fake, fake, 64, 64, 1e-6, None, fake, 4, None) == 4
    red = lib.engram_sinkhorn_step_reduce
    assert red(fake, 4, 64, None, None, 1e-6, None) == 1                         # neither output
    assert red(fake, 0, 64, fake, None, 1e-6, None) == 2
    assert red(fake, 4, 66, fake, None, 1e-6, None) == 4
    assert red(fake, 4, 64, odd, None, 1e-6, None) == 4
    fin = lib.engram_sinkhorn_finalize
    assert fin(fake, fake, fake, 0, 64, 1e-6, 1.0, fake, None) == 0              # no row: nothing to do
    assert fin(fake, fake, fake, 8, 64, 1e-6, 1.0, None, None) == 1
    assert fin(fake, fake, fake, 8, 64, 1e-6, 1.0, fake, None) == 2              # out aliases matrix
    mom = lib.engram_sinkhorn_momentum_update
    assert mom(fake, 1, fake, vp(0x20000), 0, 0.9, 1, None) == 0                 # n = 0
    assert mom(fake, 9, fake, vp(0x20000), 16, 0.9, 1, None) == 3                # dtype
    assert mom(fake, 1, fake, fake, 16, 0.9, 1, None) == 2                       # input aliases momentum
    assert mom(fake, 1, odd, vp(0x20000), 16, 0.9, 1, None) == 4
    assert mom(None, 1, fake, vp(0x20000), 16, 0.9, 1, None) == 1


def test_sinkhorn_partition_rule(lib):
    lib.engram_sinkhorn_num_partials.restype = ctypes.c_int
    lib.engram_sinkhorn_num_partials.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
    P = ctypes.c_int32()

    def parts(rows):
        assert lib.engram_sinkhorn_num_partials(rows, 5120, ctypes.byref(P)) == 0
        return P.value

    assert parts(0) == 1 and parts(16) == 1 and parts(17) == 2 and parts(16384) == 1024 and parts(10**7) == 1024
    for rows in (1, 15, 100, 8192, 16385, 10**6):
        p = parts(rows)
        chunk = -(-rows // p)
        assert 1 <= p <= 1024 and (p - 1) * chunk < rows <= p * chunk


def test_wait_timeout_check_rejects_bad_limits(lib):
    lib.engram_check_wait_timeout.restype = ctypes.c_int
    lib.engram_check_wait_timeout.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
    assert lib.engram_check_wait_timeout(0, None) == 2
    assert lib.engram_check_wait_timeout(2000001, None) == 2


def test_short_conv_backward_rejects_on_the_host(lib):
    """engram_short_conv_bwd and its partial count: a wrong P, missing pointers, dv over an input, and
    bad width or dilation come back before any CUDA call; P is (time chunks) x dilation with chunks
    of max(256, ceil(T / 256)) tokens."""
    st, vp, i32, i64 = ctypes.c_int, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    n = lib.engram_short_conv_num_partials
    n.restype, n.argtypes = st, [i64, i32, ctypes.POINTER(i32)]
    P = i32()

    def parts(T, dil):
        assert n(T, dil, ctypes.byref(P)) == 0
        return P.value

    assert parts(16384, 3) == 64 * 3 and parts(513, 3) == 3 * 3 and parts(513, 40) == 3 * 40
    assert parts(70004, 3) == 256 * 3 and parts(1, 1) == 1
    assert n(-1, 3, ctypes.byref(P)) == 2 and n(16, 0, ctypes.byref(P)) == 2 and n(16, 3, None) == 1
    b = lib.engram_short_conv_bwd
    b.restype = st
    b.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, vp, i32, vp]
    f = [vp(0x10000 + 0x1000 * i) for i in range(8)]  # dout, v, norm_w, conv_w, rstd, offsets, dv, partials
    ok = parts(513, 3)

    def call(dout=f[0], v=f[1], dt=1, nw=f[2], cw=f[3], rstd=f[4], offs=f[5], T=513, d=64, width=4, dil=3, dv=f[6],
             part=f[7], P_=ok):
        return b(dout, v, dt, nw, cw, None, rstd, offs, 1, T, d, width, dil, dv, part, P_, None)

    assert call(P_=ok + 1) == 2                      # P not the partial count
    assert call(dil=40) == 2                         # P of dilation 3 for dilation 40
    assert call(width=5) == 2 and call(dil=0) == 2   # width above 4, no dilation
    assert call(dt=7) == 3                           # no such dtype
    assert call(rstd=None) == 1 and call(dv=None) == 1 and call(part=None) == 1 and call(nw=None) == 1
    assert call(dv=f[1]) == 2 and call(dv=f[0]) == 2  # dv over V~ or over dout


def test_multi_branch_gate_rejects_on_the_host(lib):
    """engram_gate_hc_fwd / _bwd: missing pointers, a branch count other than 1, 2 or 4, rows not a
    multiple of 16 bytes, a negative clamp, no partials, in place with saved statistics, and outputs
    that overlap an input other than in place, all before any CUDA call."""
    st, vp, i32, i64, f32 = ctypes.c_int, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    T, hc, d = 8, 4, 64
    xb, kvb = T * hc * d * 2, T * (hc + 1) * d * 2  # bytes of x-like and kv-like tensors (bf16)
    base = 0x100000
    dout, x, kv, w, stat, dx, dkv, part = (vp(base + i * 0x10000) for i in range(8))
    fw = lib.engram_gate_hc_fwd
    fw.restype = st
    fw.argtypes = [vp, vp, ctypes.c_int, vp, i64, i32, i32, f32, f32, vp, vp, vp, vp, vp, vp]

    def fwd(x_=x, kv_=kv, dt=1, hc_=hc, d_=d, clamp=1e-6, out=dx, gate=stat, w_=w):
        return fw(x_, kv_, dt, w_, T, hc_, d_, 1e-6, clamp, out, gate, None, None, None, None)

    assert fwd(x_=None) == 1 and fwd(w_=None) == 1
    assert fwd(hc_=3) == 2 and fwd(dt=9) == 3 and fwd(d_=60) == 4 and fwd(clamp=-1.0) == 2
    assert fwd(out=x) == 2  # in place with a saved statistic
    bw = lib.engram_gate_hc_bwd
    bw.restype = st
    bw.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, i64, i32, i32, f32, vp, vp, vp, i32, vp]

    def bwd(dx_=dx, dkv_=dkv, part_=part, P=1, hc_=hc, clamp=1e-6):
        return bw(dout, x, kv, 1, w, stat, stat, stat, stat, T, hc_, d, clamp, dx_, dkv_, part_, P, None)

    assert bwd(part_=None) == 1 and bwd(dx_=None) == 1
    assert bwd(P=0) == 2 and bwd(hc_=8) == 2 and bwd(clamp=-0.5) == 2
    assert bwd(dx_=kv) == 2                                   # dx over the keys
    assert bwd(dx_=vp(dout.value + 16)) == 2                  # dx shifted against dout
    assert bwd(dkv_=x) == 2 and bwd(dx_=dkv) == 2             # dkv over x; dx over dkv
    assert xb < 0x10000 and kvb < 0x10000                     # the fake tensors do not overlap one another
