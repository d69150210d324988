"""Synthetic workloads for the Engram hot path: shapes, sizes and value distributions.

Each workload is a plain description (sizes + seeds) plus host-side draws of its
small inputs.  Large dense tensors (activations, the multi-GB embedding table)
are drawn on the device by `synth.device` from the same seeds.

Workloads (the sizes the benchmark and the parity tests use):

* ``tiny``: one sequence of 64 tokens, ids uniform in [0, 1000), a random
  surjection 1000 -> 770, N-gram orders {2, 3} with 2 heads each (4 tables,
  consecutive primes from 1009), fp32 table rows of 16 drawn N(0, 0.02); gate
  with d = 64 in fp32, h/k/v/dout N(0, 1), w_h/w_k N(1, 0.1), eps = 1e-6.
* ``gate_fwd_2k``: gate forward, T = 8192, d = 2048, bf16.
* ``gate_train_4k``: gate fwd + bwd + grad_w reduce, T = 16384, d = 4096, bf16.
* ``hash_gather_64k``: 16 sequences x 4096 tokens, ids Zipf(1.1) over a
  128000-id vocabulary compressed to 98560 ids (the 23 % shrink the Engram
  paper reports for its 128k tokenizer), orders {2, 3} x 8 heads = 16 tables of
  consecutive primes from 2,000,003 rows, rows of 64 bf16 drawn N(0, 0.02)
  (4.1 GB resident).
* ``gate_sweep_7k``: d = 7168, T in {4096, 32768, 131072}, plus a ragged pack of
  64 sequences with lengths uniform in [256, 4096].
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import generators as G


@dataclass
class HashSpec:
    """The fixed hyper-parameters of the multi-head N-gram hash."""

    min_order: int
    num_orders: int
    heads: int
    multipliers: np.ndarray  # uint64 [tables, max_order]
    primes: np.ndarray  # uint64 [tables]

    @property
    def tables(self) -> int:
        return self.num_orders * self.heads

    @property
    def max_order(self) -> int:
        return self.min_order + self.num_orders - 1

    @property
    def total_rows(self) -> int:
        return int(self.primes.astype(np.int64).sum())


@dataclass
class HashGatherWorkload:
    name: str
    token_ids: np.ndarray  # int32 [T]
    seq_offsets: np.ndarray  # int64 [S+1]
    compress_map: np.ndarray | None  # int32 [vocab]
    vocab: int
    vocab_c: int
    spec: HashSpec
    row_dim: int
    dtype: str  # "f32" | "bf16"
    table_seed: int
    table_std: float = 0.02
    table_host: np.ndarray | None = None  # drawn on the host for small tables

    @property
    def T(self) -> int:
        return int(self.token_ids.shape[0])


@dataclass
class GateWorkload:
    name: str
    T: int
    d: int
    dtype: str  # "f32" | "bf16"
    seed: int
    eps: float = 1e-6
    seq_lengths: np.ndarray | None = None  # ragged packs: lengths (the gate sees one T)
    extra: dict = field(default_factory=dict)


def hash_spec(seed: int, min_order: int, num_orders: int, heads: int, prime_anchor: int) -> HashSpec:
    tables = num_orders * heads
    max_order = min_order + num_orders - 1
    return HashSpec(
        min_order=min_order,
        num_orders=num_orders,
        heads=heads,
        multipliers=G.odd_multipliers(seed, tables, max_order),
        primes=G.consecutive_primes(prime_anchor, tables),
    )


def tiny_hash(seed: int = 1) -> HashGatherWorkload:
    T, vocab, vocab_c = 64, 1000, 770
    spec = hash_spec(seed * 7919 + 11, 2, 2, 2, 1009)
    table = G.normal(seed * 31 + 5, spec.total_rows * 16, 0.0, 0.02).astype(np.float32)
    return HashGatherWorkload(
        name="tiny",
        token_ids=G.uniform_int(seed * 17 + 3, T, 0, vocab).astype(np.int32),
        seq_offsets=np.array([0, T], dtype=np.int64),
        compress_map=G.surjection(seed * 13 + 1, vocab, vocab_c),
        vocab=vocab,
        vocab_c=vocab_c,
        spec=spec,
        row_dim=16,
        dtype="f32",
        table_seed=seed * 31 + 5,
        table_host=table.reshape(spec.total_rows, 16),
    )


def hash_gather_64k(seed: int = 4, num_seqs: int = 16, seq_len: int = 4096) -> HashGatherWorkload:
    vocab, vocab_c = 128000, 98560
    T = num_seqs * seq_len
    spec = hash_spec(seed * 7919 + 11, 2, 2, 8, 2_000_003)
    return HashGatherWorkload(
        name=f"hash_gather_{num_seqs}x{seq_len}",
        token_ids=G.zipf_ids(seed * 17 + 3, T, vocab, 1.1).astype(np.int32),
        seq_offsets=G.offsets_from_lengths([seq_len] * num_seqs),
        compress_map=G.surjection(seed * 13 + 1, vocab, vocab_c),
        vocab=vocab,
        vocab_c=vocab_c,
        spec=spec,
        row_dim=64,
        dtype="bf16",
        table_seed=seed * 31 + 5,
    )


def tiny_gate(seed: int = 1) -> GateWorkload:
    return GateWorkload(name="tiny", T=64, d=64, dtype="f32", seed=seed * 101 + 7)


def gate_fwd_2k(seed: int = 2) -> GateWorkload:
    return GateWorkload(name="gate_fwd_T8192_d2048", T=8192, d=2048, dtype="bf16", seed=seed * 101 + 7)


def gate_train_4k(seed: int = 3) -> GateWorkload:
    return GateWorkload(name="gate_train_T16384_d4096", T=16384, d=4096, dtype="bf16", seed=seed * 101 + 7)


def gate_sweep_7k(T: int, seed: int = 5) -> GateWorkload:
    return GateWorkload(name=f"gate_sweep_T{T}_d7168", T=T, d=7168, dtype="bf16", seed=seed * 101 + 7 + T)


def gate_ragged_7k(seed: int = 5) -> GateWorkload:
    lengths = G.ragged_lengths(seed * 977 + 1, 64, 256, 4096)
    return GateWorkload(
        name="gate_ragged64_d7168",
        T=int(lengths.sum()),
        d=7168,
        dtype="bf16",
        seed=seed * 101 + 9,
        seq_lengths=lengths,
    )


def gate_host_inputs(w: GateWorkload):
    """Host draws of a (small) gate workload: h, k, v, dout [T, d]; w_h, w_k [d] fp32.

    Activations are N(0, 1), the two RMSNorm weights N(1, 0.1).  bf16 tensors are
    returned as raw uint16 bits (round-to-nearest-even of the fp64 draw).
    """
    n = w.T * w.d
    out = {}
    for i, name in enumerate(("h", "k", "v", "dout")):
        x = G.normal(w.seed + 1000 * (i + 1), n).reshape(w.T, w.d)
        out[name] = x.astype(np.float32) if w.dtype == "f32" else G.to_bf16_bits(x)
    out["w_h"] = G.normal(w.seed + 7001, w.d, 1.0, 0.1).astype(np.float32)
    out["w_k"] = G.normal(w.seed + 7002, w.d, 1.0, 0.1).astype(np.float32)
    return out


@dataclass
class GateHcWorkload:
    """The multi-branch gate: hc branches per token sharing one value row."""

    name: str
    T: int
    hc: int
    d: int
    dtype: str
    seed: int
    eps: float = 1e-6
    clamp: float = 1e-6


def gate_hc_host_inputs(w: GateHcWorkload):
    """x [T, hc, d], kv [T, hc+1, d], dout [T, hc, d] ~ N(0, 1); w_h, w_k [hc, d] ~ N(1, 0.1) fp32."""
    out = {}
    shapes = {"x": (w.T, w.hc, w.d), "kv": (w.T, w.hc + 1, w.d), "dout": (w.T, w.hc, w.d)}
    for i, (name, shp) in enumerate(shapes.items()):
        n = shp[0] * shp[1] * shp[2]
        x = G.normal(w.seed + 3000 * (i + 1), n).reshape(shp)
        out[name] = x.astype(np.float32) if w.dtype == "f32" else G.to_bf16_bits(x)
    out["w_h"] = G.normal(w.seed + 9001, w.hc * w.d, 1.0, 0.1).astype(np.float32).reshape(w.hc, w.d)
    out["w_k"] = G.normal(w.seed + 9002, w.hc * w.d, 1.0, 0.1).astype(np.float32).reshape(w.hc, w.d)
    return out


def gate_hc_4x4k(seed: int = 6) -> GateHcWorkload:
    """The production shape: 4 branches, T = 8192 tokens, d = 4096, bf16."""
    return GateHcWorkload(name="gate_hc4_T8192_d4096", T=8192, hc=4, d=4096, dtype="bf16", seed=seed * 101 + 13)


@dataclass
class SinkhornWorkload:
    """The Engram Sinkhorn's inputs: a gradient and momentum of one [rows, head_dim] matrix."""

    name: str
    rows: int
    head_dim: int
    grad_dtype: str  # "f32" | "bf16"
    seed: int
    eps: float = 1e-6
    beta1: float = 0.9
    nesterov: bool = True


def sinkhorn_host_inputs(w: SinkhornWorkload):
    """grad [rows, head_dim] ~ N(0, 1) (fp32 or bf16 bits), momentum ~ N(0, 0.5) fp32, and
    positive row / column scales ~ U(0.5, 2) fp32 (an iteration in progress)."""
    n = w.rows * w.head_dim
    g = G.normal(w.seed + 11, n).reshape(w.rows, w.head_dim)
    return {
        "grad": g.astype(np.float32) if w.grad_dtype == "f32" else G.to_bf16_bits(g),
        "momentum": G.normal(w.seed + 12, n, 0.0, 0.5).astype(np.float32).reshape(w.rows, w.head_dim),
        "row_scale": (0.5 + 1.5 * G.uniform01(w.seed + 13, w.rows)).astype(np.float32),
        "col_scale": (0.5 + 1.5 * G.uniform01(w.seed + 14, w.head_dim)).astype(np.float32),
    }


def sinkhorn_16k_x_5120(seed: int = 7) -> SinkhornWorkload:
    """16384 rows of head_dim 5120 (the largest head_dim the release's tests use): 335 MB fp32."""
    return SinkhornWorkload(name="sinkhorn_R16384_D5120", rows=16384, head_dim=5120, grad_dtype="bf16",
                            seed=seed * 101 + 17)


@dataclass
class ShortConvWorkload:
    """The short convolution after the gate over packed sequences."""

    name: str
    lengths: list
    d: int
    width: int
    dilation: int
    dtype: str
    seed: int
    eps: float = 1e-6
    bias: bool = True
    with_h: bool = True

    @property
    def T(self) -> int:
        return int(sum(self.lengths))


def short_conv_host_inputs(w: ShortConvWorkload):
    """V~ = alpha * N(0, 1) with a per-token gate alpha ~ U(0, 1) (the gate's output), H and dout ~ N(0, 1);
    norm_w ~ N(1, 0.1), conv_w [d, width] ~ N(0, 0.5), bias ~ N(0, 0.1) fp32; seq_offsets int64."""
    T, d = w.T, w.d
    alpha = G.uniform01(w.seed + 20, T)[:, None]
    conv = (lambda a: a.astype(np.float32)) if w.dtype == "f32" else G.to_bf16_bits
    out = {"v": conv(alpha * G.normal(w.seed + 21, T * d).reshape(T, d)),
           "h": conv(G.normal(w.seed + 22, T * d).reshape(T, d)) if w.with_h else None,
           "dout": conv(G.normal(w.seed + 23, T * d).reshape(T, d)),
           "norm_w": G.normal(w.seed + 24, d, 1.0, 0.1).astype(np.float32),
           "conv_w": G.normal(w.seed + 25, d * w.width, 0.0, 0.5).astype(np.float32).reshape(d, w.width),
           "bias": G.normal(w.seed + 26, d, 0.0, 0.1).astype(np.float32) if w.bias else None,
           "seq_offsets": G.offsets_from_lengths(w.lengths)}
    return out


def short_conv_4x4k(seed: int = 8) -> ShortConvWorkload:
    """After the gate's micro-batch: 4 sequences x 4096 tokens, d = 4096 bf16, width 4, dilation 3
    (the largest N-gram order of the hash workload)."""
    return ShortConvWorkload(name="short_conv_4x4096_d4096", lengths=[4096] * 4, d=4096, width=4, dilation=3,
                             dtype="bf16", seed=seed * 101 + 19)
