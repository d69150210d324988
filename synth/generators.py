"""Seeded synthetic input generators shared by the oracle checks, the GPU tests and the bench.

This module holds no arithmetic of the Engram method itself: it only draws the
inputs (token ids, sequence lengths, the vocabulary surjection, table sizes,
hash multipliers, dense activations) that both the CPU oracle and the CUDA path
consume.  Everything is a pure function of an explicit seed.

Generators used (all published, restated here):

* SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): state_i = seed + i * 0x9E3779B97F4A7C15 (i >= 1),
  output = mix(state_i) with the Stafford "variant 13" finaliser.
* Uniform doubles in [0, 1): the top 53 bits of a SplitMix64 output times 2^-53.
* Normals: Box-Muller on pairs of 53-bit uniforms.
* Zipf(s) over ranks 1..V: inverse CDF by binary search on the fp64 cumulative
  weights r^-s; rank r maps to id r-1.
* Random permutation: argsort of SplitMix64 keys (ties have probability ~2^-64).
"""
from __future__ import annotations

import numpy as np

_GAMMA = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB
_U64 = (1 << 64) - 1


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset+1 .. offset+n of the SplitMix64 stream started at `seed`, as uint64."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = np.uint64(seed & _U64) + i * np.uint64(_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_MIX2)
        return z ^ (z >> np.uint64(31))


def splitmix64_scalar(seed: int, i: int) -> int:
    """Output number i (1-based) of the stream, in Python integers (used to cross-check the vector form)."""
    z = (seed + i * _GAMMA) & _U64
    z = ((z ^ (z >> 30)) * _MIX1) & _U64
    z = ((z ^ (z >> 27)) * _MIX2) & _U64
    return z ^ (z >> 31)


def uniform01(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n doubles in [0, 1) with 53 random bits each."""
    return (splitmix64(seed, n, offset) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """n normal draws by Box-Muller (fp64)."""
    m = (n + 1) // 2
    u = uniform01(seed, 2 * m)
    u1 = 1.0 - u[0::2]  # in (0, 1]: log is finite
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return mean + std * z[:n]


def uniform_int(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi) (int64)."""
    return lo + np.floor(uniform01(seed, n) * (hi - lo)).astype(np.int64)


def zipf_ids(seed: int, n: int, vocab: int, s: float) -> np.ndarray:
    """n ids in [0, vocab) with P(id = r-1) proportional to r^-s."""
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    u = uniform01(seed, n)
    idx = np.searchsorted(cdf, u, side="right")
    return np.minimum(idx, vocab - 1).astype(np.int64)


def permutation(seed: int, n: int) -> np.ndarray:
    """A uniformly random permutation of 0..n-1."""
    return np.argsort(splitmix64(seed, n), kind="stable").astype(np.int64)


def surjection(seed: int, vocab: int, vocab_c: int) -> np.ndarray:
    """A random onto map [0, vocab) -> [0, vocab_c), as int32.

    A random permutation picks vocab_c ids that map one-to-one onto 0..vocab_c-1
    (so the map is onto); every other id maps to a uniform target.  This stands
    in for the tokenizer compression P: V -> V', which folds surface variants of
    a token onto one canonical id.
    """
    if not 0 < vocab_c <= vocab:
        raise ValueError("need 0 < vocab_c <= vocab")
    perm = permutation(seed, vocab)
    out = np.empty(vocab, dtype=np.int64)
    out[perm[:vocab_c]] = np.arange(vocab_c)
    rest = vocab - vocab_c
    if rest:
        out[perm[vocab_c:]] = uniform_int(seed ^ 0x5DEECE66D, rest, 0, vocab_c)
    return out.astype(np.int32)


def _is_prime(n: int) -> bool:
    if n < 2:
        return False
    if n % 2 == 0:
        return n == 2
    f = 3
    while f * f <= n:
        if n % f == 0:
            return False
        f += 2
    return True


def consecutive_primes(anchor: int, count: int) -> np.ndarray:
    """The `count` smallest primes >= anchor (trial division), as uint64."""
    out = []
    n = anchor
    while len(out) < count:
        if _is_prime(n):
            out.append(n)
        n += 1
    return np.array(out, dtype=np.uint64)


def odd_multipliers(seed: int, tables: int, max_order: int) -> np.ndarray:
    """[tables, max_order] uint64 hash multipliers: SplitMix64 draws in (table, j) order, OR 1."""
    return (splitmix64(seed, tables * max_order) | np.uint64(1)).reshape(tables, max_order)


def ragged_lengths(seed: int, count: int, lo: int, hi: int) -> np.ndarray:
    """`count` sequence lengths uniform in [lo, hi] inclusive (int64)."""
    return uniform_int(seed, count, lo, hi + 1)


def offsets_from_lengths(lengths) -> np.ndarray:
    """cu_seqlens-style boundaries [0, l0, l0+l1, ...] (int64)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    out[1:] = np.cumsum(lengths)
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64/fp32 values to bfloat16 (round to nearest even) and return the raw uint16 bits.

    Used only to store synthetic inputs in bf16; both sides then read the same bits.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    nan = np.isnan(f)
    r = r.astype(np.uint16)
    r[nan] = 0x7FC0
    return r
