"""The seeded input generators: reproducible, and shaped like the workloads they stand in for."""
import numpy as np

from synth import generators as G
from synth import workloads as W


def test_splitmix64_vector_matches_scalar_definition():
    v = G.splitmix64(0x1234, 8)
    assert [int(x) for x in v] == [G.splitmix64_scalar(0x1234, i) for i in range(1, 9)]
    # first output of the stream seeded with 0 (Steele-Lea-Flood reference value)
    assert G.splitmix64_scalar(0, 1) == 0xE220A8397B1DCDAF


def test_generators_are_deterministic():
    assert np.array_equal(G.normal(5, 100), G.normal(5, 100))
    assert not np.array_equal(G.normal(5, 100), G.normal(6, 100))
    x = G.normal(7, 200_000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], dtype=np.float64)
    bits = G.to_bf16_bits(vals)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert back.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 0.0]


def test_surjection_is_onto():
    m = G.surjection(3, 1000, 770)
    assert m.min() == 0 and m.max() == 769 and len(np.unique(m)) == 770


def test_primes_and_multipliers():
    p = G.consecutive_primes(1009, 4)
    assert p.tolist() == [1009, 1013, 1019, 1021]
    assert G.consecutive_primes(2_000_003, 16)[-1] == 2_000_249
    m = G.odd_multipliers(9, 16, 3)
    assert m.shape == (16, 3) and (m & np.uint64(1)).all()


def test_workload_shapes():
    w = W.hash_gather_64k()
    assert w.T == 65536 and w.spec.tables == 16 and w.seq_offsets[-1] == 65536
    assert 0 <= w.token_ids.min() and w.token_ids.max() < 128000
    # 16 tables of ~2.0M rows x 64 bf16 = 4.10 GB
    assert abs(w.spec.total_rows * 64 * 2 / 1e9 - 4.096) < 0.01
    r = W.gate_ragged_7k()
    assert len(r.seq_lengths) == 64 and r.seq_lengths.min() >= 256 and r.seq_lengths.max() <= 4096
