"""GPU parity of the hash + gather path against the CPU oracle: bit-exact indices and rows.

Sizes: the tiny workload, the full 16 x 4096-token / 16-table / 4.1 GB workload
(every token's indices and rows), and edge cases -- empty and one-token
sequences, empty batches, tails that are not a multiple of the tile, the
largest table count and N-gram order, several row widths and both dtypes, the
identity compression map -- plus the device-side reporting of malformed inputs.
"""
import numpy as np
import pytest
import torch

import engram_conditional_memory_gb300 as ecm
import oracle
from synth import device as SD
from synth import generators as G
from synth import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _status_clean(cuda_lib):
    ecm.device_status(clear=True)
    yield


def _run(w, table, want_rows=True, want_indices=True, err=None):
    s = w.spec
    spec = ecm.HashSpec(s.min_order, s.num_orders, s.heads, s.multipliers, s.primes)
    cmap = None if w.compress_map is None else torch.from_numpy(w.compress_map).to(DEV)
    return ecm.hash_gather(spec, torch.from_numpy(w.token_ids).to(DEV), torch.from_numpy(w.seq_offsets).to(DEV),
                           table, cmap, w.vocab, w.vocab_c, want_rows=want_rows, want_indices=want_indices,
                           err_word=err)


def _oracle_idx(w):
    s = w.spec
    return oracle.hash_indices(w.token_ids, w.seq_offsets, w.compress_map, w.vocab, s.min_order, s.num_orders,
                               s.heads, s.multipliers, s.primes)


def _bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint16) if a.dtype.itemsize == 2 else a.view(np.uint32)


def _host_table(table: torch.Tensor) -> np.ndarray:
    if table.dtype == torch.bfloat16:
        return table.cpu().view(torch.int16).numpy().view(np.uint16)
    return table.cpu().numpy()


def _check(w, table, rows, idx):
    ref_idx = _oracle_idx(w)
    assert np.array_equal(idx.cpu().numpy().astype(np.int64), ref_idx)
    ref_rows = oracle.gather_rows(_host_table(table), w.spec.primes, ref_idx).reshape(w.T, -1)
    got = _host_table(rows)
    assert np.array_equal(_bits(got), _bits(ref_rows))


def test_tiny_workload_bit_exact():
    w = W.tiny_hash()
    table = SD.hash_table(w, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    rows, idx = _run(w, table, err=err)
    assert ecm.read_error_word(err) == 0
    _check(w, table, rows, idx)


def test_full_size_workload_bit_exact():
    w = W.hash_gather_64k()
    table = SD.hash_table(w, DEV)  # 4.1 GB, bf16 N(0, 0.02)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    rows, idx = _run(w, table, err=err)
    assert ecm.read_error_word(err) == 0
    ref_idx = _oracle_idx(w)
    assert np.array_equal(idx.cpu().numpy().astype(np.int64), ref_idx)
    # every gathered row against the oracle's gather from a host copy of the whole table
    host = torch.empty(table.shape, dtype=table.dtype, pin_memory=True)
    host.copy_(table)
    ref_rows = oracle.gather_rows(host.view(torch.int16).numpy().view(np.uint16), w.spec.primes, ref_idx)
    got = rows.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref_rows.reshape(w.T, -1))
    # indices-only and rows-only calls agree with the combined call
    rows2, none = _run(w, table, want_indices=False)
    assert none is None and torch.equal(rows2, rows)
    none, idx2 = _run(w, table, want_rows=False)
    assert none is None and torch.equal(idx2, idx)


def _custom(ids, lengths, min_order, num_orders, heads, row_dim, dtype, cmap=None, vocab=None, seed=0,
            anchor=1009):
    ids = np.asarray(ids, dtype=np.int32)
    spec = W.hash_spec(seed + 77, min_order, num_orders, heads, anchor)
    vocab = vocab or int(ids.max(initial=0)) + 1
    vocab_c = vocab if cmap is None else int(cmap.max()) + 1
    table = None
    if dtype == "f32":
        table = G.normal(seed + 5, spec.total_rows * row_dim, 0, 0.02).astype(np.float32).reshape(-1, row_dim)
    w = W.HashGatherWorkload(name="custom", token_ids=ids, seq_offsets=G.offsets_from_lengths(lengths),
                             compress_map=cmap, vocab=vocab, vocab_c=vocab_c, spec=spec, row_dim=row_dim,
                             dtype=dtype, table_seed=seed + 5, table_host=table)
    return w


@pytest.mark.parametrize("lengths", [[1], [2], [3], [31, 1, 0, 33], [32, 32], [0, 5, 0], [100, 1, 1, 1, 60],
                                     [17] * 9, [1000, 23]])
def test_ragged_sequences_and_tails(lengths):
    T = int(sum(lengths))
    ids = G.uniform_int(T + 3, T, 0, 500)
    cmap = G.surjection(4, 500, 321)
    w = _custom(ids, lengths, 2, 2, 3, 64, "bf16", cmap=cmap, vocab=500, seed=T)
    table = SD.hash_table(w, DEV)
    rows, idx = _run(w, table)
    _check(w, table, rows, idx)


@pytest.mark.parametrize("min_order,num_orders,heads,row_dim,dtype", [
    (1, 8, 4, 8, "bf16"),      # 32 tables, orders 1..8, 16-byte rows
    (2, 2, 8, 64, "bf16"),     # the method's shape
    (2, 2, 2, 16, "f32"),
    (3, 1, 1, 100, "f32"),     # one table, 400-byte rows
    (2, 3, 5, 24, "bf16"),     # 15 tables, 48-byte rows
    (2, 1, 32, 1024, "bf16"),  # the largest e_t row, 32 x 2 KB = 64 KB: one token per tile
])
def test_table_shapes(min_order, num_orders, heads, row_dim, dtype):
    T = 777
    ids = G.uniform_int(row_dim + heads, T, 0, 3000)
    w = _custom(ids, [400, 377], min_order, num_orders, heads, row_dim, dtype, vocab=3000, seed=heads,
                anchor=5003)
    table = SD.hash_table(w, DEV)
    rows, idx = _run(w, table)
    _check(w, table, rows, idx)


def test_empty_batch():
    w = _custom([], [0], 2, 2, 2, 64, "bf16", vocab=10)
    table = SD.hash_table(w, DEV)
    rows, idx = _run(w, table)
    assert rows.shape == (0, 4 * 64) and idx.shape == (0, 4)


def test_malformed_inputs_are_reported_not_read():
    w = W.tiny_hash()
    table = SD.hash_table(w, DEV)
    # a raw id outside the vocabulary
    bad = w.token_ids.copy()
    bad[5] = w.vocab + 3
    w_bad = W.HashGatherWorkload(**{**w.__dict__, "token_ids": bad})
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    rows, idx = _run(w_bad, table, err=err)
    assert ecm.read_error_word(err) & ecm.DEVERR_TOKEN_ID
    # tokens whose windows do not reach the bad id are unaffected
    ref = _oracle_idx(w)
    got = idx.cpu().numpy()
    assert np.array_equal(got[:5], ref[:5]) and np.array_equal(got[8:], ref[8:])
    # a compression map value outside [0, vocab_c)
    cmap = w.compress_map.copy()
    cmap[w.token_ids[3]] = w.vocab_c + 10
    w_cm = W.HashGatherWorkload(**{**w.__dict__, "compress_map": cmap})
    err.zero_()
    _run(w_cm, table, err=err)
    assert ecm.read_error_word(err) & ecm.DEVERR_COMPRESSED
    # sequence offsets that decrease
    w_so = W.HashGatherWorkload(**{**w.__dict__, "seq_offsets": np.array([0, 40, 20, 64], dtype=np.int64)})
    err.zero_()
    _run(w_so, table, err=err)
    assert ecm.read_error_word(err) & ecm.DEVERR_SEQ_OFFSETS
    assert ecm.device_status(clear=True) & (ecm.DEVERR_TOKEN_ID | ecm.DEVERR_COMPRESSED | ecm.DEVERR_SEQ_OFFSETS)


def test_indices_are_reproducible_across_grids():
    w = W.hash_gather_64k(num_seqs=4, seq_len=4096)
    spec = w.spec
    table = torch.zeros((spec.total_rows, 8), dtype=torch.bfloat16, device=DEV)  # rows irrelevant here
    w8 = W.HashGatherWorkload(**{**w.__dict__, "row_dim": 8})
    _, base = _run(w8, table, want_rows=False)
    try:
        for cap in (1, 3, 0):
            ecm.set_max_ctas(cap)
            _, idx = _run(w8, table, want_rows=False)
            assert torch.equal(idx, base)
    finally:
        ecm.set_max_ctas(0)


def test_many_sequences_offsets_in_global_memory():
    """More sequences than either kernel stages in shared memory (the gather above 511, the
    index-only kernel above 4095): the sequence-start search then reads the offsets from global
    memory.  5000 sequences of 0 to 7 tokens, rows and indices against the oracle."""
    lengths = [int(x) for x in G.uniform_int(4242, 5000, 0, 8)]
    T = sum(lengths)
    ids = G.uniform_int(4243, T, 0, 3000)
    w = _custom(ids, lengths, 2, 2, 8, 64, "bf16", vocab=3000, seed=13, anchor=5003)
    table = SD.hash_table(w, DEV)
    rows, idx = _run(w, table)
    _check(w, table, rows, idx)
    _, idx_only = _run(w, table, want_rows=False)
    assert torch.equal(idx_only, idx)
    assert ecm.device_status(clear=True) == 0


def test_rows_reproducible_across_grids():
    """One or three CTAs walk every tile, so the hash warp's ring of row-number slots wraps dozens of
    times ahead of the copies; rows and indices match the default grid bit for bit and the oracle."""
    lengths = [1500, 700, 1]
    T = sum(lengths)
    ids = G.uniform_int(91, T, 0, 3000)
    w = _custom(ids, lengths, 2, 2, 8, 64, "bf16", vocab=3000, seed=8, anchor=5003)  # 16 tables, 2 KB e_t rows
    table = SD.hash_table(w, DEV)
    base_rows, base_idx = _run(w, table)
    _check(w, table, base_rows, base_idx)
    try:
        for cap in (1, 3):
            ecm.set_max_ctas(cap)
            rows, idx = _run(w, table)
            assert torch.equal(idx, base_idx)
            assert torch.equal(rows.view(torch.int16), base_rows.view(torch.int16))
    finally:
        ecm.set_max_ctas(0)
    assert ecm.device_status(clear=True) == 0


# ----------------------------------------------------------------------------- tables in host memory

@pytest.mark.parametrize("lengths,row_dim,dtype", [([64], 16, "f32"), ([31, 1, 0, 100], 64, "bf16"),
                                                   ([4096] * 4, 64, "bf16")])
def test_host_resident_table_bit_exact(lengths, row_dim, dtype):
    T = int(sum(lengths))
    ids = G.uniform_int(T + 11, T, 0, 2000)
    cmap = G.surjection(8, 2000, 1500)
    w = _custom(ids, lengths, 2, 2, 8, row_dim, dtype, cmap=cmap, vocab=2000, seed=T + 1, anchor=20011)
    dev_table = SD.hash_table(w, DEV)
    host_table = dev_table.cpu().pin_memory()
    rows_h, idx_h = _run(w, host_table)
    rows_d, idx_d = _run(w, dev_table)
    assert torch.equal(idx_h, idx_d) and torch.equal(rows_h, rows_d)
    _check(w, dev_table, rows_h, idx_h)


def test_host_table_must_be_pinned():
    w = W.tiny_hash()
    table = torch.from_numpy(w.table_host.copy())  # pageable
    with pytest.raises(ValueError):
        _run(w, table)
    lib = ecm.load_library()
    from engram_conditional_memory_gb300.binding import _HashGatherArgs
    s = w.spec
    spec = ecm.HashSpec(s.min_order, s.num_orders, s.heads, s.multipliers, s.primes)
    ids = torch.from_numpy(w.token_ids).to(DEV)
    offs = torch.from_numpy(w.seq_offsets).to(DEV)
    out = torch.empty((w.T, 4 * 16), dtype=torch.float32, device=DEV)
    import ctypes
    args = _HashGatherArgs(ids.data_ptr(), w.T, offs.data_ptr(), 1, None, w.vocab, w.vocab, table.data_ptr(),
                           table.shape[0], 16, 0, None, out.data_ptr(), None)
    cspec = spec._c()
    assert lib.engram_hash_gather_host(ctypes.byref(cspec), ctypes.byref(args), None) == 7  # ENGRAM_ERR_DEVICE
