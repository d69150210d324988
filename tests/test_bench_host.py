"""Host-side logic of bench.py on CPU: the multi-rank path (2 gloo ranks, replicas only), the
reference arm's rank handling, and the algorithmic byte counts the roofline divides by."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 100.0 + 25.0 * rank  # rank 1 is the slow one
        slowest = bench.aggregate_max(elapsed)
        bench.barrier()
        q.put((rank, slowest, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [125.0, 125.0]
    assert got[0][2] == (0, 0, 2) and got[1][2] == (1, 1, 2)


def test_reference_arm_other_ranks_exit_quietly(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                                      "--warmup", "3"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main() == 0
    assert buf.getvalue() == ""


def test_algorithmic_bytes_per_unit():
    ab = bench.algorithmic_bytes(P=1024)
    T_all, d = bench.SEQS * bench.SEQ_LEN, bench.D
    assert ab["hash_gather"] == T_all * 4104          # 4 + 4 + 16 rows x 128 B read + written
    assert ab["gate_fwd"] == bench.MICRO_T * 32784    # 8d + 16 at d = 4096
    assert ab["gate_bwd"] == bench.MICRO_T * 57360 + 1024 * d * 4  # 14d + 16, plus the partial rows
    assert ab["gate_bwd_accumulate"] == ab["gate_bwd"] + 1024 * d * 4  # the partial rows read back too
    assert ab["gate_fwd_fold"] == ab["gate_fwd"] + 3 * 4 * d          # w_h, w_k read, the fold written
    assert ab["grad_w_reduce"] == 1024 * d * 4 + 7 * d * 4           # one array of accumulated partials


def test_oracle_step_runs_a_whole_step_on_a_small_workload():
    """The oracle step both oracle timings run (the reference arm and cpu_baseline): hash + gather of
    every token, the fold, gate fwd + bwd of every micro-batch, the ordered reduction -- here on the
    tiny workloads, with more than one call per micro-batch and per hash range."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    from synth import workloads as W

    hw = W.tiny_hash()
    g = [W.gate_host_inputs(W.GateWorkload(name=f"mb{i}", T=600, d=64, dtype="bf16", seed=40 + i)) for i in range(2)]
    mbs = [{n: x[n] for n in ("h", "k", "v", "dout")} for x in g]
    table = hw.table_host.view(np.uint32).astype(np.uint16)  # any 16-bit table of the right shape
    with ThreadPoolExecutor(3) as pool:
        t = bench.oracle_step(pool, 3, hw, np.ascontiguousarray(table), mbs, g[0]["w_h"], g[0]["w_k"])
    assert t > 0
    times, threads = bench.time_oracle_steps(hw, np.ascontiguousarray(table), mbs, g[0]["w_h"], g[0]["w_k"], 2, 1)
    assert len(times) == 2 and all(x > 0 for x in times) and threads >= 1


def test_oracle_rates_per_config_on_one_core_and_on_all():
    """The per-config oracle rates (one core, then every core) on the tiny workloads: the gate forward
    alone, the forward + backward + reduction, and the hash + gather."""
    import numpy as np

    from synth import workloads as W

    x = W.gate_host_inputs(W.GateWorkload(name="r", T=700, d=64, dtype="bf16", seed=61))
    for fwd_only in (True, False):
        r = bench.oracle_gate_rates(x, fwd_only, T_config=700 if fwd_only else 70000)
        assert r["single_core"]["cores"] == 1 and r["single_core"]["tokens_per_s"] > 0
        assert r["all_cores"]["cores"] >= 1 and r["all_cores"]["tokens_per_s"] > 0
        assert ("all 700 tokens" in r["sample"]) == fwd_only and ("first 700 of the 70000" in r["sample"]) != fwd_only
    hw = W.tiny_hash()
    table = np.ascontiguousarray(hw.table_host.view(np.uint32).astype(np.uint16))
    r = bench.oracle_hash_rates(hw, table)
    assert r["single_core"]["tokens_per_s"] > 0 and r["all_cores"]["tokens_per_s"] > 0
    assert f"all {hw.T} tokens" in r["sample"]
