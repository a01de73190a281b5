"""Host logic of bench.py (no GPU): the whole-job throughput and the
max-over-ranks timing with two gloo ranks on CPU, and the busbw arithmetic
against the worked examples of "All-Reduce, in depth"."""

import os
import socket

import pytest

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [12.5, 20.0][rank]
    m = bench.max_over_ranks(local_ms, world)
    v = bench.whole_job_gbps(1e9, 10, world, m)
    q.put((rank, m, v))
    dist.destroy_process_group()


def test_two_rank_timing_takes_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in out:
        assert m == 20.0
        assert v == pytest.approx(2 * 10 * 1e9 / 0.020 / 1e9)


def test_single_rank_passthrough():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_gbps(2e9, 5, 1, 1000.0) == pytest.approx(10.0)


def test_busbw_matches_worked_examples(golden):
    for c in golden("busbw_examples.json")["cases"]:
        # time = 2 (N-1)/N x S / busbw  <=>  busbw(S, time, N) = busbw
        t = 2 * (c["N"] - 1) / c["N"] * c["S_bytes"] / c["busbw_Bps"]
        assert t == pytest.approx(c["time_s_about"], rel=c["rel_tol"])
        assert bench.busbw_gbps(c["S_bytes"], t, c["N"]) == pytest.approx(c["busbw_Bps"] / 1e9)


def test_phase_option_reaches_the_oracle_and_the_workload_name():
    """`--phase` runs one half: the oracle gets the same phase (and the
    schedule's own parameters), the workload name says which half."""
    import sys
    argv = sys.argv
    try:
        sys.argv = ["bench.py", "--phase", "reduce_scatter", "--algo", "generalized", "--r", "0"]
        a = bench.parse()
    finally:
        sys.argv = argv
    assert bench.oracle_kw(a) == {"r": 0, "phase": "reduce_scatter"}
    assert bench.workload_name(a).endswith("r=0, phase=reduce_scatter")
    sys.argv = ["bench.py"]
    try:
        a = bench.parse()
    finally:
        sys.argv = argv
    assert a.phase == "allreduce" and bench.oracle_kw(a) == {}
    assert "phase" not in bench.workload_name(a)


def test_bulk_kernel_name_follows_the_plan_kernel_bits():
    """The bench line names the kernel that runs a plan's aligned bulk items
    from ar_plan_info.kernels: the launch-set kernels before the staged ones,
    the element-wise kernel only when nothing else runs."""
    import bench
    import collective_reduction_gb300 as ar
    assert bench.bulk_kernel_name(ar.KERNEL_FEW) == "few_kernel"
    assert bench.bulk_kernel_name(ar.KERNEL_FEW | ar.KERNEL_ELEMENTWISE) == "few_kernel"
    assert bench.bulk_kernel_name(ar.KERNEL_STREAM) == "stream_kernel"
    assert bench.bulk_kernel_name(ar.KERNEL_COPY) == "copy_kernel"
    assert bench.bulk_kernel_name(ar.KERNEL_WORD_JIT | ar.KERNEL_ELEMENTWISE) == "ar_word_kernel"
    assert bench.bulk_kernel_name(ar.KERNEL_STAGED | ar.KERNEL_DAG_JIT) == "ar_dag_kernel"
    assert bench.bulk_kernel_name(ar.KERNEL_STAGED) == "staged_kernel"
    assert bench.bulk_kernel_name(ar.KERNEL_CHAIN_WORD) == "chain_word_kernel"
    assert bench.bulk_kernel_name(ar.KERNEL_ELEMENTWISE) == "elementwise_kernel"
