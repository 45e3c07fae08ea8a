"""The benchmark's multi-rank host logic on CPU: two gloo ranks agree on the
slowest rank's time, and the whole-job figure counts every rank's work.  The
reference arm does its work on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        out.put((rank, mx))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == {0: 15.0, 1: 15.0}


def test_job_tflops_counts_every_rank():
    one = bench.job_tflops(2.0 ** 40, 10, 0.012, 1)
    assert one == pytest.approx(2.0 ** 40 * 10 / 0.012 / 1e12)
    assert bench.job_tflops(2.0 ** 40, 10, 0.012, 4) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")

    class Args:
        batch, steps, warmup, gpus = None, 1, 1, 2

    assert bench.reference_arm(Args()) == 0


def test_sdpa_context_never_raises():
    """The torch SDPA context figure is optional: without a GPU (or for
    grouped kv heads) it reports why instead of failing the benchmark line."""
    import torch
    from softmax_free_attention_gb300 import workloads
    w = workloads.Workload("ctx", B=1, h=2, hkv=2, Tq=16, Tk=16, dk=32, dv=32, dtype="bf16",
                           causal=True, qk_factor=1.0, yat_param="ln2", seed=0)
    q = torch.zeros(1, 2, 16, 32, dtype=torch.bfloat16)
    res = bench.sdpa_context(q, q, q, w, w.flops(), 2)
    if not torch.cuda.is_available():
        assert "unavailable" in res
    wg = workloads.Workload("ctx_gqa", B=1, h=2, hkv=1, Tq=16, Tk=16, dk=32, dv=32, dtype="bf16",
                            causal=True, qk_factor=1.0, yat_param="ln2", seed=0)
    assert bench.sdpa_context(q, q[:, :1], q[:, :1], wg, wg.flops(), 2) == {
        "unavailable": "grouped kv heads"}


def test_recorded_traffic_follows_the_sources_and_the_batch():
    """The roofline's DRAM traffic comes from the committed ncu summary only
    while its source hash matches the kernel sources, and scales with the
    batch (every tensor of the workload does)."""
    full = bench.recorded_traffic()
    if full is None:
        pytest.skip("the committed summary was captured on other kernel sources")
    from softmax_free_attention_gb300 import workloads
    B = workloads.WORKLOADS[bench.WORKLOAD].B
    assert bench.recorded_traffic(B) == full
    assert abs(bench.recorded_traffic(B // 4) - full / 4) <= 1e-6 * full
    # algorithmic bytes of the full launch: q, k, v read and out written once
    w = workloads.WORKLOADS[bench.WORKLOAD]
    algo = 2 * (w.B * w.h * w.Tq * (w.dk + w.dv) + w.B * w.hkv * w.Tk * (w.dk + w.dv))
    assert 0.8 * algo < full < 1.2 * algo
