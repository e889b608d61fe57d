"""bench.py's multi-rank host logic on CPU: two gloo ranks, each with its own
time and work, reduce to the slowest rank's time and the summed work (the
replicas run on the GPU machine use the same function over NCCL)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, work = bench.aggregate_ranks(10.0 + rank * 5.0, 100.0 * (rank + 1), dist, "cpu")
        out.put((rank, ms, work))
    finally:
        dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, work in res:
        assert ms == pytest.approx(15.0)     # slowest rank
        assert work == pytest.approx(300.0)  # all ranks' work


def test_aggregate_single_process_is_identity():
    assert bench.aggregate_ranks(3.5, 7.0) == (3.5, 7.0)


def test_bench_workloads_resolve_on_cpu():
    # every workload the default bench run names resolves to a layer the prefill and decode entry points
    # accept (shapes multiples of 128; a lever's formats present), and has its data description
    import synth
    for name in bench.PREFILL_EXTRA:
        cfg = bench.prefill_config(name)
        assert cfg.name == name and cfg.batches[0] == 4096
        assert cfg.H % 128 == 0 and cfg.I % 128 == 0 and (not cfg.shared_fmt or cfg.shared_I % 128 == 0)
    assert bench.prefill_config("prefill_int4g128").fmt == synth.configs.FMT_INT4_G128
    assert bench.prefill_config("prefill_fp8").fmt == synth.configs.FMT_FP8_B128
    for name in bench.MORE_PREFILL.split(","):
        assert name in bench.PREFILL_EXTRA, name
    for name in ("decode_nvfp4", "decode_mxfp4", "decode_int4"):
        assert name in bench.DATA_DESC
