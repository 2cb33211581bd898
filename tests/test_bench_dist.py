"""The replicas path of the benchmark on two gloo ranks (CPU): every rank's
times reduce to the slowest rank's (max over ranks), and the line's value is
all ranks' tokens over that time ("replicas only": sessions are independent,
so N GPUs each run their own replica with no collective on the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    import argparse

    import torch.distributed as dist

    import bench
    import synthetic
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 * (rank + 1), True)
        bench.barrier(True)
        s = synthetic.SHAPES["4b"]
        args = argparse.Namespace(steps=100, warmup=3, prompt=2048, sessions=32, gpus=world, impl="ours")
        # rank r is slower by a factor of r + 1
        res = {
            "shape": s, "decode_ms": 200.0 * (rank + 1), "decode_ctx": (2048, 2148),
            "decode_profile": {"decode_step": (220.0, 100), "gemv": (0.0, 0)},
            "decode_profile_ctx": (2148, 2248), "clocks": {}, "launches": 100,
            "prefill_ms": 16.0 * (rank + 1), "prefill_profile": {"gemm": (12.0, 144)},
            "e2e_s": 0.25 * (rank + 1), "e2e_bytes": (4, 607748),
        }
        pk = {"hbm_gbs": 6767.7, "bf16_tflops": 1929.6, "bf16_tflops_sustained": 1702.9}
        line = bench.report(args, res, world, True, pk, "measured")
        out.put((rank, got, line["value"], line["ms_per_step"], line["prefill"]["value"], line["e2e"]["value"]))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    rows = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for rank, got, value, ms, pre, e2e in rows:
        assert got == 20.0                                   # max over ranks
        assert ms == pytest.approx(400.0 / 100)              # the slowest rank's step time
        assert value == pytest.approx(2 * 100 / 0.400)       # both ranks' tokens / slowest time
        assert pre == pytest.approx(2 * 2048 / 0.032)
        assert e2e == pytest.approx(2 * 100 / 0.5)
