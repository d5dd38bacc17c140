"""Host logic of bench.py with more than one process (gloo, two ranks, CPU).

The verify pass does not shard: with --gpus N every rank runs an independent
replica, the step time is the maximum over ranks and only rank 0 prints.  The
reference arm (the CPU oracle) runs on rank 0 alone; the other ranks exit 0
without work.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = bench.dist_env()
        step_ms = bench.max_over_ranks(1.0 + rank, world)  # rank r took 1 + r ms
        bench.barrier(world)

        # the reference arm with a stub oracle step (the real one takes seconds)
        calls = []

        def fake_step(cfg, k, seed=0, layer=0, weights=None):
            calls.append(k)
            return 0.25, "weights"

        bench.oracle_layer_step = fake_step
        import oracle.oracle as O
        O.build = lambda: None

        class Args:
            k, steps, warmup, gpus = 9, 3, 1, world

        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = bench.run_reference(Args(), dict(layers=12))
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(dict(env=list(env), step_ms=step_ms, rc=rc, out=buf.getvalue(), calls=len(calls)), f)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_replicas_take_max_time_and_only_rank0_reports(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, x in enumerate(res):
        assert x["env"] == [r, world, r]
        assert x["step_ms"] == pytest.approx(2.0)  # max over ranks, seen by every rank
        assert x["rc"] == 0
    # rank 0: one JSON line for the reference arm; rank 1: no output, no oracle work
    lines = [l for l in res[0]["out"].splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["value"] == pytest.approx(9 / 0.25)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert res[0]["calls"] == 1 + 1 + 3  # weights draw, warm-up, timed steps
    assert res[1]["out"] == "" and res[1]["calls"] == 0
