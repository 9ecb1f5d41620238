"""The multi-GPU path of bench.py is N independent replicas (requests are independent; there is
no exchange step).  Its host logic -- the slowest rank's time, the whole-job rate, rank 0 alone
printing the reference arm -- runs here on CPU as world-size-2 gloo process groups."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms_max = bench.max_over_ranks(times[rank])
        rate = bench.whole_job_rate(1280, world, 10, ms_max)
        dist.barrier()
        out.put((rank, ms_max, rate))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time():
    world, times = 2, [0.75, 1.25]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, rate in res:
        assert ms_max == max(times)
        # every rank's rows over the slowest rank's time
        assert rate == pytest.approx(1280 * world * 10 / (max(times) / 1e3))


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(100, 1, 4, 2.0) == pytest.approx(200_000.0)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the other ranks of the reference arm exit without work or output."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        workload, steps, warmup, gpus, scheme = "tiny", 1, 3, 2, "accept"
    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    """Rank 0 of the reference arm prints one JSON line: the oracle timed on the host cores, on
    the same metric and workload as the CUDA arm, with its sample and a zero-copy e2e."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "0")

    class Args:
        workload, steps, warmup, gpus, scheme = "tiny", 2, 3, 1, "accept"
    bench.run_reference(Args(), budget_s=2.0)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "rows/s"
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] >= 1 and "requests" in d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("tiny")
