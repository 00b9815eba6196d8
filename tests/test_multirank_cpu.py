"""The N > 1 host logic of bench.py on CPU: two gloo ranks (replicas, no
data-path collective) reduce their step times to the maximum, the whole-job
value counts every replica's rows, and only rank 0 runs the reference arm."""

import importlib.util
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist

    bench = _bench()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    per_rank = [[0.040, 0.031, 0.060], [0.045, 0.029, 0.058]][rank]
    red = bench.max_over_ranks(per_rank, dist, torch.device("cpu"))
    out.put((rank, red, bench.job_value(world, 1 << 20, red[0])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect = [0.045, 0.031, 0.060]
    for rank, red, value in res:
        assert red == pytest.approx(expect)
        assert value == pytest.approx(2 * (1 << 20) / (0.045e-3))


def test_single_process_is_unchanged():
    bench = _bench()
    assert bench.max_over_ranks([1.0, 2.0], None, None) == [1.0, 2.0]
    assert bench.job_value(1, 1000, 2.0) == pytest.approx(1000 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    bench = _bench()
    called = []
    monkeypatch.setattr(bench, "run_oracle_subprocess", lambda *a, **k: called.append(a) or [1.0])
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup, gpus = 2, 3, 2

    bench.reference_arm(Args, "long", 1 << 20)
    assert called == [] and capsys.readouterr().out == ""


def test_replay_plan_times_exactly_k_steps():
    """The bench replays graphs of several steps: the group and one-step
    replays it plans add up to exactly the K steps it reports, for every K."""
    bench = _bench()
    for group in (1, 3, 8):
        for k in range(0, 100):
            n_group, n_single = bench.replay_plan(k, group)
            assert n_group * group + n_single == k
            assert 0 <= n_single < group
