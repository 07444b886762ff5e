"""Host-side logic of bench.py on CPU: the replicas-only rank reduction over two gloo ranks,
and the reference arm (the CPU oracle) on the small one-request workload."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took 10 + r ms and scored 1000 * (r + 1) slots
    ms, slots = bench.reduce_over_ranks(10.0 + rank, 1000 * (rank + 1), dist, "cpu")
    out[rank] = (ms, slots)
    dist.destroy_process_group()


def test_reduce_over_ranks_gloo_two_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    # every rank sees the slowest rank's time and the slots of all ranks
    assert res[0] == res[1] == (11.0, 3000)


def test_reduce_over_ranks_single_process():
    import bench
    assert bench.reduce_over_ranks(7.5, 123, None, "cpu") == (7.5, 123)


def _run_bench(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_contract_line(oracle_mod):
    r = _run_bench(["--impl", "reference", "--config", "pr1", "--steps", "2", "--warmup", "1"], {})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["steps"] == 2 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("pr1: 1 req x 1 layers")


def test_reference_arm_other_ranks_exit_quietly(oracle_mod):
    r = _run_bench(["--impl", "reference", "--config", "pr1", "--steps", "1", "--warmup", "1"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_pure_dense_runs_only_score_and_topk(monkeypatch):
    """The pure-dense variant re-runs each step's score and top-K launches for every layer
    (warm-up steps first, hints reset), nothing else; a failure lands in its JSON entry."""
    import bench

    class Event:
        def __init__(self, enable_timing=False):
            pass

        def record(self):
            pass

        def elapsed_time(self, other):
            return 12.0

    monkeypatch.setattr(torch.cuda, "Event", Event)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda: None)

    class Hint:
        resets = 0

        def reset(self):
            Hint.resets += 1

    class FakeWorkload:
        L = 2
        q = [["q0a", "q0b"], ["q1a", "q1b"]]
        w = [["w0a", "w0b"], ["w1a", "w1b"]]

        def __init__(self):
            self.hints = [Hint(), Hint()]
            self.calls = []

        def score_topk(self, s, layer, q, w, ev=None):
            self.calls.append((s, layer, q, w))

    wk = FakeWorkload()
    assert bench.time_pure_dense(wk, 3, 4) == 3.0          # 12 ms over the 4 timed steps
    assert Hint.resets == 2
    assert [c[:2] for c in wk.calls] == [(s, l) for s in range(7) for l in range(2)]
    assert wk.calls[3] == (1, 1, "q1b", "w1b")
    assert bench.pure_dense_entry(wk, 3, 4, 1.5) == {"ms_per_step": 3.0, "latency_ratio": 0.5}

    class Failing(FakeWorkload):
        def score_topk(self, *a, **k):
            raise RuntimeError("launch failed")

    assert "launch failed" in bench.pure_dense_entry(Failing(), 3, 4, 1.5)["error"]
