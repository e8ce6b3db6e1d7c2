"""Multi-rank host logic of bench.py on CPU (gloo, world size 2, no GPU).

The GPU arm runs on one GPU only: under more than one rank (or with --gpus other than 1)
it prints an "unavailable" line on rank 0 and exits before touching CUDA. The timing rule
for independent replicas (the job's time is the slowest rank's, its value N x steps / that
time) is host logic and is checked here with two gloo ranks; only rank 0 prints.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, lr, w = bench.dist_env()
    # rank k timed 1 + k seconds for its 100 steps
    total, value = bench.aggregate_over_ranks(1.0 + rank, 100, w)
    q.put((rank, r, lr, w, total, value))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29400 + os.getpid() % 500
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=180) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, lr, w, total, value in got:
        assert (r, lr, w) == (rank, rank, 2)
        assert total == 2.0                    # the slower rank's time
        assert value == pytest.approx(2 * 100 / 2.0)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_over_ranks(0.5, 10, 1) == (0.5, 20.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_step_bytes_are_the_stated_algorithmic_bytes():
    """Per sequence and layer: indexer keys (N x 128 B, FULL and REINDEX), K selected FP4
    entries (324 B each) and the window (W x 576 x 2 B): 346,292,224 B for 32 sequences at
    32768 entries, K = 2048, W = 128, FULL -> REINDEX -> REUSE."""
    import bench
    import csa2_inputs as ci
    cfg = ci.DECODE_128K
    per_seq = 2 * cfg.N * 128 + 3 * (cfg.K * 324 + cfg.W * 576 * 2)
    assert bench.algorithmic_bytes_per_step(cfg) == per_seq * cfg.B == 346_292_224


def test_reference_arm_line_has_the_contract_keys():
    """The reference arm (the oracle on the host cores) prints one JSON line with the bench
    contract's keys, its own cpu_baseline and an e2e entry that moves no bytes."""
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("env_ranks,gpus", [(None, 2), (("0", "2"), 2), (("1", "2"), 2), (("0", "4"), 1)])
def test_gpu_arm_refuses_more_than_one_gpu(env_ranks, gpus):
    """No kernel of the library runs under more than one rank: the GPU arm refuses before
    importing torch's CUDA runtime, rank 0 prints one "unavailable" line, the others nothing."""
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    if env_ranks:
        env.update(RANK=env_ranks[0], LOCAL_RANK=env_ranks[0], WORLD_SIZE=env_ranks[1])
    r = subprocess.run([sys.executable, "bench.py", "--gpus", str(gpus), "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "refused" in r.stderr
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    if env_ranks and env_ranks[0] != "0":
        assert lines == []
    else:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert "unavailable" in d and d["n_gpus"] >= 2 and "value" not in d
