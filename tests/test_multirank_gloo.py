"""The multi-rank path on CPU: two ranks over gloo.

The path shards by request with no exchange inside it: every rank runs its own
replica (block pool, allocator, scheduler, kernels).  The only cross-rank step
is the benchmark's reduction of whole-job figures: the slowest rank's time and
the units all ranks processed.  These tests run that reduction and two
independent scheduler replicas as real gloo ranks (world size 2), and check
the reference arm's rank handling.  No GPU is involved.
"""

import hashlib
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2
REPLICA_STEPS = 80


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica_spec():
    from workloads import trace_spec
    # a small pool so that preemption happens within a few dozen steps
    return trace_spec(steps=REPLICA_STEPS, num_blocks=2048, prompt_median=512)


def _sched_config(spec):
    from oracle.scheduler import SchedConfig
    return SchedConfig(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                       spec.max_model_len, spec.block_size, spec.num_blocks,
                       spec.max_model_len // spec.block_size)


def _digest(plans) -> str:
    return hashlib.sha256(json.dumps(plans, sort_keys=True).encode()).hexdigest()


def _run_cpp_replica(rank: int):
    """One rank's scheduler replica through the library's C++ host path."""
    import paged_kv_cache_36_gb300 as pkv
    from workloads import generate_arrivals
    spec = _replica_spec()
    c = _sched_config(spec)
    s = pkv.Scheduler(c.max_num_seqs, c.max_num_batched_tokens, c.chunk_size, c.max_model_len,
                      c.block_size, c.num_blocks, c.max_blocks_per_req)
    by_step = {}
    for a in generate_arrivals(spec, name=f"rank{rank}"):
        by_step.setdefault(a.step, []).append(a)
    plans, preempted = [], 0
    for step in range(spec.steps):
        for a in by_step.get(step, []):
            s.add_request(a.req_id, a.prompt_len, a.max_output)
        pc = s.step()
        _, _, _, _, slots = s.metadata()
        plans.append([pc["entries"], pc["preempted"], pc["admitted"], slots.tolist()])
        preempted += len(pc["preempted"])
        s.finish_step(True)
    return _digest(plans), preempted


def _run_oracle_replica(rank: int):
    from oracle.scheduler import NaiveScheduler
    from workloads import generate_arrivals
    spec = _replica_spec()
    ref = NaiveScheduler(_sched_config(spec), deep_checks=False)
    by_step = {}
    for a in generate_arrivals(spec, name=f"rank{rank}"):
        by_step.setdefault(a.step, []).append(a)
    plans, preempted = [], 0
    for step in range(spec.steps):
        for a in by_step.get(step, []):
            ref.add_request(a.req_id, a.prompt_len, a.max_output)
        pr = ref.step()
        _, _, _, _, slots = ref.metadata(pr)
        plans.append([pr.entries, pr.preempted, pr.admitted, list(slots)])
        preempted += len(pr.preempted)
        ref.finish_step(True)
    return _digest(plans), preempted


def _worker(rank: int, port: int, task: str, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(WORLD))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        if task == "combine":
            import bench
            # rank r took 1 + r ms over 100 (r + 1) units
            ms, units = bench.combine_ranks(1.0 + rank, 100.0 * (rank + 1), dist, "cpu")
            result = (ms, units)
        else:
            mine = _run_cpp_replica(rank)
            gathered = [None] * WORLD
            dist.all_gather_object(gathered, mine)
            result = gathered
        out.put((rank, result))
    finally:
        dist.destroy_process_group()


def _run_ranks(task: str):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, task, out)) for r in range(WORLD)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in range(WORLD):
            rank, res = out.get(timeout=240)
            results[rank] = res
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    return results


def test_combine_ranks_takes_slowest_time_and_sums_units():
    res = _run_ranks("combine")
    # every rank sees the job's figures: the max time and the summed units
    assert res[0] == res[1] == (2.0, 300.0)


def test_combine_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.combine_ranks(3.5, 42.0) == (3.5, 42.0)


def test_replica_schedulers_run_independently():
    """Each rank plans its own requests on its own pool; the plans match the
    oracle's for that rank's trace, so no rank's state leaks into another's."""
    pytest.importorskip("paged_kv_cache_36_gb300")
    res = _run_ranks("replicas")
    assert res[0] == res[1]            # all_gather hands every rank both digests
    gathered = res[0]
    for rank in range(WORLD):
        want = _run_oracle_replica(rank)
        assert tuple(gathered[rank]) == want
        assert want[1] > 0             # the small pool forces preemption
    assert gathered[0][0] != gathered[1][0]


def _reference_arm(rank: int, steps: int):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(WORLD))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--gpus", str(WORLD), "--steps", str(steps), "--warmup", "3"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_other_ranks_exit_without_work():
    p = _reference_arm(1, 1)
    assert p.returncode == 0 and p.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    p = _reference_arm(0, 1)
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == WORLD and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
