"""The N > 1 host logic on CPU: world-size-2 gloo ranks.

By default every rank runs its own full workload (weak scaling); the step time
reported is the slowest rank's and the value counts every rank's FLOPs.  With
a head split the B*H heads of one workload are dealt out in contiguous
blocks: the blocks must be disjoint and complete, and the slices the ranks
compute must equal the same rows of a one-rank run (checked here with the
fp64 oracle standing in for each rank's GPU).  The reference arm runs on rank
0 only; other ranks exit at once.
"""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + 0.5 * rank, world)   # ranks: 1.0 ms, 1.5 ms
        out[rank] = (ms, bench.whole_job_tflops(3e12, world, ms))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket

    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_ranks_take_slowest_time_and_sum_work():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, tf = res[r]
        assert ms == pytest.approx(1.5)
        assert tf == pytest.approx(2 * 3e12 / 1.5e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.whole_job_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_bench_rejects_short_warmup():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_reference_arm_prints_one_json_line():
    import json

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "0", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_head_range_blocks_are_disjoint_complete_and_even():
    sys.path.insert(0, ROOT)
    from exact_attention_82_gb300.shard import head_range

    for bh in range(0, 41):
        for world in range(1, 10):
            ranges = [head_range(bh, world, r) for r in range(world)]
            covered = []
            for start, count in ranges:
                covered += list(range(start, start + count))
            assert covered == list(range(bh)), (bh, world, ranges)  # disjoint, complete, in rank order
            sizes = [c for _, c in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        head_range(4, 2, 2)


def _shard_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from exact_attention_82_gb300.inputs import bf16_bits, make_qkv
    from exact_attention_82_gb300.shard import head_range, head_slice

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = {}
        for causal in (False, True):
            q, k, v = make_qkv(1, 5, 70, 70, 64, seed=77)   # 5 heads over 2 ranks: 3 + 2
            start, count = head_range(5, world, rank)
            qs, ks, vs = (head_slice(t, start, count).contiguous() for t in (q, k, v))
            o, lse = oracle.attn_fwd(bf16_bits(qs), bf16_bits(ks), bf16_bits(vs), 0.125, causal)
            parts = [None] * world
            dist.all_gather_object(parts, (start, count, o, lse))
            res[causal] = parts
        out[rank] = res
    finally:
        dist.destroy_process_group()


def test_two_ranks_split_heads_match_one_rank_run():
    import numpy as np

    sys.path.insert(0, ROOT)
    import oracle
    from exact_attention_82_gb300.inputs import bf16_bits, make_qkv

    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_shard_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    q, k, v = make_qkv(1, 5, 70, 70, 64, seed=77)
    for causal in (False, True):
        o_ref, lse_ref = oracle.attn_fwd(bf16_bits(q), bf16_bits(k), bf16_bits(v), 0.125, causal)
        for r in range(world):
            parts = res[r][causal]   # every rank gathered the same slices
            seen = np.zeros(5, dtype=int)
            o = np.full_like(o_ref, np.nan)
            lse = np.full_like(lse_ref, np.nan)
            for start, count, po, pl in parts:
                seen[start:start + count] += 1
                o[0, start:start + count] = po[0]
                lse[0, start:start + count] = pl[0]
            assert (seen == 1).all()                      # disjoint and complete
            assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)


def test_bench_spawns_its_own_ranks_and_rejects_a_mismatch():
    sys.path.insert(0, ROOT)
    import bench

    cmd = bench.spawn_command(["--gpus", "4", "--steps", "5"], 4, 29555)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--master-addr=127.0.0.1" in cmd
    assert "--master-port=29555" in cmd
    assert cmd[-5].endswith("bench.py") and cmd[-4:] == ["--gpus", "4", "--steps", "5"]
    # a launcher that started fewer ranks than --gpus asks for is an error, not a 1-GPU result
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 2 and "WORLD_SIZE=1" in r.stderr


def test_rank_workload_split():
    sys.path.insert(0, ROOT)
    import bench
    from exact_attention_82_gb300.inputs import WORKLOADS

    w = WORKLOADS[1]   # B=8, H=16
    parts = [bench.rank_workload(w, 3, r, "heads") for r in range(3)]
    assert [(s, c) for _, s, c in parts] == [(0, 43), (43, 43), (86, 42)]
    assert sum(p.flops for p, _, _ in parts) == pytest.approx(w.flops)
    assert all(p.B == 1 and p.H == c for p, _, c in parts)
    same, s0, c0 = bench.rank_workload(w, 3, 1, "none")
    assert same is w and (s0, c0) == (0, 128)
