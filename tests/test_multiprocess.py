"""The benchmark's multi-rank logic on CPU: two processes over gloo.

Under torchrun every rank decodes its own token stream (replicas: the path
has no exchange step); rank 0 reports all ranks' tokens over the slowest
rank's time.  Here each rank reports a different time and token count and
the aggregate is checked; the reference arm prints on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    ms = [120.0, 150.0][rank]          # each rank's timed region
    t = bench.max_over_ranks(ms, world, "cpu")
    value, t_max = bench.aggregate([t], [1000 * world], world)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, t, value, t_max))


def test_max_over_ranks_and_aggregate_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, value, t_max in out:
        assert t == 150.0 and t_max == 150.0       # the slowest rank's time
        assert value == pytest.approx(2000 / 0.150)  # all ranks' tokens over it


def test_max_over_ranks_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", PI_REF_BUDGET_S="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--gpus", "2",
                        "--workload", "opt6.7b_ffn_d4096_n16384_r128_f16"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env.update(RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--gpus", "2",
                        "--workload", "opt6.7b_ffn_d4096_n16384_r128_f16"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_stack_oracle_sample_walks_every_layer_on_the_host():
    # the CPU baseline of the layer stack, on a tiny 3-layer stack built by
    # the host generator: every token goes through every layer in order
    import torch
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import synth
    w = dict(d=64, n=256, r=16, dtype="f16", seed=9, layers=3)
    keep, hosts = [], []
    for l in range(3):
        L = synth.make_layer(64, 256, 16, "f16", alpha=0.9, density=0.1, seed=9, layer=l)
        rec = np.concatenate([L.W1, L.W2], axis=1).view(np.int16)
        g = {"A": torch.from_numpy(L.A.view(np.int16)), "Bm": torch.from_numpy(L.Bm.view(np.int16)),
             "b1": torch.from_numpy(L.b1), "b2": torch.from_numpy(L.b2)}
        keep.append((g, torch.from_numpy(rec)))
        hosts.append(L)
    done, dt, cores = bench.stack_oracle_sample(w, keep, tokens=4, warm=1, budget_s=60.0)
    assert done == 4 and dt > 0 and cores >= 1
    # the host copy of a packed layer is the layer itself
    H = bench.host_layer(w, keep[1][0], keep[1][1])
    for a, b in [(H.A, hosts[1].A), (H.Bm, hosts[1].Bm), (H.W1, hosts[1].W1),
                 (H.W2, hosts[1].W2), (H.b1, hosts[1].b1)]:
        np.testing.assert_array_equal(a, b)
    x = synth.gen_x(9, 0, 1, 64)[0]
    assert np.array_equal(oracle.layer_decode(H, x, residual=True)[3],
                          oracle.layer_decode(hosts[1], x, residual=True)[3])


def _shard_worker(rank, world, port, q):
    # one rank of a neuron-sharded layer on the CPU: the rank's partial
    # output is the oracle's over its own neurons (g, g + G, ...), the
    # exchange is the library's all-gather helper over gloo, and the sum
    # runs in rank order
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import activation_sparse_decode_rank_gb300 as pi
    from activation_sparse_decode_rank_gb300 import sharded
    import oracle
    import synth
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        d, n, r, hot = 96, 301, 16, 40
        L = synth.make_layer(d, n, r, "f16", alpha=0.9, density=0.15, seed=61)
        desc = pi.make_desc(d, n, r, "f16", False, hot)
        sd = sharded.shard_desc(desc, world, rank)
        rows = np.arange(rank, n, world)
        assert sd.n == len(rows) and sd.hot_prefix == int((rows < hot).sum())
        part_layer = synth.Layer(d, sd.n, r, "f16", False, np.ascontiguousarray(L.A[rows]), L.Bm,
                                 np.ascontiguousarray(L.b1[rows]), np.ascontiguousarray(L.W1[rows]),
                                 np.ascontiguousarray(L.W2[rows]),
                                 L.b2 if rank == 0 else np.zeros_like(L.b2), {})
        x = synth.gen_x(62, 0, 1, d)[0]
        _, idx, y, _ = oracle.layer_decode(part_layer, x)
        parts = sharded.exchange(torch.from_numpy(y.reshape(1, d)), world)
        lists = [None] * world
        dist.all_gather_object(lists, (rows[idx]).tolist())
        ysum = np.zeros(d)
        for g in range(world):  # rank order
            ysum = ysum + parts[g, 0].numpy()
        _, gidx, yfull, _ = oracle.layer_decode(L, x)
        merged = sorted(v for lst in lists for v in lst)
        q.put((rank, merged == gidx.tolist(), float(np.abs(ysum - yfull).max()),
               float(np.abs(yfull).max())))
    finally:
        dist.destroy_process_group()


def test_sharded_layer_gloo_two_ranks_matches_the_whole_layer():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, same_set, diff, scale in out:
        assert same_set                   # the shards' lists partition the active set
        assert diff <= 1e-12 * scale      # partial sums in rank order: fp64 rounding only
