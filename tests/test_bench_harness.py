"""CPU checks of bench.py's multi-rank harness (gloo, world size 2) and of its
reference arm, without a GPU: the barrier, the max of the per-rank timings and
the sum of the per-rank work are the only cross-rank operations."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.init_dist(world)
    bench.barrier(dist)
    t = bench.max_over_ranks(dist, 1.5 + rank)       # rank 1 is the slow one
    w = bench.sum_over_ranks(dist, 10.0 * (rank + 1))
    out.put((rank, t, w))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_total_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]
    assert [r[2] for r in res] == [30.0, 30.0]


def test_reference_arm_json_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, env=env,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, env=env,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""


def _partition_rank(rank, world, port, out):
    """One rank of a partitioned run on the CPU: the oracle codes this rank's
    rows (bench.py's --partition split) and rank 0 gathers every rank's
    statuses and slot bytes."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import torch.distributed as dist
    import bench
    import oracle as O
    from kvcases import host_bits, oracle_descs, oracle_geom
    from kv_cache_page_gb300 import synth
    d = bench.init_dist(world)
    case = synth.make_case("vllm_packed", num_layers=6, num_blocks=3)
    bits = [host_bits(t) for t in case.layers]
    arm = case.arms[0]
    g = oracle_geom(case, arm)
    seg = [O.segment_enc_bytes(g, r) for r in (0, 1)]
    rows, total = synth.segment_list(case, arm, seg)
    mine = synth.partition_rows(rows, world, rank)
    enc, st = O.encode(g, bits, oracle_descs(mine), total)
    part = [(r, int(s), bytes(enc[r[3]:r[3] + seg[r[2]]])) for r, s in zip(mine, st)]
    got = [None] * world if rank == 0 else None
    dist.gather_object(part, got, dst=0)
    if rank == 0:
        cat = [x for p in got for x in p]
        enc1, st1 = O.encode(g, bits, oracle_descs(rows), total)
        ok = [r for r, _, _ in cat] == rows
        ok = ok and [s for _, s, _ in cat] == [int(s) for s in st1]
        ok = ok and all(b == bytes(enc1[r[3]:r[3] + seg[r[2]]]) for r, s, b in cat if s == O.S_ENCODED)
        out.put((ok, len(cat), sorted({r[0] for r, _, _ in got[1]})))
    d.destroy_process_group()


def test_partitioned_ranks_concatenate_to_one_rank_run():
    """--partition: the ranks' rows, concatenated in rank order, are the whole
    segment list; their statuses and slots equal a one-rank run's."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_partition_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok, n, rank1_layers = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ok and n == 6 * 3 * 2
    assert rank1_layers == [3, 4, 5]
