#!/usr/bin/env python3
"""Benchmark of the GB300 KV-page codec: encode + decode GB/s of raw KV and the
HBM roofline fraction of the dominant kernel.

One step = every codec arm of the workload, encode then decode, over the whole
synthetic KV cache (resident in HBM; 4.8 GB of source pages, far larger than
the 129 MB L2, so no flush is needed between steps).  Default workload:
Qwen3-8B-shaped KV (36 layers, 8 KV heads, D=128, FP16, 4 x 8192 tokens in
16-token pages) with the FP8 K16/V8 arm (V only) and the FP8 K8/V8 arm, both
with dynamic per-token/head scales.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference] [--partition]

N > 1 runs one process per GPU (torchrun): every rank codes its own copy of the
workload (weak scaling), or with --partition its own contiguous range of the
cache's layers (strong scaling).  There is no data-path collective: a gloo
barrier, a max of the timings and sums of the work are the only cross-rank
operations.  `--impl reference` times the plain CPU oracle on a bounded sample
of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_cache_page_gb300 import codec as K  # noqa: E402
from kv_cache_page_gb300 import synth  # noqa: E402

METRIC = "codec encode/decode GB/s of raw KV (1×GB300) and % of HBM roofline"
UNIT = "GB/s"
GB = 1e9
DESC_BYTES = 24


# ----------------------------------------------------------------------------- setup
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return dist
    return None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class Arm:
    """One codec arm bound to device buffers: codec handle, descriptors,
    encoded buffer, statuses and restore destinations."""

    def __init__(self, case: synth.Case, arm: synth.Arm, dev_layers, device, part=None):
        self.case, self.arm = case, arm
        self.codec = K.Codec(dtype="fp16" if case.dtype == torch.float16 else "bf16",
                             layout=case.layout, head_dim=case.head_dim,
                             num_kv_heads=case.num_heads, block_tokens=case.block_tokens,
                             num_layers=case.num_layers, num_blocks=case.num_blocks,
                             strides=case.strides, k_codec=arm.k_codec, v_codec=arm.v_codec,
                             protect=arm.protect, rotation_seed=case.seed,
                             fixed_amax=None if case.fixed_amax is None else case.fixed_amax.numpy())
        self.seg = [self.codec.segment_bytes(r)[0] for r in (0, 1)]
        raw_seg = self.codec.segment_bytes(0)[1]
        rows, self.total = synth.segment_list(case, arm, self.seg)
        if part is not None:  # (world, rank): this rank's layers only, slots at their offsets
            rows = synth.partition_rows(rows, *part)
        self.rows = rows
        self.n = len(rows)
        self.descs = K.descriptors(rows, device)
        self.src = dev_layers
        self.enc = torch.empty(self.total, dtype=torch.uint8, device=device)
        self.status = torch.empty(self.n, dtype=torch.uint8, device=device)
        self.dst = [None if t is None else torch.empty_like(t) for t in dev_layers]
        # which layer tensors this arm touches (separate layout: K/V by role)
        mine = sorted({r[0] for r in rows})
        if case.layout == "separate":
            used = {2 * l + r for l in mine for r in arm.roles}
        else:
            used = set(mine)
        self.used = sorted(used)
        self.layout = case.layout
        self.src_view = [t if i in used else None for i, t in enumerate(dev_layers)]
        self.dst_view = [t if i in used else None for i, t in enumerate(self.dst)]
        prot = [l for l in range(case.num_layers)
                if l < arm.protect[0] or l >= case.num_layers - arm.protect[1]]
        self.prot = set(prot)
        self.n_coded = sum(1 for r in rows if r[0] not in prot)  # segments actually transformed
        self.raw_seg = raw_seg
        self.raw_bytes = self.n_coded * raw_seg
        nv = case.num_heads * case.block_tokens
        self.alg_bytes_enc = sum(raw_seg + self.seg[r[2]] for r in rows if r[0] not in prot) + \
            self.n * (DESC_BYTES + 1)
        self.alg_bytes_dec = self.alg_bytes_enc
        self.vectors = self.n_coded * nv
        codecs = sorted({c for c, r in ((arm.k_codec, 0), (arm.v_codec, 1)) if r in arm.roles and c != "none"})
        self.kname = "+".join(codecs)

    def encode(self, stream=None):
        self.codec.encode(self.src_view, self.descs, self.n, self.enc, self.total, self.status, stream)

    def decode(self, stream=None):
        self.codec.decode(self.dst_view, self.descs, self.n, self.enc, self.total, self.status, None,
                          stream)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.lines = []
        target = None
        try:
            u = torch.cuda.get_device_properties(device_index).uuid
            target = "GPU-" + str(u)
        except Exception:
            target = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if target:
            cmd += ["-i", target]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- traffic record
def recorded_traffic(kname, units):
    """DRAM bytes per launch from the committed ncu summary, scaled by units,
    when the files the kernel is compiled from are unchanged since the
    capture; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        import hashlib
        k = json.load(open(p))["kernels"].get(kname)
        if not k:
            return None
        h = hashlib.sha256()
        for f in sorted(k["sources"]):
            h.update(open(os.path.join(ROOT, f), "rb").read())
        if h.hexdigest() != k["sources_sha256"]:
            return None
        return k["dram_bytes_per_unit"] * units
    except Exception:
        return None


# ----------------------------------------------------------------------------- GPU arm
def run_gpu(args, dist, world, rank, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    case = synth.make_case(args.workload, device=device, seed=args.seed, num_layers=args.layers,
                           num_blocks=args.pages, head_dim=args.head_dim)
    part = (world, rank) if args.partition else None
    arm_list = case.arms
    if args.codecs:  # profiling: one arm with the given K and V codecs on this workload's pages
        kc, vc = args.codecs.split(",")
        roles = tuple(r for r, c in ((0, kc), (1, vc)) if c != "none")
        arm_list = [synth.Arm(f"{kc}+{vc}", kc, vc, roles, case.arms[0].protect)]
    arms = [Arm(case, a, case.layers, device, part) for a in arm_list
            if args.arm is None or a.name == args.arm]
    stream = torch.cuda.current_stream(device)

    def step(events=None):
        for a in arms:
            for fn, tag in ((a.encode, "encode"), (a.decode, "decode")):
                if events is not None:
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                    events.append((f"{a.arm.name}:{a.kname}_{tag}", a, tag, e0, e1))
                else:
                    fn()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    statuses = [a.status.cpu() for a in arms]
    n_encoded = int(sum_over_ranks(dist, sum(int((s == K.SEG_ENCODED).sum()) for s in statuses)))

    clocks = ClockSampler(local)
    time.sleep(0.3)
    events = []
    barrier(dist)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step(events)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    ms_total = max_over_ranks(dist, ms_total)
    raw_per_step = sum(2 * a.raw_bytes for a in arms)       # encode + decode
    value = sum_over_ranks(dist, raw_per_step * args.steps) / (ms_total / 1e3) / GB

    # per-kernel live durations (CUDA events on the launching stream)
    per = {}
    for name, a, tag, e0, e1 in events:
        d = per.setdefault(name, {"ms": [], "arm": a, "tag": tag})
        d["ms"].append(e0.elapsed_time(e1))
    kernels = {}
    for name, d in per.items():
        a = d["arm"]
        avg = sum(d["ms"]) / len(d["ms"])
        alg = a.alg_bytes_enc if d["tag"] == "encode" else a.alg_bytes_dec
        kernels[name] = {"launches": len(d["ms"]), "avg_ms": avg, "total_ms": sum(d["ms"]),
                         "alg_bytes": alg, "achieved_gbs": alg / (avg / 1e3) / GB,
                         "raw_gbs": a.raw_bytes / (avg / 1e3) / GB, "vectors": a.vectors}
    dom = max(kernels, key=lambda k: kernels[k]["total_ms"])
    peak, peak_kind = load_peaks()
    dk = kernels[dom]
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(dk["achieved_gbs"], 1),
                "peak": peak, "unit": "GB/s", "frac": round(dk["achieved_gbs"] / peak, 4),
                "peak_source": f"{peak_kind} hbm_gbs (copy)",
                "traffic": recorded_traffic(dom.split(":", 1)[1], dk["vectors"])}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, arms, stream, dist)
    host_link = None
    if args.host_link and world == 1:
        host_link = run_host_link(args, arms, stream)
    integrity = run_integrity(args, arms, stream, peak) if args.integrity else None

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True,
        "scaling": "strong" if args.partition else "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; see kv_cache_page_gb300/synth.py)",
        "config": {"workload": args.workload, "arms": [a.arm.name for a in arms],
                   "source_dtype": "fp16" if case.dtype == torch.float16 else "bf16",
                   "layers": case.num_layers, "pages_per_layer": case.num_blocks,
                   "kv_heads": case.num_heads, "head_dim": case.head_dim,
                   "raw_kv_bytes_per_step": raw_per_step, "segments_encoded": n_encoded,
                   "l2": "inputs larger than L2 (no flush)",
                   "parallelism": (f"layer partition x{world}" if args.partition else f"replicas x{world}")},
        "roofline": roofline,
        "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                    for k, v in kernels.items()},
        "gpu_launches": len(events),
        "clocks": clk,
        "e2e": e2e,
        "host_link": host_link,
        "integrity": integrity,
    }
    shrunk = args.layers is not None or args.pages is not None or args.arm is not None or bool(args.codecs)
    if shrunk:
        result["config"]["reduced"] = True
    if args.extra and world == 1 and not shrunk:
        result["other_workloads"] = run_extra(args, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not shrunk:
        result["cpu_baseline"] = cpu_baseline(args, case_name=args.workload, seconds=args.cpu_seconds)
    for a in arms:
        a.codec.close()
    return result




def run_e2e(args, arms, stream, dist):
    """Same step through the C ABI with host buffers: raw pages H2D from pinned
    memory, encode with the slots and statuses written straight into pinned
    host memory (offload), decode reading them from there into the engine
    pages (restore), restored pages D2H.  The slot bytes cross the host link
    inside the kernels; they count as the step's D2H (offload) and H2D
    (restore) traffic.

    The value is the median of three timed trials of the same steps.

    The step runs in chunks of args.e2e_chunk_layers layers, chunk c on stream
    c % args.e2e_streams (each chunk: its pages H2D, encode and decode of its
    segments, its restored pages D2H), so that one chunk's H2D copies, another's
    kernels and a third's D2H copies share the full-duplex host link.  A
    chunk's descriptors and statuses are a contiguous slice (the segment list
    is layer-major) and its slots sit at their absolute offsets."""
    host = []
    for a in arms:
        src_h = [t.cpu().pin_memory() if i in a.used else None for i, t in enumerate(a.src)]
        dst_h = [torch.empty_like(t, device="cpu").pin_memory() if i in a.used else None
                 for i, t in enumerate(a.src)]
        enc_h = torch.empty(a.total, dtype=torch.uint8).pin_memory()
        st_h = torch.empty(a.n, dtype=torch.uint8).pin_memory()
        host.append((src_h, dst_h, enc_h, st_h))
    h2d = d2h = 0
    for a, (src_h, dst_h, enc_h, st_h) in zip(arms, host):
        for i in a.used:
            h2d += src_h[i].numel() * 2
            d2h += dst_h[i].numel() * 2
        h2d += a.total + a.n
        d2h += a.total + a.n

    chunks = []
    for a, (src_h, dst_h, enc_h, st_h) in zip(arms, host):
        layers = [r[0] for r in a.rows]
        assert layers == sorted(layers), "segment list must be layer-major"
        order = sorted(set(layers))
        for c0 in range(0, len(order), args.e2e_chunk_layers):
            group = set(order[c0:c0 + args.e2e_chunk_layers])
            d0 = layers.index(min(group))
            d1 = len(layers) - layers[::-1].index(max(group))
            idx = [i for i in a.used if (i // 2 if a.layout == "separate" else i) in group]
            chunks.append((a, idx, d0, d1, src_h, dst_h, enc_h, st_h))
    streams = [torch.cuda.Stream(device=stream.device) for _ in range(args.e2e_streams)]
    for s in streams:
        s.wait_stream(stream)

    def step():
        for k, (a, idx, d0, d1, src_h, dst_h, enc_h, st_h) in enumerate(chunks):
            s = streams[k % len(streams)]
            descs = a.descs[d0 * DESC_BYTES:d1 * DESC_BYTES]
            with torch.cuda.stream(s):
                for i in idx:
                    a.src[i].copy_(src_h[i], non_blocking=True)
                a.codec.encode(a.src_view, descs, d1 - d0, enc_h, a.total, st_h[d0:d1], s)
                a.codec.decode(a.dst_view, descs, d1 - d0, enc_h, a.total, st_h[d0:d1], None, s)
                for i in idx:
                    dst_h[i].copy_(a.dst[i], non_blocking=True)

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, args.e2e_steps))
    raw = sum(2 * a.raw_bytes for a in arms)
    # the host side of the link is shared with other work on the machine:
    # three timed trials of `steps` steps each, the median reported, all listed
    trials = []
    for _ in range(3):
        barrier(dist)
        t0 = time.perf_counter()
        for _ in range(steps):
            step()
        torch.cuda.synchronize()
        barrier(dist)
        sec = max_over_ranks(dist, time.perf_counter() - t0)
        trials.append(sum_over_ranks(dist, raw * steps) / sec / GB)
    value = statistics.median(trials)
    link = link_ceiling(arms, host, streams)
    link_raw = raw / link["both_s"] / GB          # raw KV per second if the step were only its copies
    return {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "trials": [round(v, 2) for v in trials],
            "path": "pages copied H2D/D2H from pinned memory; slots and statuses in pinned host "
                    f"memory, moved by the kernels; chunks of {args.e2e_chunk_layers} layers "
                    f"pipelined over {args.e2e_streams} streams",
            "link_ceiling_gbs": round(link_raw, 2),
            "frac_of_link": round(value / link_raw, 4),
            "link": {k: (round(v, 2) if isinstance(v, float) else v) for k, v in link.items()}}


def link_ceiling(arms, host, streams):
    """The host link's own rate for the end-to-end step's bytes: plain
    cudaMemcpyAsync copies of exactly the bytes a step moves (the pages in and
    out, the slots and statuses once each way), H2D alone, D2H alone, and
    both at once on two streams (the link is full duplex).  Best of 3 runs,
    host clock around a device synchronize."""
    h2d_pairs, d2h_pairs = [], []
    for a, (src_h, dst_h, enc_h, st_h) in zip(arms, host):
        for i in a.used:
            h2d_pairs.append((a.src[i], src_h[i]))
            d2h_pairs.append((dst_h[i], a.dst[i]))
        h2d_pairs += [(a.enc, enc_h), (a.status, st_h)]
        d2h_pairs += [(enc_h, a.enc), (st_h, a.status)]
    bi = sum(d.numel() * d.element_size() for d, _ in h2d_pairs)
    bo = sum(d.numel() * d.element_size() for d, _ in d2h_pairs)
    s_in, s_out = streams[0], streams[1 % len(streams)]

    def run(pairs_by_stream):
        best = float("inf")
        for _ in range(3):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for s, pairs in pairs_by_stream:
                with torch.cuda.stream(s):
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best

    t_in = run([(s_in, h2d_pairs)])
    t_out = run([(s_out, d2h_pairs)])
    t_both = run([(s_in, h2d_pairs), (s_out, d2h_pairs)])
    return {"h2d_bytes": bi, "d2h_bytes": bo, "h2d_gbs": bi / t_in / GB, "d2h_gbs": bo / t_out / GB,
            "both_gbs": (bi + bo) / t_both / GB, "both_s": t_both}


def run_host_link(args, arms, stream):
    """Offload and restore with the encoded slots in pinned host memory, per arm:
    zero-copy (the kernels store the slots and statuses into host memory, or load
    them from there, through its device mapping: NVLink-C2C on GB300) against
    staged (device slots + one cudaMemcpyAsync of the slot buffer each way).
    Median of CUDA-event timings on the launching stream; GB/s of raw KV, and of
    host-link bytes (slots + statuses)."""
    out = {}
    reps = max(3, min(args.steps, 10))

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    for a in arms:
        enc_h = torch.empty(a.total, dtype=torch.uint8).pin_memory()
        st_h = torch.empty(a.n, dtype=torch.uint8).pin_memory()
        link = a.total + a.n

        def off_zero():
            a.codec.encode(a.src_view, a.descs, a.n, enc_h, a.total, st_h, stream)

        def res_zero():
            a.codec.decode(a.dst_view, a.descs, a.n, enc_h, a.total, st_h, None, stream)

        def off_staged():
            a.encode(stream)
            enc_h.copy_(a.enc, non_blocking=True)
            st_h.copy_(a.status, non_blocking=True)

        def res_staged():
            a.enc.copy_(enc_h, non_blocking=True)
            a.status.copy_(st_h, non_blocking=True)
            a.decode(stream)

        res = {}
        for tag, fn in (("offload_zero_copy", off_zero), ("restore_zero_copy", res_zero),
                        ("offload_staged", off_staged), ("restore_staged", res_staged)):
            ms = timed(fn)
            res[tag] = {"ms": round(ms, 4), "raw_gbs": round(a.raw_bytes / (ms / 1e3) / GB, 1),
                        "link_gbs": round(link / (ms / 1e3) / GB, 1)}
        res["link_bytes"] = link
        out[a.arm.name] = res
        del enc_h, st_h
    return out


def _median_ms(fn, stream, reps):
    """Median CUDA-event time of fn() on `stream` after two untimed calls."""
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def run_integrity(args, arms, stream, peak):
    """Segment headers (CRC-32 of every encoded slot), per arm.  seal / verify:
    the standalone passes after encode and before decode -- GB/s of slot bytes
    checked and, against the HBM peak, of algorithmic bytes (slots read +
    32-byte headers written or read + descriptors).  one_pass: encode_sealed
    against plain encode and decode_verified against plain decode on the same
    buffers (one pass over the slots when every coded role is FP8, uniform-8 or INT8), with the
    time each adds.  Median CUDA-event times on the launching stream."""
    out = {}
    reps = max(3, min(args.steps, 20))
    for a in arms:
        hdr = torch.empty(a.n * 32, dtype=torch.uint8, device=a.enc.device)
        res = torch.empty(a.n, dtype=torch.uint8, device=a.enc.device)
        a.encode(stream)
        slot_bytes = sum(a.seg[r[2]] for r in a.rows if r[0] not in a.prot)
        alg = slot_bytes + a.n * (32 + DESC_BYTES + 1)
        row = {}
        for tag, fn in (("seal", lambda: a.codec.seal(a.descs, a.n, a.enc, a.total, a.status, hdr, stream)),
                        ("verify", lambda: a.codec.verify(a.descs, a.n, a.enc, a.total, hdr, res, stream))):
            ms = _median_ms(fn, stream, reps)
            row[tag] = {"ms": round(ms, 4), "slot_gbs": round(slot_bytes / (ms / 1e3) / GB, 1),
                        "frac_of_hbm": round(alg / (ms / 1e3) / GB / peak, 4)}
        ok = int((res == K.SEG_ENCODED).sum())
        row["verified_encoded"] = ok
        row["slot_bytes"] = slot_bytes
        t = {
            "encode": _median_ms(lambda: a.encode(stream), stream, reps),
            "encode_sealed": _median_ms(lambda: a.codec.encode_sealed(
                a.src_view, a.descs, a.n, a.enc, a.total, a.status, hdr, stream), stream, reps),
            "decode": _median_ms(lambda: a.decode(stream), stream, reps),
            "decode_verified": _median_ms(lambda: a.codec.decode_verified(
                a.dst_view, a.descs, a.n, a.enc, a.total, hdr, res, stream), stream, reps),
        }
        one = {k + "_ms": round(v, 4) for k, v in t.items()}
        one["seal_adds"] = round(t["encode_sealed"] / t["encode"] - 1.0, 4)
        one["verify_adds"] = round(t["decode_verified"] / t["decode"] - 1.0, 4)
        one["one_pass"] = all(c.startswith("fp8") or c in ("uni8", "int8", "none")
                              for c in (a.arm.k_codec, a.arm.v_codec))
        one["restored"] = int((res == K.SEG_ENCODED).sum())
        row["one_pass"] = one
        out[a.arm.name] = row
        del hdr, res
    return out


def run_extra(args, device):
    """Per-arm encode / decode raw-KV GB/s on the other workloads (context lines;
    the headline is the default workload)."""
    out = {}
    # the head-dim sweep is one layer in its parity form; for timing it is spread
    # over 64 layers of the same law so that the data (0.5-4 GB) is far larger
    # than the 129 MB L2
    specs = [("tiny", {}), ("vllm_packed", {}),
             ("head_dim_sweep", {"head_dim": 32, "num_layers": 64}),
             ("head_dim_sweep", {"head_dim": 64, "num_layers": 64}),
             ("head_dim_sweep", {"head_dim": 128, "num_layers": 64}),
             ("head_dim_sweep", {"head_dim": 256, "num_layers": 64}), ("qwen25_7b_offload", {}),
             ("hiq_qwen3_8b", {})]
    for name, kw in specs:
        if name == args.workload and not kw:
            continue
        case = synth.make_case(name, device=device, **kw)
        label = name + (f"_d{kw['head_dim']}_x{kw['num_layers']}" if kw else "")
        subs = []
        for arm in case.arms:
            if arm.k_codec != arm.v_codec and len(arm.roles) == 2:
                # one launch per role: time them apart
                subs += [synth.Arm(f"{arm.name}.K", arm.k_codec, "none", (0,), arm.protect),
                         synth.Arm(f"{arm.name}.V", "none", arm.v_codec, (1,), arm.protect)]
            else:
                subs.append(arm)
        for arm in subs:
            a = Arm(case, arm, case.layers, device)
            for _ in range(3):
                a.encode()
                a.decode()
            torch.cuda.synchronize()
            res = {}
            for tag, fn, alg in (("encode", a.encode, a.alg_bytes_enc), ("decode", a.decode, a.alg_bytes_dec)):
                # back-to-back launches between two events on the launching
                # stream, as in the headline loop (a host sync per launch would
                # add the host's call latency to every short kernel)
                reps = max(5, args.steps)
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(reps):
                    fn()
                e1.record()
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / reps
                res[tag] = {"ms": round(ms, 4), "raw_gbs": round(a.raw_bytes / (ms / 1e3) / GB, 1),
                            "hbm_gbs": round(alg / (ms / 1e3) / GB, 1)}
            res["fits_in_l2"] = (a.raw_bytes + a.total) < 129e6
            out[f"{label}:{arm.name}"] = res
            a.codec.close()
        del case
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- CPU oracle
# One workload per codec family for the per-codec CPU baseline.
CPU_FAMILIES = (("fp8", "qwen3_8b"), ("turboquant+uniform", "vllm_packed"),
                ("uniform8", "qwen25_7b_offload"), ("int8_head", "hiq_qwen3_8b"))


def _oracle_sample(case_name, blocks):
    """Host copies of a bounded sample of the workload + per-arm oracle inputs:
    `blocks` pages of one layer that no arm protects (the workload is built
    with just enough layers for that)."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle as O
    from kvcases import host_bits, oracle_descs, oracle_geom
    probe = synth.make_case(case_name, num_layers=1, num_blocks=1)
    pf = max(a.protect[0] for a in probe.arms)
    pl = max(a.protect[1] for a in probe.arms)
    layers = pf + pl + 1
    case = synth.make_case(case_name, num_layers=layers, num_blocks=blocks)
    bits = [host_bits(t) for t in case.layers]
    work = []
    for arm in case.arms:
        g = oracle_geom(case, arm)
        seg = [O.segment_enc_bytes(g, r) for r in (0, 1)]
        rows, total = synth.segment_list(case, arm, seg, layers=[pf])
        work.append((g, rows, total, case.raw_segment_bytes))
    return O, bits, work, oracle_descs, pf


def _oracle_pass(O, bits, work, oracle_descs, threads):
    """Encode then decode every arm of the sample, segments split over threads
    (ctypes releases the GIL).  Returns raw bytes processed (both directions)."""
    done = 0

    def one(g, rows, total):
        enc, st = O.encode(g, bits, oracle_descs(rows), total)
        outs = [b.copy() for b in bits]
        O.decode(g, outs, oracle_descs(rows), enc, st)

    jobs = []
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for g, rows, total, raw_seg in work:
            chunk = -(-len(rows) // threads)
            for k in range(0, len(rows), chunk):
                jobs.append(ex.submit(one, g, rows[k:k + chunk], total))
            done += 2 * len(rows) * raw_seg
        for j in jobs:
            j.result()
    return done


def _timed_oracle(case_name, threads, seconds):
    """GB/s of raw KV of the oracle on `threads` host threads: a warm-up pass,
    then passes until `seconds` have elapsed (at least one)."""
    blocks = 4 if threads == 1 else 8 * threads
    O, bits, work, od, layer = _oracle_sample(case_name, blocks)
    _oracle_pass(O, bits, work, od, threads)
    t0 = time.perf_counter()
    done, passes = 0, 0
    while True:
        done += _oracle_pass(O, bits, work, od, threads)
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    sec = time.perf_counter() - t0
    return {"value": round(done / sec / GB, 6), "cores": threads,
            "sample": f"{case_name}: layer {layer}, pages 0..{blocks - 1}, every arm, encode+decode, "
                      f"{passes} passes in {sec:.1f} s"}


def cpu_baseline(args, case_name, seconds):
    """The oracle as it stands on the host cores: the benchmark's workload on
    all cores (the reported value) and on one core, and one workload per
    codec family on one and on all cores."""
    threads = os.cpu_count() or 1
    main = _timed_oracle(case_name, threads, seconds)
    one = _timed_oracle(case_name, 1, seconds / 2)
    per = {}
    for fam, name in CPU_FAMILIES:
        per[fam] = {"workload": name, "all_cores": _timed_oracle(name, threads, seconds / 4),
                    "one_core": _timed_oracle(name, 1, seconds / 4)}
    return {"value": main["value"], "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": main["sample"], "nproc": threads,
            "one_core": {"value": one["value"], "unit": UNIT, "cores": 1, "sample": one["sample"]},
            "per_codec": per}


def run_reference(args):
    threads = os.cpu_count() or 1
    blocks = max(threads, 8)
    O, bits, work, od, layer = _oracle_sample(args.workload, blocks)
    for _ in range(args.warmup):
        _oracle_pass(O, bits, work, od, threads)
    t0 = time.perf_counter()
    done = 0
    for _ in range(args.steps):
        done += _oracle_pass(O, bits, work, od, threads)
    sec = time.perf_counter() - t0
    value = done / sec / GB
    sample = f"{args.workload}: layer {layer}, pages 0..{blocks - 1}, every arm, encode+decode per step"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(sec * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": args.workload, "sample": sample},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="qwen3_8b", choices=list(synth.CASES))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--layers", type=int, default=None, help="shrink the workload (profiling)")
    ap.add_argument("--pages", type=int, default=None, help="pages per layer (profiling)")
    ap.add_argument("--head-dim", type=int, default=None, help="head_dim_sweep point")
    ap.add_argument("--arm", default=None, help="run only this codec arm")
    ap.add_argument("--codecs", default=None,
                    help="profiling: replace the workload's arms by one arm 'K,V' (codec names)")
    ap.add_argument("--no-extra", dest="extra", action="store_false")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunk-layers", type=int, default=4,
                    help="layers per chunk of the pipelined end-to-end step")
    ap.add_argument("--e2e-streams", type=int, default=3,
                    help="streams the end-to-end chunks rotate over")
    ap.add_argument("--no-host-link", dest="host_link", action="store_false",
                    help="skip the host-resident slot offload/restore timings")
    ap.add_argument("--no-integrity", dest="integrity", action="store_false",
                    help="skip the segment header seal/verify timings")
    ap.add_argument("--partition", action="store_true",
                    help="N > 1: rank r codes its own contiguous range of layers (strong scaling) "
                         "instead of a replica of the whole cache")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args(argv)
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    dist = init_dist(world)
    res = run_gpu(args, dist, world, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
