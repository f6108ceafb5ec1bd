"""Seeded synthetic KV caches shaped like the workloads on the source pages.

This module holds no codec arithmetic: it draws random numbers, lays them out
in the engine's page layouts and says which codec arms each workload runs.
Both the CUDA codec's tests/benchmark and the CPU oracle take their inputs
from here.

Workloads (real model KV and the pages' prompt sets are not available, so
seeded distributions stand in for them):

* ``tiny``       1 layer, 4 pages x 16 tokens, 8 KV heads, D=128, FP16, separate
                 K/V; N(0,1), K channels 3, 37, 64, 101 scaled x8 (outliers).
* ``qwen3_8b``   36 layers, 8 KV heads, D=128, FP16, 4 sequences x 8192 tokens in
                 16-token pages; K = N(0,1) x lognormal(0, 0.7) per (layer, head,
                 channel), then a half-split rotary rotation (theta 1e6, positions
                 0..8191 per sequence); V = 0.5 N(0,1).
* ``vllm_packed``  vLLM packed [4096 blocks, 8 heads, 16 tokens, 2x128] BF16 x 32
                 layers, Student-t(4); 1% of (layer, block, role) segments (seed 1)
                 get one nonfinite (half) or one |x| in (448, 1024] (half) element.
* ``head_dim_sweep``  D in {32, 64, 128, 256}, 32 KV heads, 2048 tokens, FP16, one
                 layer, N(0,1); FP8 fixed scales from a 512-token calibration draw
                 (seed 1) of the same law.
* ``qwen25_7b_offload``  28 layers, 4 KV heads, D=128, BF16, 8 x 32768 tokens;
                 heads 0-1 N(0,1), heads 2-3 Student-t(4).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import torch

__all__ = ["Case", "make_case", "CASES", "segment_list", "partition_rows"]


@dataclasses.dataclass
class Arm:
    """One codec configuration run over a workload: codec per role ("none",
    "fp8_cast", "fp8_fixed", "fp8_dynamic", "tq3", "tq4", "uni3", "uni4",
    "uni8", "int8", "tq2", "uni2") and the roles whose segments are submitted."""
    name: str
    k_codec: str
    v_codec: str
    roles: Tuple[int, ...]
    protect: Tuple[int, int] = (0, 0)


@dataclasses.dataclass
class Case:
    name: str
    dtype: torch.dtype
    layout: str                  # "separate" | "packed"
    head_dim: int
    num_heads: int
    block_tokens: int
    num_layers: int
    num_blocks: int
    strides: Tuple[int, int, int]  # (block, token, head) in elements
    layers: List[torch.Tensor]   # separate: [K0, V0, K1, V1, ...]; packed: one per layer
    arms: List[Arm]
    seed: int = 0
    fixed_amax: Optional[torch.Tensor] = None   # float32 [num_layers, 2]

    @property
    def vec_per_segment(self) -> int:
        return self.num_heads * self.block_tokens

    @property
    def raw_segment_bytes(self) -> int:
        return self.vec_per_segment * self.head_dim * 2


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _student_t(shape, nu, g, device):
    z = torch.randn(shape, generator=g, device=device)
    chi2 = torch.zeros(shape, device=device)
    for _ in range(nu):
        chi2 += torch.randn(shape, generator=g, device=device) ** 2
    return z / torch.sqrt(chi2 / nu)


def _separate_strides(T, H, D):
    return (T * H * D, H * D, D)


def _packed_strides(T, H, D):
    # [block, head, token, 2D]: block, token, head strides
    return (H * T * 2 * D, 2 * D, T * 2 * D)


def _rope_(k, positions, theta=1.0e6):
    """Half-split rotary rotation of k [..., T, H, D] (float32, in place) with
    token positions [..., T]."""
    D = k.shape[-1]
    half = D // 2
    inv = theta ** (-torch.arange(half, device=k.device, dtype=torch.float64) * 2.0 / D)
    ang = positions.to(torch.float64)[..., None] * inv          # [..., T, half]
    cos = torch.cos(ang).to(torch.float32)[..., None, :]          # [..., T, 1, half]
    sin = torch.sin(ang).to(torch.float32)[..., None, :]
    x1 = k[..., :half].clone()
    x2 = k[..., half:].clone()
    k[..., :half] = x1 * cos - x2 * sin
    k[..., half:] = x1 * sin + x2 * cos
    return k


def make_case(name: str, *, device="cpu", num_layers: Optional[int] = None,
              num_blocks: Optional[int] = None, head_dim: Optional[int] = None,
              seed: int = 0) -> Case:
    """Build a workload.  `num_layers`/`num_blocks` shrink it (the value law and
    layout stay those of the full workload); `head_dim` picks the sweep point of
    ``head_dim_sweep``."""
    T = 16
    if name == "tiny":
        L, B, H, D = num_layers or 1, num_blocks or 4, 8, 128
        g = _gen(device, seed)
        layers = []
        for _ in range(L):
            k = torch.randn(B, T, H, D, generator=g, device=device)
            k[..., [3, 37, 64, 101]] *= 8.0
            v = torch.randn(B, T, H, D, generator=g, device=device)
            layers += [k.half(), v.half()]
        return Case(name, torch.float16, "separate", D, H, T, L, B, _separate_strides(T, H, D),
                    layers, [Arm("fp8_dynamic_k8v8", "fp8_dynamic", "fp8_dynamic", (0, 1)),
                             Arm("turboquant4", "tq4", "uni4", (0, 1))], seed)

    if name in ("qwen3_8b", "hiq_qwen3_8b"):
        # the HiQCache page's model (Qwen3-8B, BF16 KV, symmetric per-head INT8
        # host copy for K and V) on the same value law, in BF16
        L, B, H, D = num_layers or 36, num_blocks or 2048, 8, 128
        dt = torch.float16 if name == "qwen3_8b" else torch.bfloat16
        g = _gen(device, seed)
        blocks_per_seq = 8192 // T
        pos = (torch.arange(B, device=device) % blocks_per_seq)[:, None] * T + \
            torch.arange(T, device=device)[None, :]                          # [B, T]
        layers = []
        for _ in range(L):
            chan = torch.exp(0.7 * torch.randn(H, D, generator=g, device=device))
            k = torch.randn(B, T, H, D, generator=g, device=device) * chan
            _rope_(k, pos)
            v = 0.5 * torch.randn(B, T, H, D, generator=g, device=device)
            layers += [k.to(dt), v.to(dt)]
        if name == "hiq_qwen3_8b":
            arms = [Arm("int8_head", "int8", "int8", (0, 1))]
        else:
            arms = [Arm("fp8_k16v8_dynamic", "none", "fp8_dynamic", (1,)),
                    Arm("fp8_k8v8_dynamic", "fp8_dynamic", "fp8_dynamic", (0, 1))]
        return Case(name, dt, "separate", D, H, T, L, B, _separate_strides(T, H, D), layers, arms,
                    seed)

    if name == "vllm_packed":
        L, B, H, D = num_layers or 32, num_blocks or 4096, 8, 128
        g = _gen(device, seed)
        layers = [_student_t((B, H, T, 2 * D), 4, g, device).to(torch.bfloat16) for _ in range(L)]
        # 1% of (layer, block, role) segments, chosen with seed 1
        gs = _gen("cpu", seed + 1)
        nseg = L * B * 2
        pick = torch.randperm(nseg, generator=gs)[: max(1, nseg // 100)]
        kinds = torch.randint(0, 4, (pick.numel(),), generator=gs)
        where = torch.randint(0, H * T * D, (pick.numel(),), generator=gs)
        mags = 448.0 + 576.0 * (1.0 - torch.rand(pick.numel(), generator=gs))  # (448, 1024]
        signs = torch.where(torch.rand(pick.numel(), generator=gs) < 0.5, -1.0, 1.0)
        for p, kd, w, m, s in zip(pick.tolist(), kinds.tolist(), where.tolist(), mags.tolist(),
                                  signs.tolist()):
            layer, rest = divmod(p, B * 2)
            blk, role = divmod(rest, 2)
            h, rem = divmod(w, T * D)
            t, e = divmod(rem, D)
            val = [math.inf * s, math.nan, m * s, m * s][kd]
            layers[layer][blk, h, t, role * D + e] = val
        return Case(name, torch.bfloat16, "packed", D, H, T, L, B, _packed_strides(T, H, D),
                    layers, [Arm("turboquant3", "tq3", "uni3", (0, 1), protect=(2, 2)),
                             Arm("turboquant2", "tq2", "uni2", (0, 1), protect=(2, 2))], seed)

    if name == "head_dim_sweep":
        L, B, H = num_layers or 1, num_blocks or 128, 32
        D = head_dim or 128
        g = _gen(device, seed)
        layers = []
        for _ in range(L):
            layers += [torch.randn(B, T, H, D, generator=g, device=device).half(),
                       torch.randn(B, T, H, D, generator=g, device=device).half()]
        gc = _gen(device, seed + 1)
        amax = torch.empty(L, 2, dtype=torch.float32)
        for l in range(L):
            for r in range(2):
                calib = torch.randn(512, H, D, generator=gc, device=device).half().float()
                amax[l, r] = calib.abs().max().cpu()
        return Case(name, torch.float16, "separate", D, H, T, L, B, _separate_strides(T, H, D),
                    layers, [Arm("fp8_fixed_k8v8", "fp8_fixed", "fp8_fixed", (0, 1)),
                             Arm("turboquant4", "tq4", "uni4", (0, 1))], seed, amax)

    if name == "qwen25_7b_offload":
        L, B, H, D = num_layers or 28, num_blocks or 16384, 4, 128
        g = _gen(device, seed)
        layers = []
        for _ in range(L):
            for _role in range(2):
                x = torch.empty(B, T, H, D, device=device)
                x[:, :, :2] = torch.randn(B, T, 2, D, generator=g, device=device)
                x[:, :, 2:] = _student_t((B, T, 2, D), 4, g, device)
                layers.append(x.to(torch.bfloat16))
        return Case(name, torch.bfloat16, "separate", D, H, T, L, B, _separate_strides(T, H, D),
                    layers, [Arm("uniform8", "uni8", "uni8", (0, 1), protect=(2, 2))], seed)

    raise ValueError(f"unknown workload {name!r}")


CASES = ("tiny", "qwen3_8b", "vllm_packed", "head_dim_sweep", "qwen25_7b_offload", "hiq_qwen3_8b")


def partition_rows(rows, world: int, rank: int):
    """The rows (layer, block, role, offset) of one rank when `world` GPUs
    share a cache: rank r takes the layers [L r / world, L (r + 1) / world) of
    the layers the rows cover, so that each rank codes whole layers of its own
    pages and the ranks' rows, concatenated in rank order, are the rows in
    their original (layer-major) order.  Slot offsets are kept."""
    layers = sorted({r[0] for r in rows})
    n = len(layers)
    mine = set(layers[n * rank // world: n * (rank + 1) // world])
    return [r for r in rows if r[0] in mine]


def segment_list(case: Case, arm: Arm, seg_bytes: Sequence[int], layers=None, blocks=None):
    """Descriptors for every (layer, block, role) of the arm, role-major within a
    block, encoded slots packed back to back in that order.  Returns (rows,
    total_bytes) where rows are (layer, block, role, offset) tuples."""
    rows = []
    off = 0
    for layer in (range(case.num_layers) if layers is None else layers):
        for blk in (range(case.num_blocks) if blocks is None else blocks):
            for role in arm.roles:
                rows.append((layer, blk, role, off))
                off += seg_bytes[role]
    return rows, off
