"""Test helpers: turn a synthetic workload into oracle inputs (no codec arithmetic)."""
import numpy as np
import torch

import oracle as O
from kv_cache_page_gb300 import synth

CODEC_IDS = {"none": O.NONE, "fp8_cast": O.FP8_CAST, "fp8_fixed": O.FP8_FIXED,
             "fp8_dynamic": O.FP8_DYNAMIC, "tq3": O.TQ3, "tq4": O.TQ4, "uni3": O.UNI3,
             "uni4": O.UNI4, "uni8": O.UNI8, "int8": O.INT8, "tq2": O.TQ2, "uni2": O.UNI2}


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a tensor as a contiguous uint16 numpy array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16).reshape(-1).copy()


def oracle_geom(case: synth.Case, arm: synth.Arm, reject_abs=448.0, sign_version=1, fixed_overflow="clip"):
    return O.make_geom(
        dtype=O.FP16 if case.dtype == torch.float16 else O.BF16,
        layout=O.SEPARATE if case.layout == "separate" else O.PACKED,
        head_dim=case.head_dim, num_heads=case.num_heads, block_tokens=case.block_tokens,
        num_layers=case.num_layers, num_blocks=case.num_blocks, strides=case.strides,
        codecs=(CODEC_IDS[arm.k_codec], CODEC_IDS[arm.v_codec]), protect=arm.protect,
        seed=case.seed, reject_abs=reject_abs, sign_version=sign_version,
        fixed_overflow={"clip": 0, "reject": 1}[fixed_overflow],
        fixed_amax=None if case.fixed_amax is None else case.fixed_amax.numpy())


def oracle_descs(rows):
    d = np.zeros(len(rows), dtype=O.DESC_DTYPE)
    if rows:
        a = np.array(rows, dtype=np.uint64)
        d["layer"], d["block"], d["role"], d["enc_offset"] = a[:, 0], a[:, 1], a[:, 2], a[:, 3]
    return d


def custom_case(*, D, H, T, L, B, dtype, layout, values="normal", seed=0):
    """A seeded synthetic case of any geometry: per-vector log-normal magnitudes
    ("normal") or Student-t(4) entries ("heavy"), clipped inside the FP8 range."""
    g = torch.Generator().manual_seed(seed)
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16

    def draw(shape):
        if values == "normal":
            x = torch.randn(shape, generator=g) * torch.exp(torch.randn(shape[:-1] + (1,), generator=g))
        elif values == "heavy":
            z = torch.randn(shape, generator=g)
            chi = sum(torch.randn(shape, generator=g) ** 2 for _ in range(4))
            x = z / torch.sqrt(chi / 4)
        return x.clamp(-440, 440).to(tdt)

    if layout == "separate":
        layers = []
        for _ in range(L):
            layers += [draw((B, T, H, D)), draw((B, T, H, D))]
        strides = synth._separate_strides(T, H, D)
    else:
        layers = [draw((B, H, T, 2 * D)) for _ in range(L)]
        strides = synth._packed_strides(T, H, D)
    amax = torch.rand(L, 2, generator=g) * 8 + 0.5
    return synth.Case("custom", tdt, layout, D, H, T, L, B, strides, layers, [], seed, amax)
