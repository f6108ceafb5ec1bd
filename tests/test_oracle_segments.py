"""Pins of the oracle's segment semantics: payload sizes, admission, layouts.

Sources: "KV precision and storage encoding" (OrbitKV), sections "FP8 and
TurboQuant" (payload sizes, range rejection, protected layers, vLLM packed and
separate layouts) and "Ownership, storage and GDS" (nonfinite / oversized
segments stay raw, >= 12.5% saving rule); "Asymmetric KV: methods and results"
(knlp), section "Memory and compatibility" (K16/V8 bytes per pair).
"""
import os

import numpy as np
import pytest
import torch

import oracle as O
from kv_cache_page_gb300 import synth
from kvcases import CODEC_IDS, host_bits, oracle_descs, oracle_geom

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _geom(codecs, D=128, H=8, T=16, L=4, B=4, dtype=O.FP16, layout=O.SEPARATE, protect=(0, 0),
          fixed_amax=None):
    strides = (T * H * D, H * D, D) if layout == O.SEPARATE else (H * T * 2 * D, 2 * D, T * 2 * D)
    return O.make_geom(dtype=dtype, layout=layout, head_dim=D, num_heads=H, block_tokens=T,
                       num_layers=L, num_blocks=B, strides=strides, codecs=codecs,
                       protect=protect, seed=1, fixed_amax=fixed_amax)


def test_payload_sizes_golden():
    rows = [l.split() for l in open(os.path.join(GOLD, "payload_sizes.txt")) if l[0] != "#"]
    for D, bits, role, pay, orig in rows:
        D, bits, pay, orig = int(D), int(bits), int(pay), int(orig)
        k = {3: O.TQ3, 4: O.TQ4}[bits]
        v = {3: O.UNI3, 4: O.UNI4}[bits]
        g = _geom((k, v), D=D)
        nv = 8 * 16
        assert O.segment_raw_bytes(g) == nv * orig
        assert O.segment_enc_bytes(g, 0 if role == "K" else 1) == nv * pay


def test_asymmetric_k16v8_golden():
    kv = dict(l.split() for l in open(os.path.join(GOLD, "asymmetric_k16v8.txt")) if l[0] != "#")
    g = _geom((O.NONE, O.FP8_FIXED), fixed_amax=np.ones((4, 2), np.float32))
    raw = O.segment_raw_bytes(g)          # one role of one page
    enc_v = O.segment_enc_bytes(g, 1)
    nv = 8 * 16
    D = 128
    assert (raw + raw) // (nv * D) == int(kv["bytes_per_pair_native"])
    assert (raw + enc_v) // (nv * D) == int(kv["bytes_per_pair_k16v8"])
    assert int(kv["slots_native"]) * 4 // 3 == int(kv["slots_k16v8"])


@pytest.mark.parametrize("codec,per_vec", [(O.FP8_DYNAMIC, 132), (O.FP8_FIXED, 128),
                                           (O.FP8_CAST, 128), (O.UNI8, 132)])
def test_other_payload_sizes(codec, per_vec):
    g = _geom((codec, codec), fixed_amax=np.ones((4, 2), np.float32))
    assert O.segment_enc_bytes(g, 0) == 128 * per_vec


def test_sizes_round_up_to_128_and_no_saving_rule():
    # D=32, H=1, T=1: one vector; TQ3 K = 12 + 2 = 14 bytes -> one 128-byte slot,
    # which is larger than the 64-byte source: kept raw (needs >= 12.5% saving)
    g = _geom((O.TQ3, O.UNI3), D=32, H=1, T=1, L=1, B=1)
    assert O.segment_enc_bytes(g, 0) == 128
    k = np.zeros(32, np.uint16)
    descs = oracle_descs([(0, 0, 0, 0)])
    _, st = O.encode(g, [k, k.copy()], descs, 128)
    assert st[0] == O.S_RAW_NO_SAVING


def _one_layer_case(values_fn, codec=O.FP8_DYNAMIC, B=6, dtype=O.FP16):
    D, H, T = 64, 2, 16
    g = _geom((codec, codec), D=D, H=H, T=T, L=1, B=B, dtype=dtype)
    rng = np.random.default_rng(0)
    k = rng.standard_normal((B, T, H, D)).astype(np.float32)
    values_fn(k)
    bits = O.f32_to_f16(k) if dtype == O.FP16 else O.f32_to_bf16(k)
    return g, bits.reshape(-1)


def test_admission_statuses():
    def plant(k):
        k[1, 3, 1, 7] = np.inf
        k[2, 0, 0, 0] = np.nan
        k[3, 15, 1, 63] = 448.5       # rounds to 448 in FP16? no: FP16 has 448.5 -> checked below
        k[4, 2, 0, 5] = -449.0
        k[5, 1, 1, 1] = 448.0         # on the boundary: admitted
    g, kb = _one_layer_case(plant)
    seg = O.segment_enc_bytes(g, 0)
    descs = oracle_descs([(0, b, 0, b * seg) for b in range(6)])
    _, st = O.encode(g, [kb, kb.copy()], descs, 6 * seg)
    assert O.f16_to_f32(np.array([O.f32_to_f16(np.array([448.5], np.float32))[0]]))[0] == 448.5
    assert list(st) == [O.S_ENCODED, O.S_RAW_NONFINITE, O.S_RAW_NONFINITE, O.S_RAW_RANGE,
                        O.S_RAW_RANGE, O.S_ENCODED]


def test_nonfinite_beats_range_and_bf16_range():
    def plant(k):
        k[0, 0, 0, 0] = 1000.0
        k[0, 0, 0, 1] = -np.inf
        k[1, 0, 0, 0] = 452.0        # exactly representable in BF16, > 448
    g, kb = _one_layer_case(plant, B=2, dtype=O.BF16)
    seg = O.segment_enc_bytes(g, 0)
    _, st = O.encode(g, [kb, kb.copy()], oracle_descs([(0, 0, 0, 0), (0, 1, 0, seg)]), 2 * seg)
    assert list(st) == [O.S_RAW_NONFINITE, O.S_RAW_RANGE]


def test_policy_protected_and_bad_descriptors():
    D, H, T, L, B = 32, 1, 16, 6, 2
    g = _geom((O.TQ4, O.NONE), D=D, H=H, T=T, L=L, B=B, protect=(2, 1))
    seg = O.segment_enc_bytes(g, 0)
    layers = []
    for _ in range(L):
        layers += [np.zeros(B * T * H * D, np.uint16), np.zeros(B * T * H * D, np.uint16)]
    layers[2 * 3] = None      # layer 3 K missing
    rows = [(0, 0, 0, 0), (1, 1, 0, 0), (2, 0, 0, 0), (4, 1, 0, seg), (5, 0, 0, 0),
            (2, 0, 1, 0),                     # V has no codec
            (6, 0, 0, 0), (2, 2, 0, 0), (3, 0, 0, 0),   # layer / block out of range, NULL pointer
            (2, 0, 0, 8), (2, 0, 0, 2 * seg - 16)]      # misaligned, slot past the end
    d = oracle_descs(rows)
    d["role"][5] = 1
    bad_role = oracle_descs([(2, 0, 2, 0)])
    d = np.concatenate([d, bad_role])
    _, st = O.encode(g, layers, d, 2 * seg)
    assert list(st) == [O.S_RAW_PROTECTED, O.S_RAW_PROTECTED, O.S_ENCODED, O.S_ENCODED,
                        O.S_RAW_PROTECTED, O.S_RAW_POLICY, O.S_BAD_DESC, O.S_BAD_DESC,
                        O.S_BAD_DESC, O.S_BAD_DESC, O.S_BAD_DESC, O.S_BAD_DESC]


def test_oversize_segments_stay_raw():
    # 64 heads x 256 tokens x D=256 x 2 bytes = 8 MiB (encoded); x2 tokens = 16 MiB: still
    # encoded; 4097 tokens -> just above 16 MiB: raw
    for T, want in ((512, O.S_ENCODED), (513, O.S_RAW_OVERSIZE)):
        g = _geom((O.FP8_CAST, O.FP8_CAST), D=256, H=64, T=T, L=1, B=1)
        x = np.zeros(T * 64 * 256, np.uint16)
        seg = O.segment_enc_bytes(g, 0)
        _, st = O.encode(g, [x, x], oracle_descs([(0, 0, 0, 0)]), seg)
        assert st[0] == want, (T, st)


def _layout_restatement(case, arm, layers_bits, rows, enc):
    """Rebuild every ENCODED slot from the per-vector oracle functions and the
    documented slot layout: vectors v = t*H + h; [codes][metadata]; zero pad."""
    D, H, T = case.head_dim, case.num_heads, case.block_tokens
    sb, st, sh = case.strides
    dt = O.FP16 if case.dtype == torch.float16 else O.BF16
    for (layer, blk, role, off) in rows:
        codec = [arm.k_codec, arm.v_codec][role]
        if case.layout == "separate":
            src = layers_bits[2 * layer + role]
            base = blk * sb
        else:
            src = layers_bits[layer]
            base = blk * sb + role * D
        idx = np.array([[base + t * st + h * sh for h in range(H)] for t in range(T)]).reshape(-1)
        x = O.src_to_f32(src[idx[:, None] + np.arange(D)[None, :]], dt)     # [T*H, D]
        if codec == "fp8_dynamic":
            s = np.array([O.fp8_scale_from_amax(O.absmax(v)) for v in x], np.float32)
            body = np.concatenate([O.fp8_encode(x, s).reshape(-1), s.view(np.uint8)])
        elif codec in ("tq2", "tq3", "tq4"):
            bits = int(codec[-1])
            c, n16 = O.tq_encode(x, bits, case.seed)
            body = np.concatenate([np.concatenate([O.pack_bits(r, bits) for r in c]), n16.view(np.uint8)])
        else:
            bits = int(codec[-1])
            c, m16, s16 = O.uniform_encode(x, bits)
            packed = c.reshape(-1) if bits == 8 else np.concatenate([O.pack_bits(r, bits) for r in c])
            body = np.concatenate([packed, np.stack([m16, s16], 1).reshape(-1).view(np.uint8)])
        seg = -(-body.size // 128) * 128
        want = np.zeros(seg, np.uint8)
        want[: body.size] = body
        assert np.array_equal(enc[off: off + seg], want), (layer, blk, role)


@pytest.mark.parametrize("name", ["tiny", "vllm_packed", "qwen3_8b", "qwen25_7b_offload"])
def test_segment_layout_restated(name):
    # 5 layers: with the first and last two protected, layer 2 is the one encoded
    case = synth.make_case(name, num_layers=5 if name in ("vllm_packed", "qwen25_7b_offload") else 1,
                           num_blocks=3)
    bits = [host_bits(t) for t in case.layers]
    for arm in case.arms:
        g = oracle_geom(case, arm)
        segb = [O.segment_enc_bytes(g, r) for r in (0, 1)]
        rows, total = synth.segment_list(case, arm, segb)
        enc, st = O.encode(g, bits, oracle_descs(rows), total)
        for r, s_ in zip(rows, st):
            prot = r[0] < arm.protect[0] or r[0] >= case.num_layers - arm.protect[1]
            if prot:
                assert s_ == O.S_RAW_PROTECTED
            elif name != "vllm_packed":
                assert s_ == O.S_ENCODED
        enc_rows = [r for r, s_ in zip(rows, st) if s_ == O.S_ENCODED]
        assert enc_rows
        _layout_restatement(case, arm, bits, enc_rows, enc)


def test_layout_invariance_separate_vs_packed():
    """The same logical vectors in the separate and the packed layout encode to
    the same bytes (the slot does not depend on the source layout)."""
    case = synth.make_case("tiny", num_blocks=2)
    k, v = case.layers[0].float(), case.layers[1].float()     # [B, T, H, D]
    packed = torch.cat([k, v], dim=-1).permute(0, 2, 1, 3).contiguous().half()   # [B, H, T, 2D]
    for arm in case.arms:
        g_sep = oracle_geom(case, arm)
        pcase = synth.Case("p", torch.float16, "packed", 128, 8, 16, 1, 2,
                           synth._packed_strides(16, 8, 128), [packed], case.arms)
        g_pk = oracle_geom(pcase, arm)
        segb = [O.segment_enc_bytes(g_sep, r) for r in (0, 1)]
        rows, total = synth.segment_list(case, arm, segb)
        e1, s1 = O.encode(g_sep, [host_bits(case.layers[0]), host_bits(case.layers[1])],
                          oracle_descs(rows), total)
        e2, s2 = O.encode(g_pk, [host_bits(packed)], oracle_descs(rows), total)
        assert np.array_equal(s1, s2) and np.array_equal(e1, e2)


def test_decode_restores_only_encoded_segments():
    case = synth.make_case("tiny", num_blocks=3)
    arm = case.arms[1]
    bits = [host_bits(t) for t in case.layers]
    bits[0][5] = 0x7C00     # +inf in block 0 of K
    g = oracle_geom(case, arm)
    segb = [O.segment_enc_bytes(g, r) for r in (0, 1)]
    rows, total = synth.segment_list(case, arm, segb)
    enc, st = O.encode(g, bits, oracle_descs(rows), total)
    assert st[0] == O.S_RAW_NONFINITE and np.all(st[1:] == O.S_ENCODED)
    out = [np.full_like(b, 0x1234) for b in bits]
    res = O.decode(g, out, oracle_descs(rows), enc, st)
    assert list(res) == list(st)
    # the raw K segment of block 0 is untouched; every encoded one is written
    seg_el = 16 * 8 * 128
    assert np.all(out[0][:seg_el] == 0x1234)
    assert not np.any(out[0][seg_el:] == 0x1234) and not np.any(out[1] == 0x1234)
    # restored values are close to the source (4-bit K / V)
    x = O.f16_to_f32(bits[1]).reshape(-1, 128)
    y = O.f16_to_f32(out[1]).reshape(-1, 128)
    assert np.max(np.abs(x - y)) < 0.5


def _exhaustive_case(dtype):
    """All 65,536 16-bit patterns laid out so that every in-range finite value
    sits in admitted segments and the rest in segments of their own."""
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = O.f16_to_f32(allp) if dtype == O.FP16 else O.bf16_to_f32(allp)
    good = allp[np.isfinite(f) & (np.abs(f) <= 448)]
    bad = allp[~(np.isfinite(f) & (np.abs(f) <= 448))]
    D, H, T = 128, 8, 16
    per = D * H * T
    ng = -(-good.size // per)
    buf = np.zeros((ng + bad.size) * per, np.uint16)
    buf[: good.size] = good
    for i, b in enumerate(bad):                 # one out-of-range value per segment
        buf[(ng + i) * per] = b
    return buf, good, bad, ng, ng + bad.size


@pytest.mark.parametrize("dtype", [O.FP16, O.BF16])
def test_fp8_cast_exhaustive_table(dtype):
    buf, good, bad, ng, B = _exhaustive_case(dtype)
    g = _geom((O.FP8_CAST, O.NONE), D=128, H=8, T=16, L=1, B=B, dtype=dtype)
    seg = O.segment_enc_bytes(g, 0)
    rows = [(0, b, 0, b * seg) for b in range(B)]
    enc, st = O.encode(g, [buf, None], oracle_descs(rows), B * seg)
    assert np.all(st[:ng] == O.S_ENCODED)
    f = O.src_to_f32(bad, dtype)
    assert np.array_equal(st[ng:], np.where(np.isfinite(f), O.S_RAW_RANGE, O.S_RAW_NONFINITE))
    codes = enc[: ng * seg][: good.size]
    src = O.src_to_f32(good, dtype)
    ref = torch.from_numpy(src).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


@pytest.mark.parametrize("codecs,want_k,want_v", [
    ((O.TQ4, O.UNI4), ["E", "R", "E", "R"], ["E", "R", "E", "E"]),
    ((O.UNI8, O.UNI8), ["E", "R", "E", "E"], ["E", "R", "E", "E"]),
    ((O.FP8_DYNAMIC, O.INT8), ["E"] * 4, ["E"] * 4)])
def test_fp16_metadata_overflow_stays_raw(codecs, want_k, want_v):
    """Under an admission bound above the FP16 range (here +inf) with BF16
    sources, a TurboQuant norm or a uniform minimum / step beyond +-65504
    cannot be stored: the segment stays raw as out of range.  FP8 (FP32
    scale) and INT8 (BF16 scale) still code it."""
    D, H, T, B = 64, 8, 16, 4                # (H = 8: at H = 2 an INT8 record saves nothing)
    k = np.random.default_rng(3).standard_normal((B, T, H, D)).astype(np.float32)
    k[1, 0, 0, :] = 1e5                                            # norm 8e5, minimum 1e5
    k[2, 3, 1, :] = np.where(np.arange(D) % 2, 6000.0, -6000.0)   # norm 48,000: fits
    k[3, 5, 0, 9] = 70000.0                                        # norm > 65504, step fits
    kb = O.f32_to_bf16(k).reshape(-1)
    g = O.make_geom(dtype=O.BF16, layout=O.SEPARATE, head_dim=D, num_heads=H, block_tokens=T,
                    num_layers=1, num_blocks=B, strides=(T * H * D, H * D, D), codecs=codecs,
                    seed=1, reject_abs=np.inf)
    seg = [O.segment_enc_bytes(g, r) for r in (0, 1)]
    rows, off = [], 0
    for b in range(B):
        for r in (0, 1):
            rows.append((0, b, r, off))
            off += seg[r]
    _, st = O.encode(g, [kb, kb.copy()], oracle_descs(rows), off)
    code = {"E": O.S_ENCODED, "R": O.S_RAW_RANGE}
    assert list(st[0::2]) == [code[c] for c in want_k]
    assert list(st[1::2]) == [code[c] for c in want_v]
