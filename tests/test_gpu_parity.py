"""GPU parity: the CUDA codec (through the C ABI) against the oracle, element by
element, on the same seeded inputs.

Rules (from the benchmark spec's tolerances): FP8 codes and scales, TurboQuant and
uniform codes, metadata, padding and every segment status bit-exact; restored
pages within 1 ulp of the 16-bit format (+-0 equal).
"""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_parity import run_parity
from kvcases import custom_case
from kv_cache_page_gb300 import synth

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_page_gb300 import build
    build.build()


ALL_CODECS = [("fp8_cast", "fp8_cast"), ("fp8_fixed", "fp8_fixed"), ("fp8_dynamic", "fp8_dynamic"),
              ("tq3", "uni3"), ("tq4", "uni4"), ("uni8", "uni8"), ("uni3", "uni4"), ("none", "fp8_dynamic"),
              ("tq4", "none"), ("tq2", "uni2"), ("uni2", "uni8")]


@pytest.mark.parametrize("name", ["tiny"])
def test_tiny_full_config(name):
    case = synth.make_case(name)
    for arm in case.arms:
        st, ulps = run_parity(case, arm)
        assert np.all(st == O.S_ENCODED)
        assert ulps == 0


def test_qwen3_8b_shape_small():
    case = synth.make_case("qwen3_8b", num_layers=2, num_blocks=24)
    for arm in case.arms:
        st, ulps = run_parity(case, arm)
        assert np.all(st == O.S_ENCODED) and ulps == 0


def test_vllm_packed_tq3_with_raw_segments():
    case = synth.make_case("vllm_packed", num_layers=6, num_blocks=40)
    st, ulps = run_parity(case, case.arms[0])
    assert np.count_nonzero(st == O.S_RAW_PROTECTED) == 4 * 40 * 2
    assert ulps == 0


def test_vllm_packed_planted_nonfinite_and_range():
    case = synth.make_case("vllm_packed", num_layers=5, num_blocks=6)
    case.arms[0].protect = (0, 0)
    L0 = case.layers[2]
    L0[1, 3, 7, 5] = float("inf")            # K of block 1
    L0[2, 0, 0, 128 + 9] = float("nan")      # V of block 2
    L0[3, 7, 15, 2] = -600.0                 # K of block 3
    L0[4, 4, 4, 200] = 448.0                 # on the bound: admitted
    st, ulps = run_parity(case, case.arms[0])
    rows = synth.segment_list(case, case.arms[0], [1, 1])[0]
    want = {(2, 1, 0): O.S_RAW_NONFINITE, (2, 2, 1): O.S_RAW_NONFINITE, (2, 3, 0): O.S_RAW_RANGE}
    for (l, b, r, _), s in zip(rows, st):
        if (l, b, r) in want:
            assert s == want[(l, b, r)]
    assert ulps == 0


@pytest.mark.parametrize("D", [32, 64, 128, 256])
def test_head_dim_sweep(D):
    case = synth.make_case("head_dim_sweep", head_dim=D, num_blocks=6)
    for arm in case.arms:
        st, ulps = run_parity(case, arm)
        assert np.all(st == O.S_ENCODED) and ulps == 0


def test_large_offload_shape_small():
    case = synth.make_case("qwen25_7b_offload", num_layers=5, num_blocks=12)
    st, ulps = run_parity(case, case.arms[0])
    assert ulps == 0


@pytest.mark.parametrize("kc,vc", ALL_CODECS)
@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("layout", ["separate", "packed"])
def test_codec_matrix(kc, vc, D, dtype, layout):
    # ragged segment (H=3, T=5: 15 vectors, not a multiple of any warp tile)
    case = custom_case(D=D, H=3, T=5, L=2, B=5, dtype=dtype, layout=layout,
                       values="heavy" if dtype == "bf16" else "normal", seed=D)
    arm = synth.Arm("m", kc, vc, (0, 1))
    st, ulps = run_parity(case, arm)
    assert ulps == 0


@pytest.mark.parametrize("kc,vc", [("tq4", "uni4"), ("tq3", "uni3"), ("tq2", "uni2"),
                                   ("fp8_dynamic", "uni8"), ("int8", "int8")])
@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("layout", ["separate", "packed"])
@pytest.mark.parametrize("offset", [16, 32])
def test_layer_pointers_16_and_32_byte_aligned(kc, vc, D, layout, offset):
    """Layer tensors 16 bytes past a 32-byte boundary (the library requires
    16-byte alignment; kernels that move 32 bytes per access take their
    16-byte path) and 32 bytes past a 256-byte one (the 32-byte path)."""
    case = custom_case(D=D, H=8, T=16, L=2, B=4, dtype="bf16", layout=layout, seed=D + offset)
    st, ulps = run_parity(case, synth.Arm("a", kc, vc, (0, 1)), layer_offset=offset)
    assert ulps == 0 and np.all(st == O.S_ENCODED)


@pytest.mark.parametrize("kc,vc", [("fp8_dynamic", "uni8"), ("fp8_fixed", "uni4"), ("fp8_cast", "uni2"),
                                   ("tq3", "uni3")])
@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("offset", [16, 32])
def test_large_ragged_segments(kc, vc, D, dtype, offset):
    """Segments of 272 vectors (17 heads x 16 tokens): the decoders' mapping
    for segments of 256+ vectors, with a ragged last step, on layer pointers
    16 bytes (16-byte stores) and 32 bytes (32-byte stores) past an aligned
    allocation."""
    case = custom_case(D=D, H=17, T=16, L=1, B=3, dtype=dtype, layout="separate", seed=D + offset)
    st, ulps = run_parity(case, synth.Arm("big", kc, vc, (0, 1)), layer_offset=offset)
    assert ulps == 0 and np.all(st == O.S_ENCODED)


@pytest.mark.parametrize("kc,vc", [("int8", "int8"), ("int8", "fp8_dynamic"), ("tq4", "int8"),
                                   ("none", "int8")])
@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("H,T", [(3, 5), (8, 16), (1, 3)])
@pytest.mark.parametrize("layout", ["separate", "packed"])
def test_int8_head_matrix(kc, vc, D, H, T, layout):
    """Symmetric per-head INT8 in token-row records (BF16 only), ragged and
    page-shaped segments, both layouts, mixed with the other codecs."""
    case = custom_case(D=D, H=H, T=T, L=2, B=4, dtype="bf16", layout=layout,
                       values="heavy" if H == 3 else "normal", seed=D + H)
    st, ulps = run_parity(case, synth.Arm("i8", kc, vc, (0, 1)))
    assert ulps == 0


def test_int8_every_bf16_maximum():
    """Every positive BF16 value up to 448 as the maximum of its own head vector
    (the rest of the vector spread below it): every scale the encoder can form
    and the largest quotients, against the oracle."""
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint16)
    a = O.bf16_to_f32(bits)
    a = a[a <= 448.0]
    D, H, T = 64, 8, 16
    per = H * T
    B = -(-a.size // per)
    rng = np.random.default_rng(7)
    x = np.zeros((B * per, D), np.float32)
    x[:a.size, 0] = np.where(np.arange(a.size) % 2 == 0, a, -a)
    x[:a.size, 1:] = a[:, None] * rng.uniform(-1, 1, (a.size, D - 1)).astype(np.float32)
    t = torch.from_numpy(x.reshape(B, T, H, D)).bfloat16()
    case = synth.Case("maxima", torch.bfloat16, "separate", D, H, T, 1, B,
                      synth._separate_strides(T, H, D), [t, t.clone()], [], 0)
    st, ulps = run_parity(case, synth.Arm("m", "int8", "int8", (0, 1)))
    assert np.all(st == O.S_ENCODED) and ulps == 0


def test_hiq_qwen3_8b_shape_small():
    case = synth.make_case("hiq_qwen3_8b", num_layers=2, num_blocks=24)
    for arm in case.arms:
        st, ulps = run_parity(case, arm)
        assert np.all(st == O.S_ENCODED) and ulps == 0


def test_int8_special_values():
    """BF16 zeros of both signs, an all-zero head (the maximum floor), heads
    below the floor, powers of two, +-448 exactly, and a planted NaN and 452.
    (H = 8: at H = 2 a 64-wide head's record pads to 256 bytes and saves nothing.)"""
    D, H, T = 64, 8, 16
    x = torch.zeros(8, T, H, D, dtype=torch.float32)
    x[1] = -0.0
    x[2, :, :, ::2] = -0.0
    x[3] = 1e-14 * torch.arange(D)                                  # below the 1e-12 floor
    x[4] = torch.tensor(2.0) ** torch.arange(-60, -60 + D).float()  # one octave per element
    x[5, :, 0, 0], x[5, :, 1, 1] = 448.0, -448.0
    x[6, 3, 1, 9] = float("nan")
    x[7, 0, 0, 0] = 452.0                                           # BF16(449) is 448
    t = x.bfloat16()
    case = synth.Case("special8", torch.bfloat16, "separate", D, H, T, 1, 8,
                      synth._separate_strides(T, H, D), [t, t.clone()], [], 0)
    st, ulps = run_parity(case, synth.Arm("s", "int8", "int8", (0, 1)))
    assert list(st[:12]) == [O.S_ENCODED] * 12
    assert list(st[12:]) == [O.S_RAW_NONFINITE, O.S_RAW_NONFINITE, O.S_RAW_RANGE, O.S_RAW_RANGE]
    assert ulps == 0


@pytest.mark.parametrize("kc,vc", [("tq4", "fp8_dynamic"), ("tq3", "uni8")])
def test_large_segments_many_steps(kc, vc):
    case = custom_case(D=128, H=32, T=16, L=1, B=3, dtype="fp16", layout="separate")
    st, ulps = run_parity(case, synth.Arm("big", kc, vc, (0, 1)))
    assert np.all(st == O.S_ENCODED) and ulps == 0


@pytest.mark.parametrize("T,coded", [(512, True), (513, False)])
def test_maximum_segment_size(T, coded):
    """A segment of exactly 16 MiB of source (64 heads x 512 tokens x 256 dims,
    FP16) is coded; one token more and it stays raw (OVERSIZE), for both roles."""
    case = custom_case(D=256, H=64, T=T, L=1, B=1, dtype="fp16", layout="separate")
    st, ulps = run_parity(case, synth.Arm("max", "fp8_dynamic", "uni8", (0, 1)))
    want = O.S_ENCODED if coded else O.S_RAW_OVERSIZE
    assert list(st) == [want, want] and ulps == 0


def _exhaustive_layers(dtype):
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = O.src_to_f32(allp, dtype)
    ok = np.isfinite(f) & (np.abs(f) <= 448)
    good, bad = allp[ok], allp[~ok]
    per = 128 * 8 * 16
    ng = -(-good.size // per)
    buf = np.zeros((ng + bad.size) * per, np.uint16)
    buf[: good.size] = good
    for i, b in enumerate(bad):
        buf[(ng + i) * per + 37] = b
    return buf, ng + bad.size


@pytest.mark.parametrize("dtype,codec", [(d, c) for d in ("fp16", "bf16")
                                         for c in ("fp8_cast", "fp8_dynamic", "uni8", "tq4", "tq2")]
                         + [("bf16", "int8")])
def test_every_16bit_pattern(dtype, codec):
    """All 65,536 source patterns: in-range finite values fill admitted pages, each
    nonfinite / out-of-range pattern sits alone in a page of its own."""
    odt = O.FP16 if dtype == "fp16" else O.BF16
    buf, B = _exhaustive_layers(odt)
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    t = torch.from_numpy(buf.view(np.int16)).view(tdt).reshape(B, 16, 8, 128)
    case = synth.Case("exh", tdt, "separate", 128, 8, 16, 1, B, synth._separate_strides(16, 8, 128),
                      [t, t.clone()], [], 0)
    vc = {"tq4": "uni4", "tq2": "uni2"}.get(codec, codec)
    st, ulps = run_parity(case, synth.Arm("exh", codec, vc, (0,)))
    f = O.src_to_f32(buf.reshape(B, -1), odt)
    bad_page = ~np.all(np.isfinite(f) & (np.abs(f) <= 448), axis=1)
    assert np.array_equal(st != O.S_ENCODED, bad_page)
    assert ulps == 0


@pytest.mark.parametrize("reject", [1.5, 3.0, 448.0])
def test_admission_at_the_bound(reject):
    """Every block holds a vector whose largest |x| is exactly reject_abs
    (admitted); odd blocks also hold one element at the next BF16 value above
    it (raw, out of range).  The vectors' norms exceed the bound, so the
    encoders' exact check runs on admitted and rejected vectors alike."""
    D, H, T, B = 128, 8, 16, 6
    g = torch.Generator().manual_seed(int(reject * 16))
    x = ((torch.rand(B, T, H, D, generator=g) * 2 - 1) * reject).bfloat16().float()
    x[:, 0, 0, 0] = reject
    x[:, 2, 5, 1] = -reject
    above = torch.tensor([reject], dtype=torch.bfloat16).view(torch.int16) + 1
    x[1::2, 5, 3, 7] = above.view(torch.bfloat16).float().item()
    t = x.bfloat16()
    case = synth.Case("bound", torch.bfloat16, "separate", D, H, T, 1, B,
                      synth._separate_strides(T, H, D), [t, t.clone()], [], 0)
    for kc, vc in [("tq4", "uni4"), ("tq3", "uni3"), ("tq2", "uni2"), ("fp8_dynamic", "int8")]:
        st, ulps = run_parity(case, synth.Arm("b", kc, vc, (0, 1)), reject_abs=reject)
        want = [O.S_RAW_RANGE if b % 2 else O.S_ENCODED for b in range(B) for _ in (0, 1)]
        assert list(st) == want and ulps == 0, (kc, vc)


def test_special_values():
    """Zeros of both signs, constant vectors, FP16 subnormals, +-448 exactly."""
    D, H, T = 64, 2, 16
    x = torch.zeros(6, T, H, D, dtype=torch.float32)
    x[1] = -0.0
    x[2, :, :, ::2] = -0.0
    x[3] = 1.375
    x[4] = torch.tensor(2.0**-24) * torch.arange(D)            # subnormal ramp
    x[5, :, 0, 0], x[5, :, 1, 1] = 448.0, -448.0
    t = x.half()
    case = synth.Case("special", torch.float16, "separate", D, H, T, 1, 6,
                      synth._separate_strides(T, H, D), [t, t.clone()], [], 0, torch.ones(1, 2))
    for kc, vc in ALL_CODECS[:6]:
        st, ulps = run_parity(case, synth.Arm("s", kc, vc, (0, 1)))
        assert np.all(st == O.S_ENCODED) and ulps == 0


def test_descriptor_edge_cases():
    case = custom_case(D=64, H=2, T=16, L=4, B=3, dtype="fp16", layout="separate")
    arm = synth.Arm("e", "tq4", "uni4", (0, 1), protect=(1, 1))
    # slots: K (TQ4) 32 x 34 = 1088 -> 1152 bytes, V (uniform-4) 32 x 36 = 1152 bytes
    rows = [(1, 0, 0, 0), (1, 1, 1, 1152), (0, 0, 0, 2304),     # layer 0 protected
            (3, 2, 1, 3456),                                      # layer 3 protected
            (4, 0, 0, 4608),                                      # layer out of range
            (2, 3, 0, 4608),                                      # block out of range
            (2, 0, 2, 4608),                                      # bad role
            (2, 0, 0, 4616),                                      # misaligned slot
            (2, 0, 0, 1 << 40),                                   # slot past the buffer
            (2, 2, 1, 4608)]
    st, _ = run_parity(case, arm, rows=rows, total=5 * 1152)
    assert list(st) == [O.S_ENCODED, O.S_ENCODED, O.S_RAW_PROTECTED, O.S_RAW_PROTECTED,
                        O.S_BAD_DESC, O.S_BAD_DESC, O.S_BAD_DESC, O.S_BAD_DESC, O.S_BAD_DESC,
                        O.S_ENCODED]


@pytest.mark.parametrize("seed", range(6))
def test_descriptor_fuzz(seed):
    """Seeded random descriptor lists: shuffled order, a source page coded into
    several slots, and invalid entries (layer, block, role, misaligned or
    out-of-range offsets) mixed in.  Statuses, slots and restores against the
    oracle; an invalid descriptor must not disturb its neighbours."""
    rng = np.random.default_rng(seed)
    kc, vc = [("fp8_dynamic", "uni4"), ("tq3", "fp8_cast"), ("uni8", "uni3"), ("tq4", "none"),
              ("fp8_fixed", "fp8_dynamic"), ("uni2", "tq2_k_only")][seed]
    if vc == "tq2_k_only":
        kc, vc = "tq2", "uni2"
    case = custom_case(D=int(rng.choice([32, 64, 128])), H=int(rng.integers(1, 9)), T=16, L=3, B=4,
                       dtype="bf16" if seed % 2 else "fp16", layout="packed" if seed % 3 == 0 else "separate",
                       values="heavy" if seed % 2 else "normal", seed=seed)
    arm = synth.Arm("fz", kc, vc, (0, 1), (1, 0) if seed % 2 else (0, 0))
    from gpu_parity import make_codec
    c = make_codec(case, arm)
    seg = [c.segment_bytes(r)[0] for r in (0, 1)]
    c.close()
    slot = max(seg + [128])
    n = 40
    rows = []
    for k in range(n):
        layer, blk, role = int(rng.integers(0, 3)), int(rng.integers(0, 4)), int(rng.integers(0, 2))
        off = k * slot
        kind = rng.random()
        if kind < 0.08:
            layer = 3 + int(rng.integers(0, 5))          # layer out of range
        elif kind < 0.14:
            blk = 4 + int(rng.integers(0, 3))            # block out of range
        elif kind < 0.18:
            role = 2                                     # bad role
        elif kind < 0.22:
            off += 8                                     # misaligned slot
        elif kind < 0.26:
            off = (n + 5) * slot                         # slot past the buffer
        rows.append((layer, blk, role, off))
    st, ulps = run_parity(case, arm, rows=rows, total=n * slot)
    assert ulps == 0
    assert np.any(st == O.S_BAD_DESC) and np.any(st == O.S_ENCODED)


def test_no_codec_for_either_role_reports_policy():
    case = custom_case(D=32, H=2, T=4, L=2, B=2, dtype="bf16", layout="packed")
    st, _ = run_parity(case, synth.Arm("n", "none", "none", (0, 1)))
    assert np.all(st == O.S_RAW_POLICY)


def test_empty_call_is_a_no_op():
    from kv_cache_page_gb300 import codec as K
    case = synth.make_case("tiny")
    from gpu_parity import make_codec
    c = make_codec(case, case.arms[0])
    c.encode([t.cuda() for t in case.layers], 0, 0, 0, 0, 0)
    c.decode([t.cuda() for t in case.layers], 0, 0, 0, 0, 0)
    torch.cuda.synchronize()
    c.close()


def test_repeat_calls_are_deterministic():
    case = synth.make_case("tiny")
    for arm in case.arms:
        a, _ = run_parity(case, arm)
        b, _ = run_parity(case, arm)
        assert np.array_equal(a, b)


@pytest.mark.parametrize("kc,vc", [("tq4", "uni4"), ("tq3", "uni3"), ("tq2", "uni2")])
@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("layout", ["separate", "packed"])
def test_per_layer_signs(kc, vc, D, dtype, layout):
    """Format version 2: every layer codes K with its own sign vector (the
    kernels generate the layer's words from the seed); 6 layers, ragged
    segments (H=3, T=11), several segments per warp and layer changes between
    them."""
    case = custom_case(D=D, H=3, T=11, L=6, B=7, dtype=dtype, layout=layout,
                       values="heavy" if dtype == "bf16" else "normal", seed=D + 1)
    arm = synth.Arm("v2", kc, vc, (0, 1))
    st, ulps = run_parity(case, arm, sign_version=2)
    assert np.all(st == O.S_ENCODED) and ulps == 0


@pytest.mark.parametrize("D", [64, 128])
def test_per_layer_signs_full_pages(D):
    """Format version 2 on whole 16-token pages of 8 heads across 36 layers."""
    case = custom_case(D=D, H=8, T=16, L=36, B=3, dtype="fp16", layout="separate", seed=5)
    for kc, vc in (("tq4", "uni4"), ("tq3", "none")):
        st, ulps = run_parity(case, synth.Arm("v2", kc, vc, (0, 1) if vc != "none" else (0,)),
                              sign_version=2)
        assert np.all(st == O.S_ENCODED) and ulps == 0


def _calibrate_around_data(case):
    """Calibration maxima per (layer, role) set against the data: layer 0 half
    the largest |x| (most segments' quotients exceed 448), layer 1 above it
    (none do), the rest at the median of the pages' maxima (about half do)."""
    amax = torch.zeros(case.num_layers, 2)
    for l in range(case.num_layers):
        for r in range(2):
            t = case.layers[2 * l + r] if case.layout == "separate" else \
                case.layers[l][..., r * case.head_dim:(r + 1) * case.head_dim]
            per_page = t.float().abs().flatten(1).amax(dim=1)
            amax[l, r] = {0: 0.5 * per_page.max(), 1: 1.01 * per_page.max()}.get(l, per_page.median())
    case.fixed_amax = amax


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("dtype,layout", [("fp16", "separate"), ("bf16", "packed")])
def test_fixed_overflow_reject(D, dtype, layout):
    """FP8 fixed scales below the data's range ("KV precision and storage
    encoding", "FP8 and TurboQuant": out-of-range values stay raw rather than
    being clipped).  Under reject, a segment with a quotient beyond +-448 is
    RAW_RANGE and the others encode, statuses and slots bit-exact against the
    oracle; under the default clip every segment encodes."""
    case = custom_case(D=D, H=4, T=16, L=4, B=8, dtype=dtype, layout=layout, seed=D + 3)
    _calibrate_around_data(case)
    arm = synth.Arm("fx", "fp8_fixed", "fp8_fixed", (0, 1))
    st, ulps = run_parity(case, arm, fixed_overflow="reject")
    assert ulps == 0
    assert np.any(st == O.S_RAW_RANGE) and np.any(st == O.S_ENCODED)
    st_clip, ulps = run_parity(case, arm)
    assert ulps == 0 and np.all(st_clip == O.S_ENCODED)


def test_fixed_overflow_reject_sealed():
    """The same through the one-pass sealing encoder and verifying decoder."""
    from gpu_parity import run_sealed_parity
    case = custom_case(D=128, H=8, T=16, L=4, B=8, dtype="fp16", layout="separate", seed=77)
    _calibrate_around_data(case)
    st, res = run_sealed_parity(case, synth.Arm("fx", "fp8_fixed", "fp8_dynamic", (0, 1)),
                                fixed_overflow="reject", tamper=2)
    assert np.any(st == O.S_RAW_RANGE) and np.any(st == O.S_ENCODED)
