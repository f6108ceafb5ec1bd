"""GPU parity of the one-call integrity paths (OrbitKV docs, "KV precision and
storage encoding", section "Ownership, storage and GDS": a CRC32 per stored
segment, checked before GPU decode; a damaged object becomes a miss).

kv_codec_encode_sealed must give the statuses, slots and headers of encode
followed by seal, and kv_codec_decode_verified the results and pages of verify
followed by decode, bit for bit against the oracle.  FP8, uniform-8 and HiQ
INT8 roles take the one-pass kernels (the warp that codes a slot also
checksums it); the other codecs take encode + seal and verify + decode,
covered here too."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_parity import run_sealed_parity
from kv_cache_page_gb300 import synth
from kvcases import custom_case

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)


def _dt(kv, default):
    """INT8_HEAD is defined for BF16 sources only."""
    return "bf16" if "int8" in kv else default


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_page_gb300 import build
    build.build()


CASES = [("tiny", 0, {}), ("tiny", 1, {}), ("qwen3_8b", 0, dict(num_layers=2, num_blocks=8)),
         ("qwen3_8b", 1, dict(num_layers=3, num_blocks=8)), ("vllm_packed", 0, dict(num_layers=5, num_blocks=6)),
         ("hiq_qwen3_8b", 0, dict(num_layers=2, num_blocks=8)),
         ("qwen25_7b_offload", 0, dict(num_layers=5, num_blocks=8)),
         ("head_dim_sweep", 0, dict(head_dim=32, num_blocks=4)),
         ("head_dim_sweep", 0, dict(head_dim=256, num_blocks=4))]


@pytest.mark.parametrize("name,arm_i,kw", CASES)
def test_sealed_and_verified_match_oracle(name, arm_i, kw):
    case = synth.make_case(name, **kw)
    st, res = run_sealed_parity(case, case.arms[arm_i], tamper=5, seed=len(name) + arm_i)
    assert np.any(st == O.S_ENCODED)
    assert np.count_nonzero(res == O.S_CORRUPT) == 5


@pytest.mark.parametrize("k,v", [("fp8_dynamic", "fp8_cast"), ("fp8_fixed", "fp8_dynamic"),
                                 ("fp8_cast", "none"), ("none", "fp8_fixed"), ("fp8_dynamic", "uni3"),
                                 ("none", "none"), ("uni8", "uni8"), ("fp8_dynamic", "uni8"),
                                 ("uni8", "fp8_fixed"), ("none", "uni8"), ("uni8", "uni4"),
                                 ("int8", "int8"), ("int8", "fp8_dynamic"), ("uni8", "int8"),
                                 ("none", "int8"), ("int8", "uni4")])
@pytest.mark.parametrize("D", [32, 64, 128, 256])
def test_role_mixes(k, v, D):
    """Two FP8 kinds (one launch per role), FP8 beside no codec, uniform-8 and
    INT8 alone, beside another one-pass codec (two one-pass launches) and
    beside no codec, a one-pass codec beside another family (the two-pass
    route) and no codec at all."""
    case = custom_case(D=D, H=3, T=5, L=3, B=4, dtype=_dt((k, v), "bf16" if D % 64 else "fp16"),
                       layout="packed" if D == 64 else "separate", seed=D)
    run_sealed_parity(case, synth.Arm("mix", k, v, (0, 1)), tamper=3 if (k, v) != ("none", "none") else 0)


@pytest.mark.parametrize("kv", [("fp8_dynamic", "fp8_fixed"), ("uni8", "uni8"), ("int8", "int8")])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("layout", ["separate", "packed"])
def test_full_pages_take_the_adjacent_chunk_decoder(D, layout, kv):
    """Segments of 512 vectors: the verifying decoder's adjacent-chunk mapping."""
    case = custom_case(D=D, H=16, T=32, L=2, B=3, dtype="bf16", layout=layout, seed=D + 7)
    run_sealed_parity(case, synth.Arm("full", kv[0], kv[1], (0, 1)), tamper=4)


@pytest.mark.parametrize("codec", ["fp8_dynamic", "uni8", "int8"])
def test_planted_nonfinite_range_and_protected_layers(codec):
    case = custom_case(D=128, H=4, T=16, L=4, B=4, dtype=_dt((codec,), "fp16"), layout="separate", seed=11)
    case.layers[2][1, 3, 2, 5] = float("inf")
    case.layers[3][2, 0, 0, 9] = float("nan")
    case.layers[4][3, 7, 1, 2] = -600.0
    case.layers[5][0, 4, 3, 100] = 448.0
    st, res = run_sealed_parity(case, synth.Arm("pl", codec, codec, (0, 1), (1, 0)), tamper=2)
    for s in (O.S_RAW_NONFINITE, O.S_RAW_RANGE, O.S_RAW_PROTECTED):
        assert np.any(st == s)
    # raw segments come back from verify with their status and stay unrestored
    raw = st != O.S_ENCODED
    assert np.array_equal(res[raw], st[raw])


@pytest.mark.parametrize("seed", range(8))
def test_descriptor_fuzz(seed):
    """Invalid descriptors (layer, block, role, misaligned or out-of-range slot)
    among valid ones, shuffled, a page coded into several slots."""
    rng = np.random.default_rng(100 + seed)
    kc, vc = [("fp8_dynamic", "fp8_dynamic"), ("fp8_fixed", "fp8_cast"), ("fp8_dynamic", "none"),
              ("tq3", "fp8_cast"), ("uni8", "uni8"), ("uni8", "fp8_dynamic"), ("int8", "int8"),
              ("fp8_fixed", "int8")][seed]
    case = custom_case(D=int(rng.choice([32, 64, 128])), H=int(rng.integers(1, 9)), T=16, L=3, B=4,
                       dtype=_dt((kc, vc), "bf16" if seed % 2 else "fp16"),
                       layout="packed" if seed % 2 else "separate",
                       values="heavy", seed=seed)
    arm = synth.Arm("fz", kc, vc, (0, 1), (1, 0) if seed % 2 else (0, 0))
    from gpu_parity import make_codec
    c = make_codec(case, arm)
    slot = max([c.segment_bytes(r)[0] for r in (0, 1)] + [128])
    c.close()
    n = 48
    rows = []
    for k in range(n):
        layer, blk, role = int(rng.integers(0, 3)), int(rng.integers(0, 4)), int(rng.integers(0, 2))
        off = k * slot
        kind = rng.random()
        if kind < 0.08:
            layer = 3 + int(rng.integers(0, 5))
        elif kind < 0.14:
            blk = 4 + int(rng.integers(0, 3))
        elif kind < 0.18:
            role = 2
        elif kind < 0.22:
            off += 8
        elif kind < 0.26:
            off = (n + 5) * slot
        rows.append((layer, blk, role, off))
    st, _ = run_sealed_parity(case, arm, rows=rows, total=n * slot, tamper=3, seed=seed)
    assert np.any(st == O.S_BAD_DESC) and np.any(st == O.S_ENCODED)


def test_host_resident_buffers():
    """Descriptors, slots, statuses, headers and results in pinned host memory."""
    case = synth.make_case("qwen3_8b", num_layers=2, num_blocks=4)
    run_sealed_parity(case, case.arms[1], buffers="host", tamper=2)


def test_format_version_2_headers():
    case = synth.make_case("tiny")
    run_sealed_parity(case, case.arms[0], sign_version=2, tamper=2)
    run_sealed_parity(case, case.arms[1], sign_version=2, tamper=2)


@pytest.mark.parametrize("kv", [("fp8_dynamic", "fp8_fixed"), ("uni8", "uni8"), ("int8", "int8")])
@pytest.mark.parametrize("T,coded", [(512, True), (513, False)])
def test_maximum_segment_size(T, coded, kv):
    """A 16 MiB source segment (64 heads x 512 tokens x 256 dims, 16-bit) is
    sealed and verified in one pass by a single warp; one token more and it
    stays raw (OVERSIZE), its header saying so."""
    case = custom_case(D=256, H=64, T=T, L=1, B=1, dtype=_dt(kv, "fp16"), layout="separate")
    st, res = run_sealed_parity(case, synth.Arm("max", kv[0], kv[1], (0, 1)),
                                tamper=1 if coded else 0)
    want = O.S_ENCODED if coded else O.S_RAW_OVERSIZE
    assert list(st) == [want, want]
    if coded:
        assert sorted(res.tolist()) == [O.S_ENCODED, O.S_CORRUPT]


@pytest.mark.parametrize("kv", [("fp8_dynamic", "fp8_cast"), ("uni8", "uni8"), ("int8", "int8")])
def test_every_16bit_pattern(kv):
    """All 65,536 16-bit patterns (FP16; BF16 for INT8) through the sealing
    encoder and the verifying decoder: in-range values fill admitted pages,
    each nonfinite or out-of-range pattern sits alone in a page of its own
    (raw, header status included)."""
    bf = "int8" in kv
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = O.src_to_f32(allp, O.BF16 if bf else O.FP16)
    ok = np.isfinite(f) & (np.abs(f) <= 448)
    good, bad = allp[ok], allp[~ok]
    per = 128 * 8 * 16
    ng = -(-good.size // per)
    buf = np.zeros((ng + bad.size) * per, np.uint16)
    buf[: good.size] = good
    for i, b in enumerate(bad):
        buf[(ng + i) * per + 37] = b
    B = ng + bad.size
    tdt = torch.bfloat16 if bf else torch.float16
    t = torch.from_numpy(buf.view(np.int16)).view(tdt).reshape(B, 16, 8, 128)
    case = synth.Case("all16", tdt, "separate", 128, 8, 16, 1, B,
                      synth._separate_strides(16, 8, 128), [t, t.clone()], [], 0, torch.ones(1, 2))
    st, res = run_sealed_parity(case, synth.Arm("all", kv[0], kv[1], (0, 1)), tamper=4)
    assert np.any(st == O.S_ENCODED) and np.any(st == O.S_RAW_NONFINITE) and np.any(st == O.S_RAW_RANGE)


@pytest.mark.parametrize("kv", [("int8", "int8"), ("uni8", "uni8")])
@pytest.mark.parametrize("D", [32, 256])
@pytest.mark.parametrize("H,T", [(1, 37), (2, 9), (5, 7)])
def test_record_and_step_geometries(kv, D, H, T):
    """Few heads per token: INT8 records complete faster than one CRC row per
    step at H = 1 (the in-loop folding lags and the final rows catch up), and
    record padding takes 2-, 4- and 16-byte stores; uniform-8 segments of one
    warp step or less take the warp-per-segment encoder."""
    case = custom_case(D=D, H=H, T=T, L=2, B=5, dtype="bf16", layout="separate", seed=D + H)
    run_sealed_parity(case, synth.Arm("geo", kv[0], kv[1], (0, 1)), tamper=2, seed=H)
