"""GPU parity of segment sealing and verification (OrbitKV docs, section
"Ownership, storage and GDS": version, original length, format, stored length
and CRC32 per encoded segment, validated on the GPU before decode; a damaged
object becomes a miss).  Headers and results bit-exact against the oracle on
the same slots, including slots and headers tampered with on the host."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_parity import SENTINEL_PAGE, make_codec, run_seal_parity
from kv_cache_page_gb300 import codec as K
from kv_cache_page_gb300 import synth
from kvcases import host_bits, oracle_descs, oracle_geom

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_page_gb300 import build
    build.build()


def _encode(case, arm):
    codec = make_codec(case, arm)
    seg = [codec.segment_bytes(r)[0] for r in (0, 1)]
    rows, total = synth.segment_list(case, arm, seg)
    n = len(rows)
    layers = [t.cuda() for t in case.layers]
    descs = K.descriptors(rows, "cuda")
    enc = torch.zeros(max(total, 16), dtype=torch.uint8, device="cuda")
    st = torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda")
    codec.encode(layers, descs, n, enc, total, st)
    torch.cuda.synchronize()
    return codec, rows, total, layers, descs, enc, st


def _headers(n, where="cuda"):
    h = torch.full((max(n, 1) * 32,), 0xEE, dtype=torch.uint8)
    return h.pin_memory() if where == "host" else h.to(where)


def _as_headers(t, n):
    return t.cpu().numpy()[: 32 * n].view(O.HEADER_DTYPE)


CASES = [("tiny", 0, {}), ("tiny", 1, {}), ("vllm_packed", 0, dict(num_layers=5, num_blocks=6)),
         ("qwen3_8b", 0, dict(num_layers=2, num_blocks=8)), ("hiq_qwen3_8b", 0, dict(num_layers=2, num_blocks=8)),
         ("qwen25_7b_offload", 0, dict(num_layers=5, num_blocks=8)),
         ("head_dim_sweep", 1, dict(head_dim=32, num_blocks=4)),
         ("head_dim_sweep", 0, dict(head_dim=256, num_blocks=4))]


@pytest.mark.parametrize("name,arm_i,kw", CASES)
def test_seal_and_verify_match_oracle(name, arm_i, kw):
    case = synth.make_case(name, **kw)
    arm = case.arms[arm_i]
    codec, rows, total, layers, descs, enc, st = _encode(case, arm)
    n = len(rows)
    g = oracle_geom(case, arm)
    enc_h, st_h = enc.cpu().numpy()[:max(total, 16)], st.cpu().numpy()[:n]
    d = oracle_descs(rows)
    hdr = _headers(n)
    codec.seal(descs, n, enc, total, st, hdr)
    torch.cuda.synchronize()
    want = O.seal(g, d, enc_h[:total], st_h)
    got = _as_headers(hdr, n)
    assert np.array_equal(got.view(np.uint8), want.view(np.uint8))
    res = torch.full((n,), 0xEE, dtype=torch.uint8, device="cuda")
    codec.verify(descs, n, enc, total, hdr, res)
    torch.cuda.synchronize()
    assert np.array_equal(res.cpu().numpy(), O.verify(g, d, enc_h[:total], want))
    assert np.array_equal(res.cpu().numpy(), st_h)
    codec.close()


@pytest.mark.parametrize("k,v,H,T,D", [("fp8_dynamic", "uni3", 3, 5, 64), ("tq3", "uni4", 1, 7, 32),
                                       ("int8", "int8", 32, 16, 256), ("uni8", "fp8_cast", 5, 16, 128)])
def test_slot_sizes_off_the_512_byte_row(k, v, H, T, D):
    """Slots of 128 * odd sizes exercise the front padding of the warp's rows."""
    dt = torch.bfloat16 if "int8" in (k, v) else torch.float16
    g = torch.Generator().manual_seed(H * T)
    layers = [torch.randn(3, T, H, D, generator=g).to(dt) for _ in range(4)]
    case = synth.Case("sz", dt, "separate", D, H, T, 2, 3, synth._separate_strides(T, H, D), layers, [],
                      0, torch.ones(2, 2))
    arm = synth.Arm("sz", k, v, (0, 1))
    codec, rows, total, _, descs, enc, st = _encode(case, arm)
    n = len(rows)
    hdr = _headers(n)
    codec.seal(descs, n, enc, total, st, hdr)
    torch.cuda.synchronize()
    want = O.seal(oracle_geom(case, arm), oracle_descs(rows), enc.cpu().numpy()[:total], st.cpu().numpy()[:n])
    assert np.array_equal(_as_headers(hdr, n).view(np.uint8), want.view(np.uint8))
    codec.close()


def test_tampering_turns_segments_into_misses():
    """Flip bytes in some slots and fields in some headers (host-side
    injection), verify on the GPU, then decode with the verify result: damaged
    segments are CORRUPT and their pages stay untouched; the rest restore."""
    case = synth.make_case("vllm_packed", num_layers=5, num_blocks=8)
    arm = case.arms[0]
    codec, rows, total, layers, descs, enc, st = _encode(case, arm)
    n = len(rows)
    g = oracle_geom(case, arm)
    d = oracle_descs(rows)
    hdr = _headers(n)
    codec.seal(descs, n, enc, total, st, hdr)
    torch.cuda.synchronize()
    st_h = st.cpu().numpy()[:n]
    coded = np.flatnonzero(st_h == O.S_ENCODED)
    rng = np.random.default_rng(3)
    victims = rng.choice(coded, size=6, replace=False)
    enc_bad = enc.cpu().numpy().copy()
    hdr_bad = _as_headers(hdr, n).copy()
    seg = [codec.segment_bytes(r)[0] for r in (0, 1)]
    for k, i in enumerate(victims):
        layer, blk, role, off = rows[i]
        if k < 3:   # payload damage: a codes byte, the metadata tail, the padding end
            pos = [1, seg[role] - 200, seg[role] - 1][k]
            enc_bad[off + pos] ^= 1 << k
        else:       # header damage
            field = ["crc32", "stored_bytes", "version"][k - 3]
            hdr_bad[i][field] ^= 1
    enc_d = torch.from_numpy(enc_bad).cuda()
    hdr_d = torch.from_numpy(hdr_bad.view(np.uint8).copy()).cuda()
    res = torch.full((n,), 0xEE, dtype=torch.uint8, device="cuda")
    codec.verify(descs, n, enc_d, total, hdr_d, res)
    torch.cuda.synchronize()
    r = res.cpu().numpy()
    assert np.array_equal(r, O.verify(g, d, enc_bad[:total], hdr_bad))
    assert set(np.flatnonzero(r == O.S_CORRUPT)) == set(victims.tolist())
    # decode with the verified statuses: victims are misses
    dst = [torch.full_like(t, 0).view(torch.int16).fill_(SENTINEL_PAGE).view(t.dtype) for t in layers]
    out_res = torch.full((n,), 0xEE, dtype=torch.uint8, device="cuda")
    codec.decode(dst, descs, n, enc_d, total, res, out_res)
    torch.cuda.synchronize()
    assert np.array_equal(out_res.cpu().numpy(), r)
    D, T, H = case.head_dim, case.block_tokens, case.num_heads
    for i in victims:
        layer, blk, role, _ = rows[i]
        page = host_bits(dst[layer][blk]).reshape(H, T, 2 * D)[:, :, role * D:(role + 1) * D]
        assert np.all(page == SENTINEL_PAGE)
    codec.close()


def test_host_resident_slots_and_headers():
    case = synth.make_case("hiq_qwen3_8b", num_layers=2, num_blocks=6)
    arm = case.arms[0]
    codec, rows, total, layers, descs, enc, st = _encode(case, arm)
    n = len(rows)
    enc_h, st_h = enc.cpu().pin_memory(), st.cpu().pin_memory()
    descs_h = K.descriptors(rows, "cpu").pin_memory()
    hdr = _headers(n, "host")
    codec.seal(descs_h, n, enc_h, total, st_h, hdr)
    res = torch.full((n,), 0xEE, dtype=torch.uint8).pin_memory()
    codec.verify(descs_h, n, enc_h, total, hdr, res)
    torch.cuda.synchronize()
    want = O.seal(oracle_geom(case, arm), oracle_descs(rows), enc_h.numpy()[:total], st_h.numpy()[:n])
    assert np.array_equal(hdr.numpy()[: 32 * n], want.view(np.uint8))
    assert np.all(res.numpy() == O.S_ENCODED)
    codec.close()


def test_headers_carry_format_version_2():
    """Sealed headers of a format-version-2 geometry carry version 2, equal to
    the oracle's, and verify passes them."""
    case = synth.make_case("vllm_packed", num_layers=5, num_blocks=3)
    assert run_seal_parity(case, case.arms[0], sign_version=2) > 0
