"""Host-only checks of the C ABI (no GPU): the library loads, exports every
declared symbol, validates geometries, and its size queries, codebooks and
sign vectors equal the oracle's (each side computes its own).
"""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle as O
from kv_cache_page_gb300 import build as kbuild
from kv_cache_page_gb300 import codec as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kv_codec.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    kbuild.build()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(kv_codec_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert set(names) == set(K.EXPORTS)
    L = C.CDLL(K.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n


def test_bounds_checked_build_exports_every_declared_symbol():
    """The debug library (every kernel access checked against the call's
    buffers) builds from the same sources and has the same entry points."""
    L = C.CDLL(kbuild.build(debug=True))
    for n in declared_functions():
        assert hasattr(L, n), n
    L.kv_codec_strerror.restype = C.c_char_p
    assert b"outside the call's buffers" in L.kv_codec_strerror(-11)


def test_abi_version_and_struct_size():
    assert K.lib().kv_codec_abi_version() == K.ABI_VERSION
    assert C.sizeof(K.Geometry) == 112


def test_fixed_overflow_field_and_earlier_struct_size():
    """fixed_overflow: clip (0) or reject (1), reserved must be 0; a geometry of
    the earlier 104-byte layout (no fixed_overflow) is still accepted."""
    kw = _kw(k_codec="fp8_fixed", v_codec="fp8_fixed", fixed_amax=np.ones((4, 2)))
    for mode in ("clip", "reject"):
        K.Codec(**kw, fixed_overflow=mode).close()
    for over in ({"fixed_overflow": 2}, {"reserved": 1}, {"struct_size": 108}, {"struct_size": 96}):
        with pytest.raises(K.KvCodecError) as e:
            K.Codec(**kw, geometry_overrides=over)
        assert e.value.code == (-7 if "struct_size" in over else -1)
    # 104 bytes: the trailing fields are not read (a nonzero reserved is ignored)
    K.Codec(**kw, geometry_overrides={"struct_size": 104, "fixed_overflow": 7, "reserved": 3}).close()


def _kw(**over):
    kw = dict(dtype="fp16", layout="separate", head_dim=128, num_kv_heads=8, block_tokens=16,
              num_layers=4, num_blocks=16, strides=(16 * 8 * 128, 8 * 128, 128),
              k_codec="tq4", v_codec="uni4", protect=(0, 0), rotation_seed=3)
    kw.update(over)
    return kw


@pytest.mark.parametrize("over,code", [
    (dict(head_dim=96), -2),
    (dict(head_dim=512), -2),
    (dict(dtype="fp16", geometry_overrides={"dtype": 7}), -1),
    (dict(geometry_overrides={"layout": 9}), -1),
    (dict(num_layers=0), -8),
    (dict(num_layers=513), -8),
    (dict(v_codec="tq3"), -4),
    (dict(v_codec="tq2"), -4),
    (dict(geometry_overrides={"k_codec": 12}), -1),
    (dict(strides=(16 * 8 * 128, 8 * 128, 100)), -5),        # head stride not 16-byte aligned
    (dict(strides=(16 * 8 * 128, 8 * 128, 64)), -3),         # heads overlap (64 < D)
    (dict(strides=(8 * 128, 8 * 128, 128)), -3),             # pages overlap tokens
    (dict(strides=(0, 8 * 128, 128)), -3),
    (dict(layout="packed", strides=(8 * 16 * 256, 256, 16 * 128)), -3),  # packed rows are 2D
    (dict(reject_abs=500.0), -1),
    (dict(reject_abs=float("inf")), -1),   # bounds above 448 could let FP16 metadata overflow
    (dict(reject_abs=-1.0), -1),
    (dict(reject_abs=float("nan")), -1),
    (dict(k_codec="fp8_fixed", v_codec="fp8_fixed"), -1),    # fixed scales missing
    (dict(geometry_overrides={"abi_version": 2}), -7),
    (dict(geometry_overrides={"struct_size": 96}), -7),
    (dict(sign_version=3), -1),
    (dict(num_kv_heads=0), -1),
    (dict(num_blocks=0), -1),
])
def test_geometry_rejections(over, code):
    with pytest.raises(K.KvCodecError) as e:
        K.Codec(**_kw(**over))
    assert e.value.code == code


def test_valid_geometries_and_layout_variants():
    K.Codec(**_kw()).close()
    # HND page layout [block, head, token, D] expressed by strides
    K.Codec(**_kw(strides=(16 * 8 * 128, 128, 16 * 128))).close()
    # vLLM packed [block, head, token, 2D]
    K.Codec(**_kw(layout="packed", strides=(8 * 16 * 256, 256, 16 * 256))).close()
    K.Codec(**_kw(k_codec="fp8_fixed", v_codec="none", fixed_amax=np.ones((4, 2)))).close()
    K.Codec(**_kw(k_codec="none", v_codec="none")).close()
    # a single page / single head: extent-1 strides do not matter
    K.Codec(**_kw(num_blocks=1, num_kv_heads=1, strides=(8, 128, 8))).close()


def _oracle_geom(k, v, D, H=8, T=16):
    return O.make_geom(dtype=O.FP16, layout=O.SEPARATE, head_dim=D, num_heads=H, block_tokens=T,
                       num_layers=2, num_blocks=2, strides=(T * H * D, H * D, D),
                       codecs=(K.CODEC[k], K.CODEC[v]), fixed_amax=np.ones((2, 2), np.float32))


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("kc,vc", [("fp8_cast", "fp8_fixed"), ("fp8_dynamic", "fp8_dynamic"),
                                   ("tq3", "uni3"), ("tq4", "uni4"), ("uni8", "uni8"), ("none", "uni4"),
                                   ("tq2", "uni2")])
@pytest.mark.parametrize("H,T", [(8, 16), (3, 5), (1, 1)])
def test_segment_bytes_match_oracle(D, kc, vc, H, T):
    c = K.Codec(**_kw(head_dim=D, num_kv_heads=H, block_tokens=T, num_layers=2, num_blocks=2,
                      strides=(T * H * D, H * D, D), k_codec=kc, v_codec=vc, fixed_amax=np.ones((2, 2))))
    g = _oracle_geom(kc, vc, D, H, T)
    for role, name in ((0, kc), (1, vc)):
        enc, raw = c.segment_bytes(role)
        assert raw == O.segment_raw_bytes(g)
        assert enc == (0 if name == "none" else O.segment_enc_bytes(g, role))
    c.close()


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("kc,vc", [("int8", "int8"), ("int8", "fp8_dynamic"), ("none", "int8")])
@pytest.mark.parametrize("H,T", [(8, 16), (3, 5), (1, 1), (32, 16)])
def test_int8_record_segment_bytes_match_oracle(D, kc, vc, H, T):
    c = K.Codec(**_kw(dtype="bf16", head_dim=D, num_kv_heads=H, block_tokens=T, num_layers=2,
                      num_blocks=2, strides=(T * H * D, H * D, D), k_codec=kc, v_codec=vc))
    g = O.make_geom(dtype=O.BF16, layout=O.SEPARATE, head_dim=D, num_heads=H, block_tokens=T,
                    num_layers=2, num_blocks=2, strides=(T * H * D, H * D, D),
                    codecs=(K.CODEC[kc], K.CODEC[vc]))
    for role, name in ((0, kc), (1, vc)):
        enc, raw = c.segment_bytes(role)
        assert raw == O.segment_raw_bytes(g)
        assert enc == (0 if name == "none" else O.segment_enc_bytes(g, role))
        if name == "int8":
            assert enc == T * O.int8_record_bytes(H, D)
    c.close()


def test_int8_needs_bf16_source():
    for kc, vc in (("int8", "none"), ("fp8_dynamic", "int8")):
        with pytest.raises(K.KvCodecError) as e:
            K.Codec(**_kw(dtype="fp16", k_codec=kc, v_codec=vc))
        assert e.value.code == -10


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("D", [32, 64, 128, 256])
def test_codebook_bitwise_equal_to_oracle(bits, D):
    cent, bnd = K.codebook(bits, D)
    ocent, obnd = O.codebook(bits, D)
    assert np.array_equal(cent.view(np.uint32), ocent.view(np.uint32))
    assert np.array_equal(bnd.view(np.uint32), obnd.view(np.uint32))


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("seed", [0, 1, 12345, 2**64 - 1])
def test_signs_equal_to_oracle(D, seed):
    assert np.array_equal(K.signs(seed, D), O.signs(seed, D))


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("seed", [0, 99, 2**64 - 1])
def test_layer_signs_equal_to_oracle(D, seed):
    for layer in (0, 1, 7, 511):
        assert np.array_equal(K.layer_signs(seed, layer, D), O.signs_layer(seed, layer, D)), layer
    assert np.array_equal(K.layer_signs(seed, 0, D), K.signs(seed, D))


def test_layer_signs_refuse_bad_arguments():
    with pytest.raises(K.KvCodecError):
        K.layer_signs(0, 512, 64)
    with pytest.raises(K.KvCodecError):
        K.layer_signs(0, 0, 48)


@pytest.mark.parametrize("v", [0, 1, 2])
def test_sign_versions_accepted(v):
    c = K.Codec(dtype="bf16", layout="separate", head_dim=128, num_kv_heads=8, block_tokens=16,
                num_layers=4, num_blocks=2, strides=(16 * 8 * 128, 8 * 128, 128), k_codec="tq4",
                v_codec="uni4", sign_version=v)
    c.close()


def test_call_argument_checks_need_no_gpu():
    c = K.Codec(**_kw())
    buf = 16 * 1024
    # n_segments == 0 is a no-op
    c.encode([None] * 8, 0, 0, 0, 0, 0, stream=0)
    with pytest.raises(K.KvCodecError) as e:     # wrong pointer count for the layout
        c.encode([0x1000] * 7, 0x2000, 1, 0x3000, buf, 0x4000, stream=0)
    assert e.value.code == -1
    with pytest.raises(K.KvCodecError) as e:     # misaligned layer pointer
        c.encode([0x1008] * 8, 0x2000, 1, 0x3000, buf, 0x4000, stream=0)
    assert e.value.code == -5
    with pytest.raises(K.KvCodecError) as e:     # misaligned encoded buffer
        c.decode([0x1000] * 8, 0x2000, 1, 0x3004, buf, 0x4000, stream=0)
    assert e.value.code == -5
    with pytest.raises(K.KvCodecError) as e:     # missing status array
        c.encode([0x1000] * 8, 0x2000, 1, 0x3000, buf, None, stream=0)
    assert e.value.code == -1
    for call in (c.encode, c.decode):             # more than 2^31 - 1 segments in one call
        with pytest.raises(K.KvCodecError) as e:
            call([0x1000] * 8, 0x2000, 1 << 31, 0x3000, buf, 0x4000, stream=0)
        assert e.value.code == -1
    c.close()


def test_seal_verify_argument_checks_need_no_gpu():
    c = K.Codec(**_kw())
    with pytest.raises(K.KvCodecError) as e:
        c.seal(0x2000, 1, None, 1024, 0x4000, 0x5000, stream=0)
    assert e.value.code == -1
    with pytest.raises(K.KvCodecError) as e:
        c.seal(0x2000, 1, 0x3008, 1024, 0x4000, 0x5000, stream=0)      # slots not 16-aligned
    assert e.value.code == -5
    with pytest.raises(K.KvCodecError) as e:
        c.verify(0x2000, 1, 0x3000, 1024, 0x5004, 0x6000, stream=0)    # headers not 8-aligned
    assert e.value.code == -5
    with pytest.raises(K.KvCodecError) as e:
        c.verify(0x2000, 1, 0x3000, 1024, 0x5000, None, stream=0)
    assert e.value.code == -1
    c.seal(0, 0, 0, 0, 0, 0, stream=0)                                 # n = 0: no-op
    c.verify(0, 0, 0, 0, 0, 0, stream=0)
    assert K.HEADER_DTYPE.itemsize == 32 == O.HEADER_DTYPE.itemsize
    c.close()


def test_sealed_and_verified_argument_checks_need_no_gpu():
    c = K.Codec(**_kw())
    buf = 16 * 1024
    c.encode_sealed([None] * 8, 0, 0, 0, 0, 0, 0, stream=0)             # n = 0: no-op
    c.decode_verified([None] * 8, 0, 0, 0, 0, 0, 0, stream=0)
    cases = [
        (lambda: c.encode_sealed([0x1000] * 8, 0x2000, 1, 0x3000, buf, 0x4000, None, stream=0), -1),
        (lambda: c.encode_sealed([0x1000] * 8, 0x2000, 1, 0x3000, buf, 0x4000, 0x5004, stream=0), -5),
        (lambda: c.encode_sealed([0x1000] * 8, 0x2000, 1, 0x3008, buf, 0x4000, 0x5000, stream=0), -5),
        (lambda: c.encode_sealed([0x1000] * 7, 0x2000, 1, 0x3000, buf, 0x4000, 0x5000, stream=0), -1),
        (lambda: c.decode_verified([0x1000] * 8, 0x2000, 1, 0x3000, buf, 0x5000, None, stream=0), -1),
        (lambda: c.decode_verified([0x1000] * 8, 0x2000, 1, 0x3000, buf, None, 0x6000, stream=0), -1),
        (lambda: c.decode_verified([0x1000] * 8, 0x2000, 1, 0x3000, buf, 0x5004, 0x6000, stream=0), -5),
        (lambda: c.decode_verified([0x1008] * 8, 0x2000, 1, 0x3000, buf, 0x5000, 0x6000, stream=0), -5),
    ]
    for call, code in cases:
        with pytest.raises(K.KvCodecError) as e:
            call()
        assert e.value.code == code
    c.close()


def test_strerror_covers_codes():
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "kv_codec.h")).read()
    codes = [int(c) for c in re.findall(r"#define KV_ERR_\w+ (-\d+)", hdr)]
    assert sorted(codes) == list(range(-len(codes), 0))
    for code in [0] + codes:
        assert K.strerror(code) != "unknown error", code
    assert K.strerror(-99) == "unknown error"
