"""Pins of format version 2: one TurboQuant sign vector per (seed, layer, head dim).

"KV precision and storage encoding" (OrbitKV), section "FP8 and TurboQuant",
names a versioned sign generator that is the implementation's own.  Version 2
here: layer l draws its W = ceil(D/64) words from the version-1 SplitMix64
stream after the W*l words of the layers below it (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014).  The pins:
layer 0 is the version-1 vector; the words of layers 0..2 are the generator's
published first outputs for seed 0; whole segments of a version-2 geometry
equal the per-vector codec run with their layer's signs; headers carry the
version and a header of the other version is a mismatch.
"""
import numpy as np
import pytest

import oracle as O
from kvcases import oracle_descs

HEAD_DIMS = (32, 64, 128, 256)
# SplitMix64, seed 0: its first three outputs, as published with the reference
# implementation (and pinned for version 1 in test_oracle_codecs.py)
PUBLISHED = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def _bits(word, n):
    return np.array([(word >> i) & 1 for i in range(n)], np.uint8)


@pytest.mark.parametrize("D", HEAD_DIMS)
@pytest.mark.parametrize("seed", [0, 7, 2**63 + 5])
def test_layer_zero_is_version_one(D, seed):
    assert np.array_equal(O.signs_layer(seed, 0, D), O.signs(seed, D))


def test_layers_take_successive_published_words():
    # D = 64: one word per layer, so layers 0, 1, 2 are outputs 0, 1, 2
    for layer in range(3):
        assert np.array_equal(O.signs_layer(0, layer, 64), _bits(PUBLISHED[layer], 64))
    # D = 32: the low half of one word per layer
    for layer in range(3):
        assert np.array_equal(O.signs_layer(0, layer, 32), _bits(PUBLISHED[layer], 32))
    # D = 128: two words per layer, so layer 1 starts with output 2
    assert np.array_equal(O.signs_layer(0, 1, 128)[:64], _bits(PUBLISHED[2], 64))
    assert np.array_equal(O.signs_layer(0, 0, 128), np.concatenate([_bits(PUBLISHED[0], 64),
                                                                     _bits(PUBLISHED[1], 64)]))


@pytest.mark.parametrize("D", HEAD_DIMS)
def test_layers_differ_and_are_balanced(D):
    s = np.stack([O.signs_layer(3, layer, D) for layer in range(64)])
    assert len({r.tobytes() for r in s}) == 64
    assert abs(s.mean() - 0.5) < 0.05


def _geom(D, H, T, L, B, sign_version, codecs=(O.TQ4, O.UNI4)):
    return O.make_geom(dtype=O.BF16, layout=O.SEPARATE, head_dim=D, num_heads=H, block_tokens=T,
                       num_layers=L, num_blocks=B, strides=(T * H * D, H * D, D), codecs=codecs,
                       seed=11, sign_version=sign_version)


@pytest.mark.parametrize("D,bits", [(128, 4), (64, 3), (32, 2), (256, 4)])
def test_segments_use_their_layer_signs(D, bits):
    H, T, L, B = 2, 16, 4, 2
    tq = {2: O.TQ2, 3: O.TQ3, 4: O.TQ4}[bits]
    uni = {2: O.UNI2, 3: O.UNI3, 4: O.UNI4}[bits]
    rng = np.random.default_rng(D + bits)
    x = rng.standard_normal((L, 2, B, T, H, D)).astype(np.float32)
    src = O.f32_to_bf16(x)
    xs = O.bf16_to_f32(src)
    layers = [src[l, r].reshape(-1).copy() for l in range(L) for r in range(2)]
    g2 = _geom(D, H, T, L, B, 2, (tq, uni))
    g1 = _geom(D, H, T, L, B, 1, (tq, uni))
    seg = [O.segment_enc_bytes(g2, r) for r in (0, 1)]
    rows, off = [], 0
    for l in range(L):
        for b in range(B):
            for r in range(2):
                rows.append((l, b, r, off))
                off += seg[r]
    enc2, st2 = O.encode(g2, layers, oracle_descs(rows), off)
    enc1, st1 = O.encode(g1, layers, oracle_descs(rows), off)
    assert np.all(st2 == O.S_ENCODED) and np.all(st1 == O.S_ENCODED)
    nv = T * H
    cb = D * bits // 8
    for (l, b, r, o) in rows:
        s2, s1 = enc2[o:o + seg[r]], enc1[o:o + seg[r]]
        if r == 1 or l == 0:
            assert np.array_equal(s2, s1)          # V (uniform) and layer 0 do not depend on it
            continue
        neg = O.signs_layer(11, l, D)
        c, n16 = O.tq_encode_with_signs(xs[l, 0, b].reshape(nv, D), bits, neg)
        want = np.concatenate([np.concatenate([O.pack_bits(v, bits) for v in c]), n16.view(np.uint8)])
        assert np.array_equal(s2[:want.size], want), (l, b)
        assert not np.array_equal(s2, s1)
    # restore: each layer's K pages from its own signs
    out = [np.zeros_like(a) for a in layers]
    res = O.decode(g2, out, oracle_descs(rows), enc2, st2)
    assert np.all(res == O.S_ENCODED)
    for (l, b, r, o) in rows:
        if r:
            continue
        s = enc2[o:o + seg[0]]
        c = O.unpack_bits(s[:nv * cb], nv * D, bits).reshape(nv, D)
        n16 = s[nv * cb:nv * cb + 2 * nv].view(np.uint16)
        y = O.tq_decode_with_signs(c, n16, bits, O.signs_layer(11, l, D))
        got = out[2 * l].reshape(B, nv, D)[b]
        assert np.array_equal(got, O.f32_to_bf16(y)), (l, b)


def test_header_carries_the_format_version():
    D, H, T, L, B = 64, 2, 16, 3, 1
    rng = np.random.default_rng(1)
    src = O.f32_to_bf16(rng.standard_normal((L, 2, B, T, H, D)).astype(np.float32))
    layers = [src[l, r].reshape(-1).copy() for l in range(L) for r in range(2)]
    g2, g1 = _geom(D, H, T, L, B, 2), _geom(D, H, T, L, B, 1)
    seg = [O.segment_enc_bytes(g2, r) for r in (0, 1)]
    rows = [(l, 0, r, (2 * l + r) * max(seg)) for l in range(L) for r in range(2)]
    d = oracle_descs(rows)
    enc, st = O.encode(g2, layers, d, 2 * L * max(seg))
    h2 = O.seal(g2, d, enc, st)
    assert np.all(h2["version"] == 2)
    assert np.all(O.verify(g2, d, enc, h2) == O.S_ENCODED)
    # the same slots under a version-1 geometry: header version mismatch -> miss
    assert np.all(O.verify(g1, d, enc, h2) == O.S_CORRUPT)
    h1 = O.seal(g1, d, enc, st)
    assert np.all(h1["version"] == 1)
    assert np.all(O.verify(g2, d, enc, h1) == O.S_CORRUPT)
