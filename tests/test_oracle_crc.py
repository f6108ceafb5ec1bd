"""Pins of the oracle's segment header and CRC-32 (OrbitKV docs, section
"Ownership, storage and GDS": version, original length, format, stored length
and CRC32 per encoded segment, checked before GPU decode; a damaged object
becomes a miss).  The bit-serial CRC is pinned to the published check value
and to zlib's table-driven implementation (a library special case); sealing
and verifying are pinned by tampering with every field and byte class."""
import zlib

import numpy as np
import pytest

import oracle as O
from kvcases import host_bits, oracle_descs, oracle_geom
from kv_cache_page_gb300 import synth


def test_crc32_check_value():
    # the catalogue "check" value of CRC-32 (ISO-HDLC / zlib): CRC of ASCII 123456789
    assert O.crc32(b"123456789") == 0xCBF43926
    assert O.crc32(b"") == 0


@pytest.mark.parametrize("n", list(range(0, 70)) + [127, 128, 129, 4096, 16896, 1 << 20])
def test_crc32_equals_zlib(n):
    rng = np.random.default_rng(n)
    b = rng.integers(0, 256, n, dtype=np.uint8)
    assert O.crc32(b) == zlib.crc32(b.tobytes())


def test_crc32_is_affine_in_the_message():
    """CRC(a ^ b ^ c) = CRC(a) ^ CRC(b) ^ CRC(c) for messages of one length (the
    register preset and final complement make it affine, not linear)."""
    rng = np.random.default_rng(1)
    for n in (1, 16, 100, 1152):
        a, b, c = (rng.integers(0, 256, n, dtype=np.uint8) for _ in range(3))
        assert O.crc32(a ^ b ^ c) == O.crc32(a) ^ O.crc32(b) ^ O.crc32(c)


def _encoded(name="tiny", arm_index=0, **kw):
    case = synth.make_case(name, **kw)
    arm = case.arms[arm_index]
    g = oracle_geom(case, arm)
    seg = [O.segment_enc_bytes(g, r) for r in (0, 1)]
    rows, total = synth.segment_list(case, arm, seg)
    enc, st = O.encode(g, [host_bits(t) for t in case.layers], oracle_descs(rows), total)
    return case, arm, g, rows, seg, enc, st


def test_header_fields():
    case, arm, g, rows, seg, enc, st = _encoded()
    h = O.seal(g, oracle_descs(rows), enc, st)
    assert O.HEADER_DTYPE.itemsize == 32
    for (layer, blk, role, off), hh, s in zip(rows, h, st):
        assert hh["version"] == 1
        # FP8 dynamic = 3, FP16 = 1, head_dim 128 = 2^7
        assert hh["format"] == 3 | (1 << 8) | (7 << 16)
        assert hh["orig_bytes"] == 16 * 8 * 128 * 2
        assert hh["status"] == s == O.S_ENCODED
        assert hh["stored_bytes"] == seg[role]
        assert hh["crc32"] == zlib.crc32(enc[off:off + seg[role]].tobytes())


def test_verify_accepts_sealed_and_rejects_tampering():
    case, arm, g, rows, seg, enc, st = _encoded("vllm_packed", num_layers=5, num_blocks=4)
    d = oracle_descs(rows)
    h = O.seal(g, d, enc, st)
    assert np.array_equal(O.verify(g, d, enc, h), st)        # raw statuses pass through
    coded = np.flatnonzero(st == O.S_ENCODED)
    raw = np.flatnonzero(st != O.S_ENCODED)
    assert coded.size and raw.size
    i = int(coded[3])
    off, role = rows[i][3], rows[i][2]
    # one flipped bit anywhere in the slot (codes, metadata, padding)
    for pos in (0, seg[role] // 2, seg[role] - 1):
        bad = enc.copy()
        bad[off + pos] ^= 0x10
        r = O.verify(g, d, bad, h)
        assert r[i] == O.S_CORRUPT
        assert np.array_equal(np.delete(r, i), np.delete(st, i))
    # every header field
    for field, val in (("version", 2), ("format", int(h[i]["format"]) ^ 1),
                       ("orig_bytes", int(h[i]["orig_bytes"]) + 2),
                       ("stored_bytes", int(h[i]["stored_bytes"]) - 128),
                       ("crc32", int(h[i]["crc32"]) ^ 0x80000000), ("status", 10)):
        hb = h.copy()
        hb[i][field] = val
        assert O.verify(g, d, enc, hb)[i] == O.S_CORRUPT, field
    # a raw segment's header claiming stored bytes
    j = int(raw[0])
    hb = h.copy()
    hb[j]["stored_bytes"] = 128
    assert O.verify(g, d, enc, hb)[j] == O.S_CORRUPT
    # a raw header swapped in for an encoded segment makes it a miss, not a decode
    hb = h.copy()
    hb[i] = h[j]
    hb[i]["format"] = h[i]["format"]
    assert O.verify(g, d, enc, hb)[i] == h[j]["status"] != O.S_ENCODED


def test_bad_descriptors():
    case, arm, g, rows, seg, enc, st = _encoded()
    d = oracle_descs(rows[:2] + [(5, 0, 0, 0), (0, 0, 2, 0), (0, 0, 0, 8), (0, 0, 0, len(enc))])
    stx = np.concatenate([st[:2], np.full(4, O.S_ENCODED, np.uint8)])
    h = O.seal(g, d, enc, stx)
    assert list(h["status"][2:]) == [O.S_BAD_DESC] * 4
    assert list(O.verify(g, d, enc, h)) == [O.S_ENCODED] * 2 + [O.S_BAD_DESC] * 4
