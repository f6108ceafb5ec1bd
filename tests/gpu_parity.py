"""Run a workload through the CUDA codec (via the C ABI) and through the oracle
on the same bits, and compare.  Used by the GPU tests and the smoke check.

Comparison rules: statuses bit-exact; ENCODED slots byte-exact (codes,
metadata and zero padding); restored pages within one unit in the last place
of the 16-bit format (+0 and -0 equal), which the kernels in fact meet
exactly; restore results byte-exact.  Bounds: every buffer a call may write
sits between guard zones that must stay untouched, slot-buffer bytes outside
the accepted descriptors' slots keep their sentinel, and encode leaves its
source pages unchanged.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from kv_cache_page_gb300 import codec as K
from kv_cache_page_gb300 import synth
from kvcases import host_bits, oracle_descs, oracle_geom

SENTINEL_ENC = 0xAB
SENTINEL_PAGE = 0x7BCD  # an ordinary finite value, never produced by chance in bulk


def make_codec(case: synth.Case, arm: synth.Arm, reject_abs=448.0, sign_version=1,
               fixed_overflow="clip") -> K.Codec:
    return K.Codec(dtype="fp16" if case.dtype == torch.float16 else "bf16", layout=case.layout,
                   head_dim=case.head_dim, num_kv_heads=case.num_heads,
                   block_tokens=case.block_tokens, num_layers=case.num_layers,
                   num_blocks=case.num_blocks, strides=case.strides, k_codec=arm.k_codec,
                   v_codec=arm.v_codec, protect=arm.protect, rotation_seed=case.seed,
                   reject_abs=reject_abs, sign_version=sign_version, fixed_overflow=fixed_overflow,
                   fixed_amax=None if case.fixed_amax is None else case.fixed_amax.numpy())


def ulp_diff_16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units of the last place between 16-bit float patterns
    (sign-magnitude -> monotone integers; +0 and -0 both map to 0)."""
    def key(x):
        x = x.astype(np.int64)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(key(a) - key(b))


def compare_pages(got: np.ndarray, want: np.ndarray, what: str):
    if np.array_equal(got, want):
        return 0
    d = ulp_diff_16(got, want)
    bad = np.flatnonzero(d > 1)
    assert bad.size == 0, (f"{what}: {bad.size} elements differ by > 1 ulp; first at {bad[:5]}: "
                           f"got {got[bad[:5]]} want {want[bad[:5]]}")
    return int(np.count_nonzero(d))


def _buffer(t: torch.Tensor, where: str, device) -> torch.Tensor:
    """`t` as a device tensor, or as a pinned host tensor that the kernels reach
    through its device mapping."""
    if where == "host":
        return t.cpu().pin_memory()
    return t.to(device)


GUARD = 4096           # sentinel bytes on each side of every buffer a call may write
SENTINEL_GUARD = 0x5A


class Guarded:
    """A copy of `t` placed GUARD + offset_bytes bytes into an allocation filled
    with SENTINEL_GUARD and followed by GUARD more sentinel bytes, in device or
    pinned host memory (`where`).  The kernels get `.t`; `check()` asserts that
    nothing outside it was written (a write past either end of a caller buffer,
    e.g. from a wrong index in a ragged last step, lands in a guard).  With
    offset_bytes = 16 the copy is 16- but not 32-byte aligned."""

    def __init__(self, t: torch.Tensor, where: str, device, offset_bytes: int = 0):
        t = t.contiguous()
        nbytes = t.numel() * t.element_size()
        self.lead, self.nbytes = GUARD + offset_bytes, nbytes
        raw = torch.full((self.lead + nbytes + GUARD,), SENTINEL_GUARD, dtype=torch.uint8)
        self.raw = raw.pin_memory() if where == "host" else raw.to(device)
        self.t = self.raw[self.lead:self.lead + nbytes].view(t.dtype).view(t.shape)
        self.t.copy_(t.to(self.t.device))
        assert self.t.data_ptr() % 32 == offset_bytes % 32

    def check(self, what: str):
        r = self.raw.cpu().numpy()
        bad = np.flatnonzero(np.concatenate([r[:self.lead], r[self.lead + self.nbytes:]]) != SENTINEL_GUARD)
        assert bad.size == 0, f"{what}: {bad.size} guard bytes written"


def guarded_layers(case: synth.Case, device, offset_bytes: int = 0):
    return [Guarded(t, "device", device, offset_bytes) for t in case.layers]


def check_slot_gaps(enc: np.ndarray, rows, seg, status, what: str):
    """Bytes of the slot buffer outside the slot of every descriptor the call
    accepted (status other than BAD_DESC) still hold SENTINEL_ENC."""
    free = np.ones(enc.size, bool)
    for (layer, blk, role, off), st in zip(rows, status):
        if st != O.S_BAD_DESC and role <= 1:
            free[off:off + seg[role]] = False
    bad = np.flatnonzero(free & (enc != SENTINEL_ENC))
    assert bad.size == 0, f"{what}: {bad.size} bytes written outside the slots, first at {bad[:5]}"


def run_parity(case: synth.Case, arm: synth.Arm, rows=None, total=None, device="cuda",
               reject_abs=448.0, check_decode=True, buffers="device", layer_offset=0, sign_version=1,
               fixed_overflow="clip"):
    """Encode + decode `case` with `arm` on the GPU and in the oracle; assert parity.
    buffers="host" keeps descriptors, slots, statuses and results in pinned host
    memory (the kernels read and write them over the host link).  layer_offset
    places the source and restored layer tensors that many bytes past an aligned
    allocation (16: the 16-byte alignment the library requires, not 32).
    sign_version 2: TurboQuant sign vectors per layer (format version 2).
    fixed_overflow "reject": FP8 fixed-scale segments with a quotient beyond
    +-448 stay raw.  Returns (status array, number of restored elements off by
    one ulp)."""
    codec = make_codec(case, arm, reject_abs, sign_version, fixed_overflow)
    g = oracle_geom(case, arm, reject_abs, sign_version, fixed_overflow)
    seg = [codec.segment_bytes(r)[0] for r in (0, 1)]
    assert seg == [0 if c == "none" else O.segment_enc_bytes(g, r)
                   for r, c in enumerate((arm.k_codec, arm.v_codec))]
    if rows is None:
        rows, total = synth.segment_list(case, arm, seg)
    elif total is None:
        total = max([r[3] + seg[r[2]] for r in rows if r[2] <= 1 and r[3] < (1 << 32)] + [16])
    n = len(rows)
    src = guarded_layers(case, device, layer_offset)
    dev_layers = [x.t for x in src]
    host_layers = [host_bits(t) for t in case.layers]
    descs = _buffer(K.descriptors(rows, "cpu"), buffers, device)
    out_g = Guarded(torch.full((max(total, 16),), SENTINEL_ENC, dtype=torch.uint8), buffers, device)
    status_g = Guarded(torch.full((max(n, 1),), 0xEE, dtype=torch.uint8), buffers, device)
    out, status = out_g.t, status_g.t
    codec.encode(dev_layers, descs, n, out, total, status)
    torch.cuda.synchronize()
    for k, x in enumerate(src):
        x.check(f"source layer {k}")
        assert np.array_equal(host_bits(x.t), host_layers[k]), f"encode wrote source layer {k}"
    out_g.check("slot buffer")
    status_g.check("status array")
    enc_ref, st_ref = O.encode(g, host_layers, oracle_descs(rows), total)
    st_gpu = status[:n].cpu().numpy()
    assert np.array_equal(st_gpu, st_ref), f"status mismatch at {np.flatnonzero(st_gpu != st_ref)[:10]}"
    enc_gpu = out[:total].cpu().numpy()
    check_slot_gaps(enc_gpu, rows, seg, st_ref, "encode")
    for (layer, blk, role, off), s in zip(rows, st_ref):
        if s == O.S_ENCODED:
            a, b = enc_gpu[off:off + seg[role]], enc_ref[off:off + seg[role]]
            if not np.array_equal(a, b):
                bad = np.flatnonzero(a != b)
                raise AssertionError(f"slot (layer {layer}, block {blk}, role {role}) differs at "
                                     f"{bad.size} bytes, first {bad[:8]}: got {a[bad[:8]]} want {b[bad[:8]]}")
        elif s == O.S_BAD_DESC:
            pass
    ulps = 0
    if check_decode:
        # decode the oracle's encoding on the GPU into sentinel-filled pages
        dst_g = guarded_layers(case, device, layer_offset)
        dst_dev = [x.t for x in dst_g]
        for t in dst_dev:
            t.view(torch.int16).fill_(SENTINEL_PAGE)
        dst_host = [np.full_like(h, SENTINEL_PAGE) for h in host_layers]
        enc_h = torch.zeros(max(total, 16), dtype=torch.uint8)
        enc_h[:total] = torch.from_numpy(enc_ref)
        enc_dev = _buffer(enc_h, buffers, device)
        st_dev = _buffer(torch.from_numpy(st_ref), buffers, device)
        result_g = Guarded(torch.full((max(n, 1),), 0xEE, dtype=torch.uint8), buffers, device)
        result = result_g.t
        codec.decode(dst_dev, descs, n, enc_dev, total, st_dev, result)
        torch.cuda.synchronize()
        for k, x in enumerate(dst_g):
            x.check(f"restored layer {k}")
        result_g.check("result array")
        assert np.array_equal(enc_dev.cpu().numpy(), enc_h.numpy()), "decode wrote the slot buffer"
        res_ref = O.decode(g, dst_host, oracle_descs(rows), enc_ref, st_ref)
        assert np.array_equal(result[:n].cpu().numpy(), res_ref)
        for k, (d_dev, d_host) in enumerate(zip(dst_dev, dst_host)):
            ulps += compare_pages(host_bits(d_dev), d_host, f"layer tensor {k}")
    codec.close()
    return st_ref, ulps


def run_seal_parity(case: synth.Case, arm: synth.Arm, device="cuda", sign_version=1):
    """Encode on the GPU, seal the slots (CRC-32 headers) and verify them; the
    headers must equal the oracle's bit for bit and verify must pass every
    segment's status through.  Returns the number of sealed ENCODED slots."""
    codec = make_codec(case, arm, sign_version=sign_version)
    seg = [codec.segment_bytes(r)[0] for r in (0, 1)]
    rows, total = synth.segment_list(case, arm, seg)
    n = len(rows)
    layers = [t.to(device) for t in case.layers]
    descs = K.descriptors(rows, device)
    enc = torch.zeros(max(total, 16), dtype=torch.uint8, device=device)
    st = torch.zeros(max(n, 1), dtype=torch.uint8, device=device)
    hdr_g = Guarded(torch.zeros(max(n, 1) * 32, dtype=torch.uint8), "device", device)
    res_g = Guarded(torch.zeros(max(n, 1), dtype=torch.uint8), "device", device)
    hdr, res = hdr_g.t, res_g.t
    codec.encode(layers, descs, n, enc, total, st)
    enc_before = enc.cpu().numpy()
    codec.seal(descs, n, enc, total, st, hdr)
    codec.verify(descs, n, enc, total, hdr, res)
    torch.cuda.synchronize()
    hdr_g.check("header array")
    res_g.check("result array")
    assert np.array_equal(enc.cpu().numpy(), enc_before), "seal or verify wrote the slot buffer"
    g = oracle_geom(case, arm, sign_version=sign_version)
    st_h = st.cpu().numpy()[:n]
    want = O.seal(g, oracle_descs(rows), enc.cpu().numpy()[:total], st_h)
    assert np.array_equal(hdr.cpu().numpy()[:32 * n], want.view(np.uint8)), "headers differ"
    assert np.array_equal(res.cpu().numpy()[:n], st_h), "verify rejected a sealed slot"
    codec.close()
    return int(np.count_nonzero(st_h == O.S_ENCODED))


def run_sealed_parity(case: synth.Case, arm: synth.Arm, rows=None, total=None, device="cuda",
                      buffers="device", tamper=0, seed=0, sign_version=1, fixed_overflow="clip"):
    """The one-call paths against the oracle.  encode_sealed: statuses, ENCODED
    slots and all headers equal the oracle's encode followed by seal.
    decode_verified, on the oracle's slots and headers with `tamper` ENCODED
    segments damaged on the host (a slot byte or a header field each): results
    equal the oracle's verify followed by decode with those results, damaged
    segments are CORRUPT and their pages keep the sentinel, the rest restore.
    Returns (statuses, verified results)."""
    codec = make_codec(case, arm, sign_version=sign_version, fixed_overflow=fixed_overflow)
    g = oracle_geom(case, arm, sign_version=sign_version, fixed_overflow=fixed_overflow)
    seg = [codec.segment_bytes(r)[0] for r in (0, 1)]
    if rows is None:
        rows, total = synth.segment_list(case, arm, seg)
    elif total is None:
        total = max([r[3] + seg[r[2]] for r in rows if r[2] <= 1 and r[3] < (1 << 32)] + [16])
    n = len(rows)
    d = oracle_descs(rows)
    host_layers = [host_bits(t) for t in case.layers]
    src = guarded_layers(case, device)
    dev_layers = [x.t for x in src]
    descs = _buffer(K.descriptors(rows, "cpu"), buffers, device)
    bufs = [Guarded(torch.full((max(total, 16),), SENTINEL_ENC, dtype=torch.uint8), buffers, device),
            Guarded(torch.full((max(n, 1),), 0xEE, dtype=torch.uint8), buffers, device),
            Guarded(torch.full((max(n, 1) * 32,), 0xEE, dtype=torch.uint8), buffers, device)]
    out, status, hdr = (x.t for x in bufs)
    codec.encode_sealed(dev_layers, descs, n, out, total, status, hdr)
    torch.cuda.synchronize()
    for k, x in enumerate(src):
        x.check(f"source layer {k}")
        assert np.array_equal(host_bits(x.t), host_layers[k]), f"encode wrote source layer {k}"
    for x, what in zip(bufs, ("slot buffer", "status array", "header array")):
        x.check(what)
    enc_ref, st_ref = O.encode(g, host_layers, d, total)
    hdr_ref = O.seal(g, d, enc_ref, st_ref)
    st_gpu = status[:n].cpu().numpy()
    assert np.array_equal(st_gpu, st_ref), f"status mismatch at {np.flatnonzero(st_gpu != st_ref)[:10]}"
    enc_gpu = out[:total].cpu().numpy()
    check_slot_gaps(enc_gpu, rows, seg, st_ref, "encode_sealed")
    for (layer, blk, role, off), s in zip(rows, st_ref):
        if s == O.S_ENCODED:
            assert np.array_equal(enc_gpu[off:off + seg[role]], enc_ref[off:off + seg[role]]), \
                f"slot (layer {layer}, block {blk}, role {role}) differs"
    got = hdr[:32 * n].cpu().numpy()
    want = hdr_ref.view(np.uint8)
    if not np.array_equal(got, want):
        bad = np.flatnonzero((got.reshape(n, 32) != want.reshape(n, 32)).any(axis=1))
        raise AssertionError(f"headers differ at segments {bad[:10]}: got {got.view(O.HEADER_DTYPE)[bad[:3]]} "
                             f"want {hdr_ref[bad[:3]]}")
    # verify + decode of the oracle's slots and headers, some damaged
    enc_bad = np.zeros(max(total, 16), dtype=np.uint8)
    enc_bad[:total] = enc_ref
    hdr_bad = hdr_ref.copy()
    coded = np.flatnonzero(st_ref == O.S_ENCODED)
    victims = np.random.default_rng(seed).choice(coded, size=min(tamper, coded.size), replace=False)
    for k, i in enumerate(victims):
        layer, blk, role, off = rows[i]
        if k % 2 == 0:
            enc_bad[off + (k * 977) % seg[role]] ^= 1 << (k % 8)
        else:
            hdr_bad[i][["crc32", "stored_bytes", "version", "format", "orig_bytes"][(k // 2) % 5]] ^= 1
    dst_g = guarded_layers(case, device)
    dst_dev = [x.t for x in dst_g]
    for t in dst_dev:
        t.view(torch.int16).fill_(SENTINEL_PAGE)
    dst_host = [np.full_like(h, SENTINEL_PAGE) for h in host_layers]
    enc_dev = _buffer(torch.from_numpy(enc_bad), buffers, device)
    hdr_dev = _buffer(torch.from_numpy(hdr_bad.view(np.uint8).copy()), buffers, device)
    result_g = Guarded(torch.full((max(n, 1),), 0xEE, dtype=torch.uint8), buffers, device)
    result = result_g.t
    codec.decode_verified(dst_dev, descs, n, enc_dev, total, hdr_dev, result)
    torch.cuda.synchronize()
    for k, x in enumerate(dst_g):
        x.check(f"restored layer {k}")
    result_g.check("result array")
    assert np.array_equal(enc_dev.cpu().numpy(), enc_bad), "decode wrote the slot buffer"
    ver = O.verify(g, d, enc_bad[:total], hdr_bad)
    res_ref = O.decode(g, dst_host, d, enc_bad[:total], ver)
    res = result[:n].cpu().numpy()
    assert np.array_equal(res, res_ref), f"results differ at {np.flatnonzero(res != res_ref)[:10]}"
    assert set(np.flatnonzero(res == O.S_CORRUPT).tolist()) == set(victims.tolist())
    for k, (a, b) in enumerate(zip(dst_dev, dst_host)):
        assert compare_pages(host_bits(a), b, f"layer tensor {k}") == 0
    codec.close()
    return st_ref, res
