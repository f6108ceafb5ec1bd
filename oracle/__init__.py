"""Plain CPU oracle of the KV-page codec (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product path never does.  It
shares no code with the CUDA codec in ``kv_cache_page_gb300``: the arithmetic
lives in ``kvoracle.c`` (plain scalar C, one IEEE operation at a time), and this
module only marshals numpy arrays into it.

Functions without an independent pin are marked "parity unpinned" in their
docstrings (none at present; see the tests under ``tests/test_oracle_*``).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvoracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_LIB = None

# Interface numbers (written independently of the product's header).
FP16, BF16 = 1, 2
SEPARATE, PACKED = 1, 2
NONE, FP8_CAST, FP8_FIXED, FP8_DYNAMIC, TQ3, TQ4, UNI3, UNI4, UNI8, INT8, TQ2, UNI2 = range(12)
(S_ENCODED, S_RAW_NONFINITE, S_RAW_RANGE, S_RAW_PROTECTED, S_RAW_POLICY,
 S_RAW_OVERSIZE, S_RAW_NO_SAVING, S_BAD_DESC, S_CORRUPT) = range(1, 10)
# segment header {u32 version, u32 format, u64 orig_bytes, u64 stored_bytes, u32 crc32, u32 status}
HEADER_DTYPE = np.dtype([("version", "<u4"), ("format", "<u4"), ("orig_bytes", "<u8"),
                         ("stored_bytes", "<u8"), ("crc32", "<u4"), ("status", "<u4")])


def build(force: bool = False) -> str:
    """Compile kvoracle.c with gcc (no FMA contraction, no fast-math)."""
    with _lock:
        if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
            tmp = _SO + f".{os.getpid()}.tmp"
            subprocess.check_call([
                "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _SO)
    return _SO


class Geom(C.Structure):
    _fields_ = [
        ("dtype", C.c_int32), ("layout", C.c_int32), ("head_dim", C.c_int32),
        ("num_heads", C.c_int32), ("block_tokens", C.c_int32), ("num_layers", C.c_int32),
        ("num_blocks", C.c_int64), ("stride_block", C.c_int64), ("stride_token", C.c_int64),
        ("stride_head", C.c_int64), ("codec", C.c_int32 * 2), ("protect_first", C.c_int32),
        ("protect_last", C.c_int32), ("seed", C.c_uint64), ("reject_abs", C.c_float),
        ("sign_version", C.c_int32), ("fixed_amax", C.POINTER(C.c_float)),
        ("fixed_overflow", C.c_int32), ("reserved", C.c_int32),
    ]


DESC_DTYPE = np.dtype([("layer", "<u4"), ("block", "<u4"), ("role", "<u4"),
                       ("reserved", "<u4"), ("enc_offset", "<u8")])

_P = np.ctypeslib.ndpointer
_f32 = _P(np.float32, flags="C")
_u16 = _P(np.uint16, flags="C")
_u8 = _P(np.uint8, flags="C")
_f64 = _P(np.float64, flags="C")
_i8 = _P(np.int8, flags="C")


def lib():
    global _LIB
    if _LIB is None:
        L = C.CDLL(build())
        sig = {
            "kvo_f16_to_f32_array": [_u16, C.c_int64, _f32],
            "kvo_bf16_to_f32_array": [_u16, C.c_int64, _f32],
            "kvo_f32_to_f16_array": [_f32, C.c_int64, _u16],
            "kvo_f32_to_bf16_array": [_f32, C.c_int64, _u16],
            "kvo_f32_to_e4m3_array": [_f32, C.c_int64, _u8],
            "kvo_e4m3_to_f32_array": [_u8, C.c_int64, _f32],
            "kvo_pairwise_sum": [_f32, C.c_int],
            "kvo_fp8_scale_from_amax": [C.c_float],
            "kvo_absmax": [_f32, C.c_int],
            "kvo_fp8_encode_many": [_f32, C.c_int64, C.c_int, _f32, _u8],
            "kvo_signs": [C.c_uint64, C.c_int, _u8],
            "kvo_signs_layer": [C.c_uint64, C.c_int, C.c_int, _u8],
            "kvo_tq_encode_many_signs": [_f32, C.c_int64, C.c_int, C.c_int, _u8, _u8, _u16],
            "kvo_tq_decode_many_signs": [_u8, _u16, C.c_int64, C.c_int, C.c_int, _u8, _f32],
            "kvo_splitmix64_next": [C.POINTER(C.c_uint64)],
            "kvo_wht": [_f32, C.c_int],
            "kvo_wht_scale": [C.c_int],
            "kvo_lloyd_max_gauss": [C.c_int, _f64],
            "kvo_codebook": [C.c_int, C.c_int, _f32, _f32],
            "kvo_tq_encode_many": [_f32, C.c_int64, C.c_int, C.c_int, C.c_uint64, _u8, _u16],
            "kvo_tq_decode_many": [_u8, _u16, C.c_int64, C.c_int, C.c_int, C.c_uint64, _f32],
            "kvo_uniform_encode_many": [_f32, C.c_int64, C.c_int, C.c_int, _u8, _u16, _u16],
            "kvo_uniform_decode_many": [_u8, _u16, _u16, C.c_int64, C.c_int, _f32],
            "kvo_tq_index_many": [_f32, C.c_int64, C.c_int, C.c_int, _u8],
            "kvo_int8_scale": [C.c_float],
            "kvo_int8_encode_many": [_f32, C.c_int64, C.c_int, _i8, _u16],
            "kvo_int8_decode_many": [_i8, _u16, C.c_int64, C.c_int, _f32],
            "kvo_int8_record_bytes": [C.c_int, C.c_int],
            "kvo_crc32": [C.c_void_p, C.c_uint64],
            "kvo_seal": [C.POINTER(Geom), C.c_void_p, C.c_uint32, C.c_void_p, C.c_uint64,
                         C.c_void_p, C.c_void_p],
            "kvo_verify": [C.POINTER(Geom), C.c_void_p, C.c_uint32, C.c_void_p, C.c_uint64,
                           C.c_void_p, C.c_void_p],
            "kvo_pack_bits": [_u8, C.c_int, C.c_int, _u8],
            "kvo_unpack_bits": [_u8, C.c_int, C.c_int, _u8],
            "kvo_segment_enc_bytes": [C.POINTER(Geom), C.c_int],
            "kvo_segment_raw_bytes": [C.POINTER(Geom)],
            "kvo_encode": [C.POINTER(Geom), C.POINTER(C.c_void_p), C.c_void_p, C.c_uint32,
                           C.c_void_p, C.c_uint64, C.c_void_p],
            "kvo_decode": [C.POINTER(Geom), C.POINTER(C.c_void_p), C.c_void_p, C.c_uint32,
                           C.c_void_p, C.c_uint64, C.c_void_p, C.c_void_p],
        }
        res = {"kvo_pairwise_sum": C.c_float, "kvo_fp8_scale_from_amax": C.c_float,
               "kvo_absmax": C.c_float, "kvo_wht_scale": C.c_float,
               "kvo_splitmix64_next": C.c_uint64, "kvo_segment_enc_bytes": C.c_int64,
               "kvo_segment_raw_bytes": C.c_int64, "kvo_int8_scale": C.c_uint16,
               "kvo_int8_record_bytes": C.c_int64, "kvo_crc32": C.c_uint32}
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res.get(name, None)
        _LIB = L
    return _LIB


# ---------------------------------------------------------------- scalars
def _arr(fn, x, in_dt, out_dt):
    x = np.ascontiguousarray(x, dtype=in_dt)
    out = np.empty(x.shape, dtype=out_dt)
    getattr(lib(), fn)(x.reshape(-1), x.size, out.reshape(-1))
    return out


def f16_to_f32(bits):  return _arr("kvo_f16_to_f32_array", bits, np.uint16, np.float32)
def bf16_to_f32(bits): return _arr("kvo_bf16_to_f32_array", bits, np.uint16, np.float32)
def f32_to_f16(x):     return _arr("kvo_f32_to_f16_array", x, np.float32, np.uint16)
def f32_to_bf16(x):    return _arr("kvo_f32_to_bf16_array", x, np.float32, np.uint16)
def f32_to_e4m3(x):    return _arr("kvo_f32_to_e4m3_array", x, np.float32, np.uint8)
def e4m3_to_f32(c):    return _arr("kvo_e4m3_to_f32_array", c, np.uint8, np.float32)


def src_to_f32(bits, dtype):
    return f16_to_f32(bits) if dtype == FP16 else bf16_to_f32(bits)


def f32_to_src(x, dtype):
    return f32_to_f16(x) if dtype == FP16 else f32_to_bf16(x)


def pairwise_sum(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return np.float32(lib().kvo_pairwise_sum(a, a.size))


def fp8_scale_from_amax(amax):
    return np.float32(lib().kvo_fp8_scale_from_amax(float(amax)))


def absmax(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return np.float32(lib().kvo_absmax(x, x.size))


def fp8_encode(x, scales):
    """x: [nvec, D] float32, scales: [nvec] float32 -> codes [nvec, D] uint8."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.ascontiguousarray(scales, dtype=np.float32).reshape(-1)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().kvo_fp8_encode_many(x.reshape(-1), x.shape[0], x.shape[1], s, out.reshape(-1))
    return out


def signs(seed, D):
    out = np.empty(D, dtype=np.uint8)
    lib().kvo_signs(seed, D, out)
    return out


def signs_layer(seed, layer, D):
    """Format version 2: the sign vector of one layer."""
    out = np.empty(D, dtype=np.uint8)
    lib().kvo_signs_layer(seed, layer, D, out)
    return out


def splitmix64(seed, n):
    st = C.c_uint64(seed)
    return [lib().kvo_splitmix64_next(C.byref(st)) for _ in range(n)]


def wht(a):
    a = np.array(a, dtype=np.float32, copy=True)
    lib().kvo_wht(a, a.size)
    return a


def wht_scale(D):
    return np.float32(lib().kvo_wht_scale(D))


def lloyd_max_gauss(bits):
    c = np.empty(1 << bits, dtype=np.float64)
    lib().kvo_lloyd_max_gauss(bits, c)
    return c


def codebook(bits, D):
    cent = np.empty(1 << bits, dtype=np.float32)
    bnd = np.zeros(1 << bits, dtype=np.float32)
    lib().kvo_codebook(bits, D, cent, bnd)
    return cent, bnd[: (1 << bits) - 1].copy()


def tq_index(y, bits, D):
    """Centroid index of each value of y (already in the rotated, unit-norm domain)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    lib().kvo_tq_index_many(y.reshape(-1), y.size, bits, D, out.reshape(-1))
    return out


def tq_encode(x, bits, seed):
    x = np.ascontiguousarray(x, dtype=np.float32)
    nvec, D = x.shape
    codes = np.empty((nvec, D), dtype=np.uint8)
    norm = np.empty(nvec, dtype=np.uint16)
    lib().kvo_tq_encode_many(x.reshape(-1), nvec, D, bits, seed, codes.reshape(-1), norm)
    return codes, norm


def tq_encode_with_signs(x, bits, neg):
    x = np.ascontiguousarray(x, dtype=np.float32)
    nvec, D = x.shape
    codes = np.empty((nvec, D), dtype=np.uint8)
    norm = np.empty(nvec, dtype=np.uint16)
    lib().kvo_tq_encode_many_signs(x.reshape(-1), nvec, D, bits, np.ascontiguousarray(neg, dtype=np.uint8),
                                   codes.reshape(-1), norm)
    return codes, norm


def tq_decode_with_signs(codes, norm16, bits, neg):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    nvec, D = codes.shape
    out = np.empty((nvec, D), dtype=np.float32)
    lib().kvo_tq_decode_many_signs(codes.reshape(-1), np.ascontiguousarray(norm16, dtype=np.uint16), nvec,
                                   D, bits, np.ascontiguousarray(neg, dtype=np.uint8), out.reshape(-1))
    return out


def tq_decode(codes, norm16, bits, seed):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    nvec, D = codes.shape
    out = np.empty((nvec, D), dtype=np.float32)
    lib().kvo_tq_decode_many(codes.reshape(-1), np.ascontiguousarray(norm16, dtype=np.uint16),
                             nvec, D, bits, seed, out.reshape(-1))
    return out


def uniform_encode(x, bits):
    x = np.ascontiguousarray(x, dtype=np.float32)
    nvec, D = x.shape
    codes = np.empty((nvec, D), dtype=np.uint8)
    m16 = np.empty(nvec, dtype=np.uint16)
    s16 = np.empty(nvec, dtype=np.uint16)
    lib().kvo_uniform_encode_many(x.reshape(-1), nvec, D, bits, codes.reshape(-1), m16, s16)
    return codes, m16, s16


def uniform_decode(codes, m16, s16):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    nvec, D = codes.shape
    out = np.empty((nvec, D), dtype=np.float32)
    lib().kvo_uniform_decode_many(codes.reshape(-1), np.ascontiguousarray(m16, dtype=np.uint16),
                                  np.ascontiguousarray(s16, dtype=np.uint16), nvec, D,
                                  out.reshape(-1))
    return out


def int8_scale(amax) -> int:
    """BF16 bits of the per-head INT8 scale for an absolute maximum."""
    return int(lib().kvo_int8_scale(float(np.float32(amax))))


def int8_encode(x):
    """[HIQ "Building the INT8 codec"]: int8 codes and BF16 scale bits per row."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    nvec, D = x.shape
    codes = np.empty((nvec, D), dtype=np.int8)
    s16 = np.empty(nvec, dtype=np.uint16)
    lib().kvo_int8_encode_many(x.reshape(-1), nvec, D, codes.reshape(-1), s16)
    return codes, s16


def int8_decode(codes, s16):
    """code * scale in FP32 (exact); the caller rounds to BF16."""
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    nvec, D = codes.shape
    out = np.empty((nvec, D), dtype=np.float32)
    lib().kvo_int8_decode_many(codes.reshape(-1), np.ascontiguousarray(s16, dtype=np.uint16),
                               nvec, D, out.reshape(-1))
    return out


def int8_record_bytes(H, D) -> int:
    return int(lib().kvo_int8_record_bytes(H, D))


def pack_bits(codes, bits):
    codes = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1)
    out = np.zeros((codes.size * bits + 7) // 8, dtype=np.uint8)
    lib().kvo_pack_bits(codes, codes.size, bits, out)
    return out


def unpack_bits(packed, n, bits):
    packed = np.ascontiguousarray(packed, dtype=np.uint8).reshape(-1)
    out = np.empty(n, dtype=np.uint8)
    lib().kvo_unpack_bits(packed, n, bits, out)
    return out


# ---------------------------------------------------------------- segments
def make_geom(*, dtype, layout, head_dim, num_heads, block_tokens, num_layers, num_blocks,
              strides, codecs, protect=(0, 0), seed=0, reject_abs=448.0, fixed_amax=None,
              sign_version=1, fixed_overflow=0):
    """Build the oracle's geometry.  `strides` = (block, token, head) in elements;
    `fixed_amax` = float32 [num_layers, 2] calibration absmax (FP8 fixed mode);
    `sign_version` 1: one TurboQuant sign vector per (seed, head dim), 2: one
    per layer as well (format version 2); `fixed_overflow` 0: FP8 fixed-scale
    quotients beyond +-448 are clipped, 1: such a segment stays raw."""
    g = Geom()
    g.dtype, g.layout, g.head_dim = dtype, layout, head_dim
    g.num_heads, g.block_tokens, g.num_layers = num_heads, block_tokens, num_layers
    g.num_blocks = num_blocks
    g.stride_block, g.stride_token, g.stride_head = strides
    g.codec[0], g.codec[1] = codecs
    g.protect_first, g.protect_last = protect
    g.seed = seed
    g.sign_version = sign_version
    g.fixed_overflow = fixed_overflow
    g.reject_abs = reject_abs
    if fixed_amax is not None:
        fa = np.ascontiguousarray(fixed_amax, dtype=np.float32).reshape(-1)
        g._keep = fa
        g.fixed_amax = fa.ctypes.data_as(C.POINTER(C.c_float))
    return g


def segment_enc_bytes(g, role):
    return int(lib().kvo_segment_enc_bytes(C.byref(g), role))


def segment_raw_bytes(g):
    return int(lib().kvo_segment_raw_bytes(C.byref(g)))


def _ptrs(layers):
    arr = (C.c_void_p * len(layers))()
    for i, a in enumerate(layers):
        arr[i] = None if a is None else a.ctypes.data
    return arr


def encode(g, layers, descs, out_bytes, out=None):
    """layers: list of uint16 numpy arrays (raw 16-bit patterns); for the
    separate layout [K0, V0, K1, V1, ...], for the packed layout one per layer.
    Returns (encoded buffer uint8[out_bytes], status uint8[n])."""
    descs = np.ascontiguousarray(descs, dtype=DESC_DTYPE)
    if out is None:
        out = np.zeros(out_bytes, dtype=np.uint8)
    status = np.zeros(len(descs), dtype=np.uint8)
    lib().kvo_encode(C.byref(g), _ptrs(layers), descs.ctypes.data, len(descs),
                     out.ctypes.data, out_bytes, status.ctypes.data)
    return out, status


def decode(g, layers, descs, enc, status):
    """Restores ENCODED segments into `layers` (modified in place); returns the
    per-segment result codes."""
    descs = np.ascontiguousarray(descs, dtype=DESC_DTYPE)
    enc = np.ascontiguousarray(enc, dtype=np.uint8)
    status = np.ascontiguousarray(status, dtype=np.uint8)
    result = np.zeros(len(descs), dtype=np.uint8)
    lib().kvo_decode(C.byref(g), _ptrs(layers), descs.ctypes.data, len(descs),
                     enc.ctypes.data, enc.size, status.ctypes.data, result.ctypes.data)
    return result


# ---------------------------------------------------------------- headers
def crc32(data) -> int:
    """CRC-32 (reflected 0xEDB88320, preset and final complement), bit-serial."""
    b = np.ascontiguousarray(np.frombuffer(bytes(data), np.uint8) if isinstance(data, (bytes, bytearray))
                             else data, dtype=np.uint8).reshape(-1)
    return int(lib().kvo_crc32(b.ctypes.data if b.size else None, b.size))


def seal(g, descs, buf, status):
    """Segment headers (HEADER_DTYPE[n]) for the slots in `buf`."""
    descs = np.ascontiguousarray(descs, dtype=DESC_DTYPE)
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    status = np.ascontiguousarray(status, dtype=np.uint8)
    out = np.zeros(len(descs), dtype=HEADER_DTYPE)
    lib().kvo_seal(C.byref(g), descs.ctypes.data, len(descs), buf.ctypes.data, buf.size,
                   status.ctypes.data, out.ctypes.data)
    return out


def verify(g, descs, buf, headers):
    """Per-segment result: the header's status when header and checksum hold,
    S_CORRUPT when not, S_BAD_DESC for an invalid descriptor."""
    descs = np.ascontiguousarray(descs, dtype=DESC_DTYPE)
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    headers = np.ascontiguousarray(headers, dtype=HEADER_DTYPE)
    out = np.zeros(len(descs), dtype=np.uint8)
    lib().kvo_verify(C.byref(g), descs.ctypes.data, len(descs), buf.ctypes.data, buf.size,
                     headers.ctypes.data, out.ctypes.data)
    return out
