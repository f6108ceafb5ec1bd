"""ctypes binding of the C ABI in ``include/kv_codec.h`` (argument marshalling only).

Every step of encode and decode runs in the CUDA kernels of ``libkvcodec.so``;
this module only turns Python arguments (torch tensors, ints, tuples) into the
pointers and sizes of the C calls.  There is no fallback: if the library has
not been built the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# KV_CODEC_DEBUG=1 loads the bounds-checked build (build(debug=True)) instead
LIB_PATH = os.path.join(_PKG, "libkvcodec_debug.so" if os.environ.get("KV_CODEC_DEBUG") == "1"
                        else "libkvcodec.so")
ABI_VERSION = 1
MAX_LAYERS = 512

# enums of include/kv_codec.h
DT = {"fp16": 1, "bf16": 2}
LAYOUT = {"separate": 1, "packed": 2}
CODEC = {"none": 0, "fp8_cast": 1, "fp8_fixed": 2, "fp8_dynamic": 3, "tq3": 4, "tq4": 5,
         "uni3": 6, "uni4": 7, "uni8": 8, "int8": 9, "tq2": 10, "uni2": 11}
SEG_ENCODED, SEG_RAW_NONFINITE, SEG_RAW_RANGE, SEG_RAW_PROTECTED = 1, 2, 3, 4
SEG_RAW_POLICY, SEG_RAW_OVERSIZE, SEG_RAW_NO_SAVING, SEG_BAD_DESC, SEG_CORRUPT = 5, 6, 7, 8, 9
# kv_segment_header
HEADER_DTYPE = np.dtype([("version", "<u4"), ("format", "<u4"), ("orig_bytes", "<u8"),
                         ("stored_bytes", "<u8"), ("crc32", "<u4"), ("status", "<u4")])

DESC_DTYPE = np.dtype([("layer", "<u4"), ("block", "<u4"), ("role", "<u4"),
                       ("reserved", "<u4"), ("enc_offset", "<u8")])

EXPORTS = ("kv_codec_create", "kv_codec_destroy", "kv_codec_segment_bytes", "kv_codec_encode",
           "kv_codec_decode", "kv_codec_seal", "kv_codec_verify", "kv_codec_strerror",
           "kv_codec_codebook", "kv_codec_signs", "kv_codec_layer_signs",
           "kv_codec_abi_version", "kv_codec_encode_sealed", "kv_codec_decode_verified")


class Geometry(C.Structure):
    _fields_ = [
        ("abi_version", C.c_uint32), ("struct_size", C.c_uint32), ("dtype", C.c_uint32),
        ("layout", C.c_uint32), ("head_dim", C.c_uint32), ("num_kv_heads", C.c_uint32),
        ("block_tokens", C.c_uint32), ("num_layers", C.c_uint32), ("num_blocks", C.c_uint64),
        ("stride_block", C.c_int64), ("stride_token", C.c_int64), ("stride_head", C.c_int64),
        ("k_codec", C.c_uint32), ("v_codec", C.c_uint32), ("protect_first", C.c_uint32),
        ("protect_last", C.c_uint32), ("rotation_seed", C.c_uint64), ("reject_abs", C.c_float),
        ("sign_version", C.c_uint32), ("fixed_amax", C.POINTER(C.c_float)),
        ("fixed_overflow", C.c_uint32), ("reserved", C.c_uint32),
    ]

FIXED_OVERFLOW = {"clip": 0, "reject": 1}


class KvCodecError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


_LIB = None


def lib():
    """Load libkvcodec.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m kv_cache_page_gb300.build` (nvcc, sm_103a)")
        L = C.CDLL(LIB_PATH)
        vp = C.c_void_p
        L.kv_codec_create.argtypes = [C.POINTER(Geometry), C.POINTER(vp)]
        L.kv_codec_destroy.argtypes = [vp]
        L.kv_codec_segment_bytes.argtypes = [vp, C.c_uint32, C.POINTER(C.c_uint64), C.POINTER(C.c_uint64)]
        L.kv_codec_encode.argtypes = [vp, C.POINTER(vp), C.c_uint32, vp, C.c_uint32, vp, C.c_uint64, vp, vp]
        L.kv_codec_decode.argtypes = [vp, C.POINTER(vp), C.c_uint32, vp, C.c_uint32, vp, C.c_uint64, vp,
                                      vp, vp]
        L.kv_codec_seal.argtypes = [vp, vp, C.c_uint32, vp, C.c_uint64, vp, vp, vp]
        L.kv_codec_verify.argtypes = [vp, vp, C.c_uint32, vp, C.c_uint64, vp, vp, vp]
        L.kv_codec_encode_sealed.argtypes = [vp, C.POINTER(vp), C.c_uint32, vp, C.c_uint32, vp, C.c_uint64,
                                             vp, vp, vp]
        L.kv_codec_decode_verified.argtypes = [vp, C.POINTER(vp), C.c_uint32, vp, C.c_uint32, vp,
                                               C.c_uint64, vp, vp, vp]
        L.kv_codec_strerror.argtypes = [C.c_int]
        L.kv_codec_strerror.restype = C.c_char_p
        L.kv_codec_codebook.argtypes = [C.c_uint32, C.c_uint32, C.POINTER(C.c_float), C.POINTER(C.c_float)]
        L.kv_codec_signs.argtypes = [C.c_uint64, C.c_uint32, C.POINTER(C.c_uint8)]
        L.kv_codec_layer_signs.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.POINTER(C.c_uint8)]
        L.kv_codec_abi_version.restype = C.c_uint32
        for f in ("kv_codec_create", "kv_codec_destroy", "kv_codec_segment_bytes", "kv_codec_encode",
                  "kv_codec_decode", "kv_codec_seal", "kv_codec_verify", "kv_codec_codebook",
                  "kv_codec_signs", "kv_codec_layer_signs"):
            getattr(L, f).restype = C.c_int
        _LIB = L
    return _LIB


def strerror(code: int) -> str:
    return lib().kv_codec_strerror(code).decode()


def _check(code: int, what: str):
    if code != 0:
        raise KvCodecError(code, what)


def codebook(bits: int, head_dim: int):
    cent = np.zeros(1 << bits, np.float32)
    bnd = np.zeros(1 << bits, np.float32)
    _check(lib().kv_codec_codebook(bits, head_dim, cent.ctypes.data_as(C.POINTER(C.c_float)),
                                   bnd.ctypes.data_as(C.POINTER(C.c_float))), "kv_codec_codebook")
    return cent, bnd[:-1].copy()


def signs(seed: int, head_dim: int):
    out = np.zeros(head_dim, np.uint8)
    _check(lib().kv_codec_signs(seed, head_dim, out.ctypes.data_as(C.POINTER(C.c_uint8))), "kv_codec_signs")
    return out


def layer_signs(seed: int, layer: int, head_dim: int):
    out = np.zeros(head_dim, np.uint8)
    _check(lib().kv_codec_layer_signs(seed, layer, head_dim, out.ctypes.data_as(C.POINTER(C.c_uint8))),
           "kv_codec_layer_signs")
    return out


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def descriptors(rows, device=None):
    """(layer, block, role, enc_offset) rows -> uint8 tensor of packed kv_segment_desc."""
    import torch
    d = np.zeros(len(rows), dtype=DESC_DTYPE)
    if len(rows):
        a = np.asarray(rows, dtype=np.uint64)
        d["layer"], d["block"], d["role"], d["enc_offset"] = a[:, 0], a[:, 1], a[:, 2], a[:, 3]
    t = torch.from_numpy(d.view(np.uint8).copy())
    return t.to(device) if device is not None else t


class Codec:
    """A registered KV geometry (one `kv_codec_t` handle)."""

    def __init__(self, *, dtype: str, layout: str, head_dim: int, num_kv_heads: int,
                 block_tokens: int, num_layers: int, num_blocks: int, strides: Sequence[int],
                 k_codec: str, v_codec: str, protect=(0, 0), rotation_seed: int = 0,
                 reject_abs: float = 448.0, fixed_amax=None, sign_version: int = 1,
                 fixed_overflow: str = "clip", geometry_overrides=None):
        g = Geometry()
        g.abi_version, g.struct_size = ABI_VERSION, C.sizeof(Geometry)
        g.dtype, g.layout = DT[dtype], LAYOUT[layout]
        g.head_dim, g.num_kv_heads, g.block_tokens = head_dim, num_kv_heads, block_tokens
        g.num_layers, g.num_blocks = num_layers, num_blocks
        g.stride_block, g.stride_token, g.stride_head = strides
        g.k_codec, g.v_codec = CODEC[k_codec], CODEC[v_codec]
        g.protect_first, g.protect_last = protect
        g.rotation_seed, g.reject_abs = rotation_seed, reject_abs
        g.sign_version = sign_version
        g.fixed_overflow = FIXED_OVERFLOW[fixed_overflow]
        self._amax = None
        if fixed_amax is not None:
            self._amax = np.ascontiguousarray(np.asarray(fixed_amax, dtype=np.float32).reshape(-1))
            g.fixed_amax = self._amax.ctypes.data_as(C.POINTER(C.c_float))
        for k, v in (geometry_overrides or {}).items():
            setattr(g, k, v)
        self.geometry = g
        self.layout = layout
        self.num_layers = num_layers
        h = C.c_void_p()
        _check(lib().kv_codec_create(C.byref(g), C.byref(h)), "kv_codec_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().kv_codec_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def segment_bytes(self, role: int):
        enc, raw = C.c_uint64(), C.c_uint64()
        _check(lib().kv_codec_segment_bytes(self._h, role, C.byref(enc), C.byref(raw)),
               "kv_codec_segment_bytes")
        return enc.value, raw.value

    def _layer_array(self, layers):
        n = len(layers)
        arr = (C.c_void_p * max(n, 1))()
        for i, t in enumerate(layers):
            arr[i] = _ptr(t)
        return arr, n

    def encode(self, layers, descs, n_segments: int, out, out_bytes: int, status, stream=None):
        """layers: list of device tensors (or pointers; separate: [K0, V0, ...], packed:
        one per layer); descs: uint8 tensor of descriptors; out / status: tensors.
        descs, out and status may be device or pinned host tensors (the kernel then
        writes the slots and statuses straight into host memory).  Enqueues on
        `stream` (default: torch's current stream)."""
        arr, n = self._layer_array(layers)
        _check(lib().kv_codec_encode(self._h, arr, n, _ptr(descs), n_segments, _ptr(out), out_bytes,
                                     _ptr(status), _stream_handle(stream)), "kv_codec_encode")

    def decode(self, layers, descs, n_segments: int, enc, enc_bytes: int, status, result=None,
               stream=None):
        """Restore ENCODED segments into `layers` (device tensors).  descs, enc, status
        and result may be device or pinned host tensors (the kernel then reads the slots
        from host memory itself).  Enqueues on `stream` (default: torch's current
        stream); make a consuming stream wait on an event recorded after it."""
        arr, n = self._layer_array(layers)
        _check(lib().kv_codec_decode(self._h, arr, n, _ptr(descs), n_segments, _ptr(enc), enc_bytes,
                                     _ptr(status), _ptr(result), _stream_handle(stream)),
               "kv_codec_decode")

    def seal(self, descs, n_segments: int, buf, buf_bytes: int, status, headers, stream=None):
        """One 32-byte kv_segment_header per descriptor into `headers` (a uint8 tensor
        of 32 * n bytes, or HEADER_DTYPE memory), CRC-32 of every ENCODED slot.
        Buffers: device or pinned host tensors."""
        _check(lib().kv_codec_seal(self._h, _ptr(descs), n_segments, _ptr(buf), buf_bytes, _ptr(status),
                                   _ptr(headers), _stream_handle(stream)), "kv_codec_seal")

    def encode_sealed(self, layers, descs, n_segments: int, out, out_bytes: int, status, headers,
                      stream=None):
        """encode followed by seal, in one pass over the slots when every coded role is
        FP8, uniform-8 or INT8 (the encoding warp checksums the slot it has just written)."""
        arr, n = self._layer_array(layers)
        _check(lib().kv_codec_encode_sealed(self._h, arr, n, _ptr(descs), n_segments, _ptr(out), out_bytes,
                                            _ptr(status), _ptr(headers), _stream_handle(stream)),
               "kv_codec_encode_sealed")

    def decode_verified(self, layers, descs, n_segments: int, enc, enc_bytes: int, headers, result,
                        stream=None):
        """verify followed by decode of the verified segments: result[i] as verify gives
        it (SEG_ENCODED once restored); a segment failing its header or CRC-32 check is
        SEG_CORRUPT and its page is left untouched.  One pass when every coded role is FP8,
        uniform-8 or INT8."""
        arr, n = self._layer_array(layers)
        _check(lib().kv_codec_decode_verified(self._h, arr, n, _ptr(descs), n_segments, _ptr(enc),
                                              enc_bytes, _ptr(headers), _ptr(result), _stream_handle(stream)),
               "kv_codec_decode_verified")

    def verify(self, descs, n_segments: int, buf, buf_bytes: int, headers, result, stream=None):
        """Check slots against their headers: result[i] = the header's status, or
        SEG_CORRUPT on a header or CRC-32 mismatch (a miss for decode)."""
        _check(lib().kv_codec_verify(self._h, _ptr(descs), n_segments, _ptr(buf), buf_bytes,
                                     _ptr(headers), _ptr(result), _stream_handle(stream)),
               "kv_codec_verify")
