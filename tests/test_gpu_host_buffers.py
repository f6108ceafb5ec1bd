"""GPU parity of the host-resident path: descriptors, encoded slots, statuses and
results in pinned host memory, which the kernels read and write through its
device mapping (over NVLink-C2C on GB300).  Offload writes the slots straight
into host memory; restore reads them from there and scatters into the engine
pages ("Building a quantized HiCache for SGLang", section "CPU to GPU: restoration";
OrbitKV docs, "upload encoded bytes and GPU decode").

Same bar as the device-buffer parity tests: statuses, slots and results
bit-exact against the oracle, pages within 1 ulp (in fact exact).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from gpu_parity import SENTINEL_ENC, make_codec, run_parity
from kv_cache_page_gb300 import codec as K
from kv_cache_page_gb300 import synth

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_page_gb300 import build
    build.build()


@pytest.mark.parametrize("k,v", [("fp8_dynamic", "fp8_dynamic"), ("fp8_fixed", "fp8_cast"),
                                 ("tq4", "uni4"), ("tq3", "uni3"), ("uni8", "uni8"),
                                 ("none", "fp8_dynamic")])
def test_host_slots_qwen3_8b_shape(k, v):
    case = synth.make_case("qwen3_8b", num_layers=2, num_blocks=12)
    if "fp8_fixed" in (k, v):  # calibration maxima per (layer, role)
        g = torch.Generator().manual_seed(1)
        case = dataclasses.replace(case, fixed_amax=torch.rand(2, 2, generator=g) * 8 + 0.5)
    arm = synth.Arm(f"{k}/{v}", k, v, (0, 1), (0, 0))
    st, ulps = run_parity(case, arm, buffers="host")
    assert ulps == 0
    assert np.all(st[st != O.S_RAW_POLICY] == O.S_ENCODED)


def test_host_slots_int8_records():
    case = synth.make_case("hiq_qwen3_8b", num_layers=2, num_blocks=12)
    st, ulps = run_parity(case, case.arms[0], buffers="host")
    assert ulps == 0 and np.all(st == O.S_ENCODED)


def test_host_slots_packed_layout_with_raw_segments():
    case = synth.make_case("vllm_packed", num_layers=6, num_blocks=24)
    st, ulps = run_parity(case, case.arms[0], buffers="host")
    assert np.count_nonzero(st == O.S_RAW_PROTECTED) == 4 * 24 * 2
    assert np.count_nonzero(st == O.S_ENCODED) > 0
    assert ulps == 0


def _tiny_setup():
    case = synth.make_case("tiny")
    arm = case.arms[0]
    codec = make_codec(case, arm)
    seg = [codec.segment_bytes(r)[0] for r in (0, 1)]
    rows, total = synth.segment_list(case, arm, seg)
    layers = [t.cuda() for t in case.layers]
    return case, arm, codec, rows, total, layers


def test_host_and_device_slots_are_identical():
    """The same encode into a device buffer and into pinned host memory (statuses
    on the device, slots on the host, and the other way round)."""
    case, arm, codec, rows, total, layers = _tiny_setup()
    n = len(rows)
    descs = K.descriptors(rows, "cuda")
    out_d = torch.full((total,), SENTINEL_ENC, dtype=torch.uint8, device="cuda")
    st_d = torch.zeros(n, dtype=torch.uint8, device="cuda")
    codec.encode(layers, descs, n, out_d, total, st_d)
    out_h = torch.full((total,), SENTINEL_ENC, dtype=torch.uint8).pin_memory()
    st_h = torch.zeros(n, dtype=torch.uint8).pin_memory()
    descs_h = K.descriptors(rows, "cpu").pin_memory()  # referenced until the kernels finish
    codec.encode(layers, descs, n, out_h, total, st_d.clone())
    codec.encode(layers, descs_h, n, out_d.clone(), total, st_h)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu())
    assert torch.equal(st_h, st_d.cpu())
    codec.close()


def test_pageable_host_buffer_is_refused():
    case, arm, codec, rows, total, layers = _tiny_setup()
    n = len(rows)
    descs = K.descriptors(rows, "cuda")
    st = torch.zeros(n, dtype=torch.uint8, device="cuda")
    pageable = torch.full((total,), SENTINEL_ENC, dtype=torch.uint8)
    assert not pageable.is_pinned()
    with pytest.raises(K.KvCodecError) as ei:
        codec.encode(layers, descs, n, pageable, total, st)
    assert ei.value.code == -9
    with pytest.raises(K.KvCodecError) as ei:
        codec.decode(layers, descs, n, pageable, total, st)
    assert ei.value.code == -9
    torch.cuda.synchronize()
    assert torch.all(pageable == SENTINEL_ENC)  # nothing ran
    codec.close()


def test_restore_on_transfer_stream_orders_before_consumer():
    """Restore from host slots on a side (transfer) stream, record an event, and
    let the default stream consume the pages after waiting on it: the consumer
    sees the restored values, never the sentinel it wrote before."""
    case, arm, codec, rows, total, layers = _tiny_setup()
    n = len(rows)
    descs = K.descriptors(rows, "cuda")
    enc = torch.empty(total, dtype=torch.uint8, device="cuda")
    st = torch.empty(n, dtype=torch.uint8, device="cuda")
    codec.encode(layers, descs, n, enc, total, st)
    ref = [torch.empty_like(t) for t in layers]
    codec.decode(ref, descs, n, enc, total, st)
    torch.cuda.synchronize()
    enc_h, st_h = enc.cpu().pin_memory(), st.cpu().pin_memory()
    descs_h = K.descriptors(rows, "cpu").pin_memory()
    transfer = torch.cuda.Stream()
    for trial in range(4):
        dst = [torch.full_like(t, 7.0) for t in layers]
        torch.cuda.synchronize()
        with torch.cuda.stream(transfer):
            codec.decode(dst, descs_h, n, enc_h, total, st_h, stream=transfer)
            ready = torch.cuda.Event()
            ready.record(transfer)
        torch.cuda.current_stream().wait_event(ready)
        sums = [(d.float() - r.float()).abs().sum() for d, r in zip(dst, ref)]
        assert all(float(s) == 0.0 for s in sums), trial
    codec.close()


def test_layer_chunks_pipelined_over_streams_match_one_call():
    """Offload + restore in chunks of layers, chunk c on stream c % 3 (pages
    H2D, encode into pinned host slots, decode from them, pages D2H), as a
    pipelined offload path would run it: slots, statuses and restored pages
    equal those of one call over all segments."""
    case = synth.make_case("qwen3_8b", num_layers=7, num_blocks=10)
    arm = case.arms[1]
    codec = make_codec(case, arm)
    seg = [codec.segment_bytes(r)[0] for r in (0, 1)]
    rows, total = synth.segment_list(case, arm, seg)
    n = len(rows)
    layers = [t.cuda() for t in case.layers]
    # one call, device buffers
    descs = K.descriptors(rows, "cuda")
    enc1 = torch.zeros(total, dtype=torch.uint8, device="cuda")
    st1 = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out1 = [torch.zeros_like(t) for t in layers]
    codec.encode(layers, descs, n, enc1, total, st1)
    codec.decode(out1, descs, n, enc1, total, st1)
    torch.cuda.synchronize()
    # chunks of 3 layers on 3 streams, pages staged through pinned host memory
    src_h = [t.cpu().pin_memory() for t in case.layers]
    dst_h = [torch.zeros_like(t).pin_memory() for t in case.layers]
    src_d = [torch.zeros_like(t) for t in layers]
    dst_d = [torch.zeros_like(t) for t in layers]
    enc_h = torch.zeros(total, dtype=torch.uint8).pin_memory()
    st_h = torch.zeros(n, dtype=torch.uint8).pin_memory()
    streams = [torch.cuda.Stream() for _ in range(3)]
    torch.cuda.synchronize()
    lay = [r[0] for r in rows]
    for c, l0 in enumerate(range(0, case.num_layers, 3)):
        group = range(l0, min(l0 + 3, case.num_layers))
        d0, d1 = lay.index(group[0]), len(lay) - lay[::-1].index(group[-1])
        idx = [2 * l + r for l in group for r in (0, 1)]
        s = streams[c % 3]
        with torch.cuda.stream(s):
            for i in idx:
                src_d[i].copy_(src_h[i], non_blocking=True)
            codec.encode(src_d, descs[d0 * 24:d1 * 24], d1 - d0, enc_h, total, st_h[d0:d1], stream=s)
            codec.decode(dst_d, descs[d0 * 24:d1 * 24], d1 - d0, enc_h, total, st_h[d0:d1], stream=s)
            for i in idx:
                dst_h[i].copy_(dst_d[i], non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(st_h, st1.cpu())
    assert torch.equal(enc_h, enc1.cpu())
    for a, b in zip(dst_h, out1):
        assert torch.equal(a.view(torch.int16), b.cpu().view(torch.int16))
    codec.close()
