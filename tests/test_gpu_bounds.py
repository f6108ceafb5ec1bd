"""The bounds-checked debug library on the GPU (libkvcodec_debug.so, built
from the same sources with -DKVC_BOUNDS_CHECK).

Every global load and store of its kernels is checked against the buffers the
call was given (layer tensors, slot buffer, descriptors, statuses, results,
headers); an access outside them is skipped and the call returns
KV_ERR_INTERNAL.  (1) Parity cases covering every kernel family, both layouts,
every head dim, ragged last steps, full 512-vector segments, host-resident
buffers, invalid descriptors, the CRC passes and the one-pass integrity
kernels run through the debug library in a child process: results equal the
oracle's and no call reports an access outside its buffers.  (2) With the
check's slot-buffer range cut short (KVC_DEBUG_SLOT_MARGIN), the call whose
last slot ends at the buffer's end reports KV_ERR_INTERNAL and leaves the held
back bytes unwritten.  The accesses it flags are in bounds in fact, so nothing
out of range is touched."""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_page_gb300 import build
    build.build(debug=True)


def _child(body, **env):
    """Run PRELUDE + body in a child process that loads the debug library."""
    e = dict(os.environ, KV_CODEC_DEBUG="1",
             PYTHONPATH=os.pathsep.join([os.path.join(ROOT, "tests"), ROOT]), **env)
    r = subprocess.run([sys.executable, "-c", PRELUDE + textwrap.dedent(body)], cwd=ROOT, env=e,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"child failed:\n{r.stdout[-3000:]}\n{r.stderr[-3000:]}"
    return r.stdout


PRELUDE = """
import numpy as np
import torch
import oracle as O
from kv_cache_page_gb300 import codec, synth
from gpu_parity import run_parity, run_seal_parity, run_sealed_parity
from kvcases import custom_case
assert codec.LIB_PATH.endswith("libkvcodec_debug.so"), codec.LIB_PATH
"""


def test_parity_cases_stay_inside_their_buffers():
    out = _child("""
    n = 0
    # the workloads' own arms (planted raw segments, protected layers)
    for name, kw in (("tiny", {}), ("vllm_packed", dict(num_layers=5, num_blocks=3)),
                     ("hiq_qwen3_8b", dict(num_layers=1, num_blocks=4)),
                     ("qwen25_7b_offload", dict(num_layers=5, num_blocks=3)),
                     ("qwen3_8b", dict(num_layers=2, num_blocks=4))):
        c = synth.make_case(name, **kw)
        for arm in c.arms:
            run_parity(c, arm)
            n += 1
    # every family at every head dim, ragged steps (H = 3, T = 5), both layouts
    for D in (32, 64, 128, 256):
        for kc, vc in (("tq4", "uni4"), ("tq3", "uni3"), ("tq2", "uni2"), ("fp8_fixed", "uni8"),
                       ("fp8_dynamic", "fp8_cast"), ("int8", "int8")):
            for layout in ("separate", "packed"):
                case = custom_case(D=D, H=3, T=5, L=3, B=4, dtype="bf16", layout=layout, seed=D)
                run_parity(case, synth.Arm("dbg", kc, vc, (0, 1)))
                n += 1
    # 512-vector segments: the adjacent-chunk decoders and multi-step segments
    for kc, vc in (("fp8_dynamic", "fp8_fixed"), ("uni8", "uni4"), ("tq4", "uni2")):
        case = custom_case(D=128, H=16, T=32, L=2, B=3, dtype="fp16", layout="separate", seed=3)
        run_parity(case, synth.Arm("full", kc, vc, (0, 1)))
        n += 1
    # host-resident descriptors, slots, statuses and results
    c = synth.make_case("tiny")
    for arm in c.arms:
        run_parity(c, arm, buffers="host")
        n += 1
    # invalid descriptors among valid ones
    case = custom_case(D=64, H=4, T=8, L=3, B=4, dtype="fp16", layout="separate", seed=9)
    arm = synth.Arm("bad", "fp8_dynamic", "uni8", (0, 1))
    from gpu_parity import make_codec
    cd = make_codec(case, arm)
    slot = max(cd.segment_bytes(0)[0], cd.segment_bytes(1)[0])
    cd.close()
    rows = [(1, 2, 0, 0), (7, 0, 0, slot), (1, 9, 1, 2 * slot), (1, 1, 2, 3 * slot), (1, 3, 1, 4 * slot + 8),
            (2, 0, 1, 40 * slot), (1, 0, 1, 5 * slot)]
    run_parity(case, arm, rows=rows, total=6 * slot)
    n += 1
    # the CRC passes and the one-pass integrity kernels (FP8, uniform-8, two-pass route)
    c = synth.make_case("tiny")
    run_seal_parity(c, c.arms[0])
    for arm in (synth.Arm("s8", "fp8_dynamic", "fp8_cast", (0, 1)), synth.Arm("su", "uni8", "uni8", (0, 1)),
                synth.Arm("si", "int8", "int8", (0, 1)), synth.Arm("s2", "tq3", "fp8_cast", (0, 1))):
        case = custom_case(D=128, H=4, T=16, L=3, B=4, dtype="bf16", layout="separate", seed=5)
        run_sealed_parity(case, arm, tamper=2)
        n += 3
    print("cases", n)
    """)
    assert "cases" in out


def test_held_back_slot_bytes_are_reported_and_left_unwritten():
    """The check's slot range ends 64 bytes before the buffer does: encode of a
    call whose last slot reaches the buffer's end and decode of it both report
    KV_ERR_INTERNAL; the held back bytes keep their sentinel."""
    _child("""
    from gpu_parity import make_codec
    case = synth.make_case("tiny")
    arm = case.arms[0]
    cd = make_codec(case, arm)
    seg = [cd.segment_bytes(r)[0] for r in (0, 1)]
    rows, total = synth.segment_list(case, arm, seg)
    assert max(r[3] + seg[r[2]] for r in rows) == total
    layers = [t.cuda() for t in case.layers]
    descs = codec.descriptors(rows, "cuda")
    out = torch.full((total,), 0xA5, dtype=torch.uint8, device="cuda")
    status = torch.zeros(len(rows), dtype=torch.uint8, device="cuda")
    try:
        cd.encode(layers, descs, len(rows), out, total, status)
        raise SystemExit("encode reported nothing")
    except codec.KvCodecError as e:
        assert e.code == -11, e
    torch.cuda.synchronize()
    assert torch.all(out[total - 64:] == 0xA5), "a flagged store was performed"
    assert not torch.all(out[: total - 64] == 0xA5), "the rest was not encoded"
    dst = [torch.zeros_like(t) for t in layers]
    try:
        cd.decode(dst, descs, len(rows), out, total, status)
        raise SystemExit("decode reported nothing")
    except codec.KvCodecError as e:
        assert e.code == -11, e
    cd.close()
    print("flagged")
    """, KVC_DEBUG_SLOT_MARGIN="64")
