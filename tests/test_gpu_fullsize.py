"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (one encode and one decode call per codec arm over the whole
cache), checked on sampled segments that the oracle codes one by one: every
status of the sample, the encoded slot bytes and the restored pages.

Samples: the first and last segment, seeded random ones, and every segment the
GPU reported raw (the injected nonfinite / out-of-range ones)."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_parity import compare_pages, make_codec
from kv_cache_page_gb300 import codec as K
from kv_cache_page_gb300 import synth
from kvcases import host_bits, oracle_descs, oracle_geom

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_page_gb300 import build
    build.build()


def _page(case, layer, blk, role):
    """Host bits of one page of the tensor that holds (layer, role)."""
    t = case.layers[2 * layer + role] if case.layout == "separate" else case.layers[layer]
    return host_bits(t[blk])


def _check_arm(case, arm, n_random=40, seed=0):
    codec = make_codec(case, arm)
    seg = [codec.segment_bytes(r)[0] for r in (0, 1)]
    rows, total = synth.segment_list(case, arm, seg)
    n = len(rows)
    descs = K.descriptors(rows, "cuda")
    enc = torch.empty(total, dtype=torch.uint8, device="cuda")
    st = torch.empty(n, dtype=torch.uint8, device="cuda")
    codec.encode(case.layers, descs, n, enc, total, st)
    dst = [torch.empty_like(t) for t in case.layers]
    codec.decode(dst, descs, n, enc, total, st)
    torch.cuda.synchronize()
    st_h = st.cpu().numpy()
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(n, size=min(n_random, n), replace=False).tolist()) | {0, n - 1}
    pick |= set(np.flatnonzero(st_h != O.S_ENCODED)[:200].tolist())
    # oracle geometry of a single page: every sampled segment is block 0 of its own buffer
    one = synth.Case(case.name, case.dtype, case.layout, case.head_dim, case.num_heads,
                     case.block_tokens, case.num_layers, 1, case.strides, [], case.arms, case.seed,
                     case.fixed_amax)
    g = oracle_geom(one, arm)
    checked = 0
    for i in sorted(pick):
        layer, blk, role, off = rows[i]
        page = _page(case, layer, blk, role)
        ptrs = [None] * (2 * case.num_layers if case.layout == "separate" else case.num_layers)
        slot = 2 * layer + role if case.layout == "separate" else layer
        ptrs[slot] = page
        d = oracle_descs([(layer, 0, role, 0)])
        e_ref, s_ref = O.encode(g, ptrs, d, seg[role])
        assert st_h[i] == s_ref[0], (i, rows[i], st_h[i], s_ref[0])
        if s_ref[0] != O.S_ENCODED:
            continue
        got = enc[off:off + seg[role]].cpu().numpy()
        assert np.array_equal(got, e_ref), (i, rows[i])
        out = np.full_like(page, 0x7BCD)
        ptrs[slot] = out
        O.decode(g, ptrs, d, e_ref, s_ref)
        mine = host_bits(dst[2 * layer + role] if case.layout == "separate" else dst[layer])
        # dst holds the whole tensor; take this page's elements
        per_page = page.size
        mine = mine[blk * per_page:(blk + 1) * per_page]
        if case.layout == "packed":   # compare only this role's halves of the rows
            D = case.head_dim
            m = np.zeros(per_page, bool).reshape(-1, 2 * D)
            m[:, role * D:(role + 1) * D] = True
            m = m.reshape(-1)
            assert compare_pages(mine[m], out[m], f"segment {i}") == 0
        else:
            assert compare_pages(mine, out, f"segment {i}") == 0
        checked += 1
    codec.close()
    return checked, int(np.count_nonzero(st_h != O.S_ENCODED))


@pytest.mark.parametrize("name,kw", [("qwen3_8b", {}), ("vllm_packed", {}),
                                     ("head_dim_sweep", {"head_dim": 32}),
                                     ("head_dim_sweep", {"head_dim": 64}),
                                     ("head_dim_sweep", {"head_dim": 128}),
                                     ("head_dim_sweep", {"head_dim": 256}),
                                     ("qwen25_7b_offload", {}), ("hiq_qwen3_8b", {}),
                                     ("tiny", {})])
def test_full_size_sampled(name, kw):
    case = synth.make_case(name, device="cuda", **kw)
    for arm in case.arms:
        checked, raw = _check_arm(case, arm)
        assert checked > 0
        if name == "vllm_packed":
            assert raw > 0          # injected and protected segments are present
    del case
    torch.cuda.empty_cache()
