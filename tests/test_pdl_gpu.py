"""Programmatic dependent launch of the decode (ekv_set_pdl), against the float64 oracle.

Back-to-back calls over several layers' caches overlap each call's prologue and first
page fills with the previous call's tail; every call must still match the oracle,
including batches with empty sequences (whose zero output is written only after the
grid-dependency wait) and one-page sequences (whose only page is a last page, fetched
after the wait). A cache-writer append launched between two calls writes the last page
of each sequence; the call after it must see the new token. The calls also replay from a
CUDA graph, where the programmatic launch becomes a programmatic edge.
"""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl
from oracle import writer as ow

from _helpers import assert_close, oracle_decode, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


LAYER_SETS = [
    # (lens, Hq, Hkv, D, v_format, scale_mode, extra)
    ([700, 0, 33, 1500, 16, 1, 250], 32, 8, 128, "e4m3", 0, {}),
    ([1200, 3, 17, 900, 1, 64, 2000, 5], 32, 4, 128, "mixed", 1, dict(p_compact=0.4, p_base=0.3)),
    ([300, 1, 45, 800], 16, 2, 64, "fp16", 0, {}),
]


@pytest.mark.parametrize("si", range(len(LAYER_SETS)))
def test_back_to_back_layers_match_the_oracle(ekv_lib, torch_cuda, si):
    torch = torch_cuda
    lens, hq, hkv, d, fmt, sm, kw = LAYER_SETS[si]
    layers = [wl.make_decode_case(lens, hq, hkv, d, v_format=fmt, scale_mode=sm, seed=500 + 10 * si + l,
                                  pool_pages=sum((x + 15) // 16 for x in lens) + 7, **kw)
              for l in range(4)]
    devs = [to_device(c) for c in layers]
    ctx = ekv_lib.Context(hq, hkv, d, len(lens), pdl=True)
    B = len(lens)
    outs = [torch.full((B, hq, d), float("nan"), dtype=torch.float16, device="cuda") for _ in layers]
    lses = [torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda") for _ in layers]
    refs = [oracle_decode(c) for c in layers]
    for rep in range(3):                              # the calls of all layers without a sync
        for dv, o, l in zip(devs, outs, lses):
            ctx.decode(dv, o, l)
        torch.cuda.synchronize()
        assert ctx.error() == (0, 0)
        for o, l, (ro, rl) in zip(outs, lses, refs):
            assert_close(o, l, ro, rl)
        empty = np.array(lens) == 0
        for o in outs:
            assert np.all(o.float().cpu().numpy()[empty] == 0)


def test_append_between_calls_is_seen(ekv_lib, torch_cuda):
    torch = torch_cuda
    hq, hkv, d = 32, 8, 128
    final = np.array([40, 16, 100, 17, 1, 64], np.int32)
    steps = 12
    cases = [wl.make_decode_case(final, hq, hkv, d, v_format="mixed", scale_mode=1, seed=600 + l,
                                 pool_pages=40, p_compact=0.4, p_base=0.2) for l in range(2)]
    devs = [to_device(c) for c in cases]
    ctx = ekv_lib.Context(hq, hkv, d, len(final), pdl=True)
    B = len(final)
    rng = np.random.default_rng(601)
    k_ref = [c.k_pages.copy() for c in cases]
    v_ref = [c.v_pages.copy() for c in cases]
    for s in range(steps):
        pos = np.maximum(final - steps + s, 0).astype(np.int32)       # the token of this step
        lens = pos + 1
        outs = []
        for l, (c, dv) in enumerate(zip(cases, devs)):
            dv.seq_lens.copy_(torch.from_numpy(lens))                    # the caller grows the lengths
            kn = rng.standard_normal((B, hkv, d)).astype(np.float16)
            vn = rng.standard_normal((B, hkv, d)).astype(np.float16)
            ekv_lib.ekv_append_kv(ctx.handle, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(),
                                  dv.k_pages, dv.v_pages, c.v_page_stride, c.num_pages, dv.v_scales,
                                  c.scale_mode, dv.page_mode, c.uniform_mode, dv.block_table,
                                  c.block_table.shape[1], torch.from_numpy(pos).cuda(), B)
            k_ref[l], v_ref[l] = ow.append_token(k_ref[l], v_ref[l], c.v_scales, c.scale_mode, c.page_mode,
                                                 c.uniform_mode, c.block_table, pos, kn, vn)
            o = torch.empty((B, hq, d), dtype=torch.float16, device="cuda")
            lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
            ctx.decode(dv, o, lse)                                       # right after the append
            outs.append((o, lse))
        torch.cuda.synchronize()
        assert ctx.error() == (0, 0)
        for l, c in enumerate(cases):
            ref = wl.DecodeCase(**{**c.__dict__})
            ref.k_pages, ref.v_pages, ref.seq_lens = k_ref[l], v_ref[l], lens
            ro, rl = oracle_decode(ref)
            assert_close(outs[l][0], outs[l][1], ro, rl)


def test_programmatic_edges_in_a_cuda_graph(ekv_lib, torch_cuda):
    torch = torch_cuda
    lens = [500, 0, 37, 1000, 1]
    layers = [wl.make_decode_case(lens, 32, 8, 128, v_format="mixed", scale_mode=1, seed=700 + l,
                                  pool_pages=sum((x + 15) // 16 for x in lens) + 5, p_compact=0.5)
              for l in range(3)]
    devs = [to_device(c) for c in layers]
    ctx = ekv_lib.Context(32, 8, 128, len(lens), pdl=True)
    outs = [torch.empty((len(lens), 32, 128), dtype=torch.float16, device="cuda") for _ in layers]
    lses = [torch.empty((len(lens), 32), dtype=torch.float32, device="cuda") for _ in layers]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for dv, o, l in zip(devs, outs, lses):
            ctx.decode(dv, o, l)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for dv, o, l in zip(devs, outs, lses):
            ctx.decode(dv, o, l)
    rng = np.random.default_rng(701)
    for rep in range(3):
        if rep:
            for c, dv in zip(layers, devs):
                c.q = rng.standard_normal(c.q.shape).astype(np.float16)
                dv.q.copy_(torch.from_numpy(c.q))
            torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert ctx.error() == (0, 0)
        for c, o, l in zip(layers, outs, lses):
            ro, rl = oracle_decode(c)
            assert_close(o, l, ro, rl)


def test_switch_values_and_the_cuda_core_consumer(ekv_lib, torch_cuda):
    # the switch takes 0 or 1 only; the CUDA-core consumer (variant 1) ignores it and runs
    # in plain stream order with the same results
    torch = torch_cuda
    ctx = ekv_lib.Context(32, 8, 128, 4, variant=1, pdl=True)
    assert ekv_lib.raw_status("ekv_set_pdl", ctx.handle, 2) == ekv_lib.EKV_ERR_INVALID_ARG
    lens = [300, 0, 17, 1000]
    case = wl.make_decode_case(lens, 32, 8, 128, v_format="mixed", scale_mode=1, seed=800,
                               pool_pages=sum((x + 15) // 16 for x in lens) + 3)
    dv = to_device(case)
    out = torch.empty((4, 32, 128), dtype=torch.float16, device="cuda")
    lse = torch.empty((4, 32), dtype=torch.float32, device="cuda")
    for _ in range(2):
        ctx.decode(dv, out, lse)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    ro, rl = oracle_decode(case)
    assert_close(out, lse, ro, rl)

