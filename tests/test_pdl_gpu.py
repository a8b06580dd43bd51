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



def _decode_into(ekv_lib, ctx, case, d, v, mode, scales, out, lse, stream):
    ekv_lib.ekv_paged_decode(ctx.handle, d.q, d.k_pages, v, case.v_page_stride, case.num_pages, scales,
                             case.scale_mode, mode, case.uniform_mode, d.block_table,
                             case.block_table.shape[1], d.seq_lens, case.batch, 0.0, out, lse, stream)


def _reps_match(outs, lses, ref):
    ro, rl = ref
    for o, l in zip(outs, lses):
        assert_close(o, l, ro, rl)


def test_decode_right_after_each_transition(ekv_lib, torch_cuda):
    """ElasticKV's step order (Sec. 3.4, "Transition protocols": a page's new state is
    visible only after its transition completes): a transition of the library, then at
    once, in the same stream, a decode with the programmatic launch switched on that
    reads the pages just transitioned, non-last pages included. The transitions run on a
    second context, so the rule that ends the overlap after them holds across contexts.
    Each step order is repeated a few hundred times; every decode must match the oracle
    on the post-transition state."""
    torch = torch_cuda
    from oracle import base as ob
    from oracle import demote as odm
    lens = [700, 33, 1500, 16, 250, 1]
    hq, hkv, d = 32, 8, 128
    case = wl.make_decode_case(lens, hq, hkv, d, v_format="mixed", scale_mode=1, seed=910, poison=False,
                               pool_pages=sum((x + 15) // 16 for x in lens) + 4, p_compact=0.3, p_base=0.2)
    B, P, n = case.batch, case.num_pages, 16 * hkv * d
    used = sorted({int(case.block_table[b, j]) for b in range(B) for j in range((lens[b] + 15) // 16)})
    ids_np = np.array([p for p in used if case.page_mode[p] == 0], np.int32)
    last = {int(case.block_table[b, (lens[b] - 1) // 16]) for b in range(B)}
    assert any(p not in last for p in ids_np)          # non-last pages are transitioned
    dv = to_device(case)
    dec = ekv_lib.Context(hq, hkv, d, B, pdl=True)
    trans = ekv_lib.Context(hq, hkv, d, B)
    st = torch.cuda.current_stream()
    ids = torch.from_numpy(ids_np).cuda()
    v0, m0, s0 = dv.v_pages.clone(), dv.page_mode.clone(), dv.v_scales.clone()
    v, mode, sc = v0.clone(), m0.clone(), s0.clone()
    reps = 200

    def new_outs():
        return ([torch.empty((B, hq, d), dtype=torch.float16, device="cuda") for _ in range(reps)],
                [torch.empty((B, hq), dtype=torch.float32, device="cuda") for _ in range(reps)])

    def oracle_state(vv, mm, ss):
        c = wl.DecodeCase(**{**case.__dict__})
        c.v_pages, c.page_mode, c.v_scales = vv, mm, ss
        return oracle_decode(c)

    # E4M3 demotion, then decode (pages reset by copies before each demotion)
    outs, lses = new_outs()
    for r in range(reps):
        v.copy_(v0)
        mode.copy_(m0)
        sc.copy_(s0)
        ekv_lib.ekv_demote_pages(trans.handle, v, case.v_page_stride, P, ids, len(ids_np), mode, sc, st)
        _decode_into(ekv_lib, dec, case, dv, v, mode, sc, outs[r], lses[r], st)
    torch.cuda.synchronize()
    assert dec.error() == (0, 0) and trans.error() == (0, 0)
    rv, rm, rs = odm.demote_pages(case.v_pages, ids_np, case.page_mode, case.v_scales, hkv, d)
    assert np.array_equal(mode.cpu().numpy(), rm) and np.array_equal(v.cpu().numpy(), rv)
    _reps_match(outs, lses, oracle_state(rv, rm, rs))

    # BASE demotion then decode, promotion then decode, alternating on the same pages
    v.copy_(v0)
    mode.copy_(m0)
    low = torch.empty((len(ids_np), n), dtype=torch.uint8, device="cuda")
    outs_b, lses_b = new_outs()
    outs_p, lses_p = new_outs()
    for r in range(reps):
        ekv_lib.ekv_demote_pages_base(trans.handle, v, case.v_page_stride, P, ids, len(ids_np), mode, low, st)
        _decode_into(ekv_lib, dec, case, dv, v, mode, s0, outs_b[r], lses_b[r], st)
        ekv_lib.ekv_promote_pages(trans.handle, v, case.v_page_stride, P, ids, len(ids_np), mode, low, st)
        _decode_into(ekv_lib, dec, case, dv, v, mode, s0, outs_p[r], lses_p[r], st)
    torch.cuda.synchronize()
    assert dec.error() == (0, 0) and trans.error() == (0, 0)
    bv, bm, _, _ = ob.demote_to_base(case.v_pages, ids_np, case.page_mode, hkv, d)
    assert torch.equal(v, v0)                          # exact round trips
    _reps_match(outs_b, lses_b, oracle_state(bv, bm, case.v_scales))
    _reps_match(outs_p, lses_p, oracle_state(case.v_pages, case.page_mode, case.v_scales))
    dec.close()
    trans.close()


def test_elastic_decode_right_after_pair_packing(ekv_lib, torch_cuda):
    """The pair-structured layout: two located transitions pack pairs (A, B) of TARGET
    pages into A's slot (A in place, then B into half 1 of A's slot), and the elastic
    decode, launched at once with the programmatic switch on, reads the packed values
    through the value block table written before the transitions. Repeated a few
    hundred times from the same start; every decode must match the oracle."""
    torch = torch_cuda
    from oracle import elastic as oe
    lens = [16 * 30, 16 * 21 + 5, 37, 16 * 12]
    hq, hkv, d = 32, 8, 128
    case = wl.make_decode_case(lens, hq, hkv, d, v_format="fp16", seed=920, poison=False,
                               pool_pages=sum((x + 15) // 16 for x in lens) + 2)
    B, P = case.batch, case.num_pages
    bt = case.block_table
    pairs = [(int(bt[b, j]), int(bt[b, j + 1])) for b in (0, 1, 3) for j in range(0, 10, 2)]
    a_np = np.array([x for x, _ in pairs], np.int32)
    b_np = np.array([y for _, y in pairs], np.int32)
    vtab = 2 * bt.copy()
    for x, y in pairs:
        vtab[bt == y] = 2 * x + 1
    r1 = oe.transition(oe.OP_TO_E4M3, case.v_pages, a_np, None, None, np.zeros(P, np.uint8),
                       np.ones((P, hkv), np.float32), None, hkv, d)
    r2 = oe.transition(oe.OP_TO_E4M3, r1[0], b_np, 2 * b_np, 2 * a_np + 1, r1[1], r1[2], None, hkv, d)
    ref = oe.paged_decode_elastic(case.q, case.k_pages, r2[0], r2[2], 1, r2[1], 0, bt, vtab, None, 1,
                                  case.seq_lens)
    dv = to_device(case)
    dec = ekv_lib.Context(hq, hkv, d, B, pdl=True)
    trans = ekv_lib.Context(hq, hkv, d, B)
    st = torch.cuda.current_stream()
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()   # noqa: E731
    v0, vtab0, vtab_d = dv.v_pages.clone(), t(2 * bt), t(vtab)
    a, b, srcb, dstb = t(a_np), t(b_np), t(2 * b_np), t(2 * a_np + 1)
    v = v0.clone()
    mode = torch.zeros(P, dtype=torch.uint8, device="cuda")
    sc = torch.ones((P, hkv), dtype=torch.float32, device="cuda")
    vt = vtab0.clone()
    reps = 200
    outs = [torch.empty((B, hq, d), dtype=torch.float16, device="cuda") for _ in range(reps)]
    lses = [torch.empty((B, hq), dtype=torch.float32, device="cuda") for _ in range(reps)]
    for r in range(reps):
        v.copy_(v0)
        mode.zero_()
        sc.fill_(1.0)
        vt.copy_(vtab_d)                                 # the caller's value table, before the transitions
        ekv_lib.ekv_transition_pages(trans.handle, oe.OP_TO_E4M3, v, case.v_page_stride, P, P, a, None, None,
                                     len(a_np), mode, sc, None, st)
        ekv_lib.ekv_transition_pages(trans.handle, oe.OP_TO_E4M3, v, case.v_page_stride, P, P, b, srcb, dstb,
                                     len(b_np), mode, sc, None, st)
        ekv_lib.ekv_paged_decode_elastic(dec.handle, dv.q, dv.k_pages, v, case.v_page_stride, P, P, sc, 1, mode,
                                         0, dv.block_table, vt, bt.shape[1], None, 1, dv.seq_lens, B, 0.0,
                                         outs[r], lses[r], st)
    torch.cuda.synchronize()
    assert dec.error() == (0, 0) and trans.error() == (0, 0)
    assert np.array_equal(v.cpu().numpy(), r2[0]) and np.array_equal(mode.cpu().numpy(), r2[1])
    _reps_match(outs, lses, ref)
    dec.close()
    trans.close()
