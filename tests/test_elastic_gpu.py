"""GPU parity of ElasticKV's pair-structured value layout through the C ABI, against
the oracle: pairs packed into one value slot by two located transitions (BASE and E4M3),
decode through the value block table (freed slots filled with garbage), the structured
TARGET-BASE-TARGET boundaries, the batch-level has_base = 0 path, identity locations
matching the plain decode bit for bit, bad locations reported, and the compact-prefill
gather from the same layouts bit for bit."""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl
from oracle import elastic as oe

from _helpers import assert_close, gpu_decode

pytestmark = pytest.mark.gpu
VARIANTS = [0, 1]


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _t(torch, x):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _elastic_decode(ekv_lib, torch, ctx, case, v_pages, page_mode, vtab, bnd, has_base, scales, scale_mode):
    B, Hq, D = case.batch, case.num_q_heads, case.head_dim
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    ekv_lib.ekv_paged_decode_elastic(ctx.handle, _t(torch, case.q), _t(torch, case.k_pages), _t(torch, v_pages),
                                     v_pages.shape[1], case.num_pages, v_pages.shape[0], _t(torch, scales),
                                     scale_mode, _t(torch, page_mode), 0, _t(torch, case.block_table),
                                     _t(torch, vtab), case.block_table.shape[1], _t(torch, bnd), has_base,
                                     _t(torch, case.seq_lens), B, 0.0, out, lse)
    torch.cuda.synchronize()
    return out, lse


def _transition(ekv_lib, torch, ctx, op, v, mode, ids, src, dst, scales, low, H, D):
    vd, md = _t(torch, v), _t(torch, mode)
    sd = _t(torch, scales) if scales is not None else None
    ld = _t(torch, low) if low is not None else None
    ekv_lib.ekv_transition_pages(ctx.handle, op, vd, v.shape[1], v.shape[0], len(mode), _t(torch, np.array(ids, np.int32)),
                                 _t(torch, None if src is None else np.array(src, np.int32)),
                                 _t(torch, None if dst is None else np.array(dst, np.int32)), len(ids), md, sd, ld)
    torch.cuda.synchronize()
    return (vd.cpu().numpy(), md.cpu().numpy(), None if sd is None else sd.cpu().numpy(),
            None if ld is None else ld.cpu().numpy())


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("op", [oe.OP_TO_BASE, oe.OP_TO_E4M3])
@pytest.mark.parametrize("hkv,d", [(2, 64), (8, 128)])
def test_packed_pairs(ekv_lib, torch_cuda, variant, op, hkv, d):
    torch = torch_cuda
    lens = [16 * 9, 16 * 7 + 5, 37]
    case = wl.make_decode_case(lens, 4 * hkv, hkv, d, v_format="fp16", seed=120 + op, pool_pages=30, poison=False)
    P, H = case.num_pages, hkv
    n = 16 * H * d
    ctx = ekv_lib.Context(4 * hkv, hkv, d, len(lens), variant=variant)
    bt = case.block_table
    # pairs of consecutive logical pages (j, j+1) for j = 2, 4 of sequences 0 and 1
    pairs = [(int(bt[b, j]), int(bt[b, j + 1])) for b in (0, 1) for j in (2, 4)]
    a = [x for x, _ in pairs]
    bb = [y for _, y in pairs]
    mode = np.zeros(P, np.uint8)
    scales = np.ones((P, H), np.float32)
    low = np.zeros((len(pairs), n), np.uint8)
    # GPU: two calls (A in place, then B into half 1 of A's slot)
    v1, m1, s1, l1 = _transition(ekv_lib, torch, ctx, op, case.v_pages, mode, a, None, None, scales, low, H, d)
    v2, m2, s2, l2 = _transition(ekv_lib, torch, ctx, op, v1, m1, bb, [2 * y for y in bb],
                                 [2 * x + 1 for x in a], s1, low, H, d)
    assert ctx.error() == (0, 0)
    r1 = oe.transition(op, case.v_pages, a, None, None, mode, scales, low, H, d)
    r2 = oe.transition(op, r1[0], bb, [2 * y for y in bb], [2 * x + 1 for x in a], r1[1], r1[2], low, H, d)
    assert np.array_equal(v2, r2[0]) and np.array_equal(m2, r2[1])
    if op == oe.OP_TO_E4M3:
        assert np.array_equal(s2, r2[2])
    else:
        assert np.array_equal(l1, r1[3]) and np.array_equal(l2, r2[3])
    vtab = 2 * bt.copy()
    for x, y in pairs:
        vtab[bt == y] = 2 * x + 1
    for y in bb:                                      # freed slots: garbage
        v2[y] = 0x7E
    out, lse = _elastic_decode(ekv_lib, torch, ctx, case, v2, m2, vtab, None, 1, s2, 1)
    assert ctx.error() == (0, 0)
    ref_out, ref_lse = oe.paged_decode_elastic(case.q, case.k_pages, v2, s2, 1, m2, 0, bt, vtab, None, 1,
                                               case.seq_lens)
    assert_close(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("variant", VARIANTS)
def test_boundaries_and_has_base(ekv_lib, torch_cuda, variant):
    torch = torch_cuda
    lens = [16 * 8, 16 * 6 - 3, 20]
    hkv, d = 4, 128
    case = wl.make_decode_case(lens, 16, hkv, d, v_format="fp16", seed=130, pool_pages=24, poison=False)
    P = case.num_pages
    bt = case.block_table
    bnd = np.array([[2, 6], [1, 5], [0, 0]], np.int32)
    base_pages = [int(bt[b, j]) for b in range(3) for j in range(bnd[b, 0], bnd[b, 1])]
    ctx = ekv_lib.Context(16, hkv, d, 3, variant=variant)
    v1, m1, _, _ = _transition(ekv_lib, torch, ctx, oe.OP_TO_BASE, case.v_pages, np.zeros(P, np.uint8), base_pages,
                               None, None, None, None, hkv, d)
    out, lse = _elastic_decode(ekv_lib, torch, ctx, case, v1, None, 2 * bt, bnd, 1, None, 0)
    assert ctx.error() == (0, 0)
    ref_out, ref_lse = oe.paged_decode_elastic(case.q, case.k_pages, v1, None, 0, None, 0, bt, 2 * bt, bnd, 1,
                                               case.seq_lens)
    assert_close(out, lse, ref_out, ref_lse)
    # has_base = 0: native path, every page TARGET (the original pool), modes ignored
    junk = np.full(P, 2, np.uint8)
    out, lse = _elastic_decode(ekv_lib, torch, ctx, case, case.v_pages, junk, 2 * bt, bnd, 0, None, 0)
    assert ctx.error() == (0, 0)
    ref_out, ref_lse = oe.paged_decode_elastic(case.q, case.k_pages, case.v_pages, None, 0, junk, 0, bt, 2 * bt,
                                               bnd, 0, case.seq_lens)
    assert_close(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("variant", VARIANTS)
def test_identity_locations_match_plain_decode_bitwise(ekv_lib, torch_cuda, variant):
    torch = torch_cuda
    lens = [300, 17, 90]
    case = wl.make_decode_case(lens, 32, 8, 128, v_format="mixed", scale_mode=1, seed=131, pool_pages=30,
                               p_compact=0.35, p_base=0.35)
    ctx = ekv_lib.Context(32, 8, 128, 3, variant=variant)
    from _helpers import to_device
    out0, lse0 = gpu_decode(ctx, to_device(case))
    out1, lse1 = _elastic_decode(ekv_lib, torch, ctx, case, case.v_pages, case.page_mode, 2 * case.block_table,
                                 None, 1, case.v_scales, 1)
    assert ctx.error() == (0, 0)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_bad_locations_are_reported(ekv_lib, torch_cuda):
    torch = torch_cuda
    case = wl.make_decode_case([40, 40], 8, 2, 64, v_format="fp16", seed=132, pool_pages=8, poison=False)
    ctx = ekv_lib.Context(8, 2, 64, 2)
    vtab = 2 * case.block_table.copy()
    vtab[1, 1] += 1                                   # odd location for a TARGET page
    out, lse = _elastic_decode(ekv_lib, torch, ctx, case, case.v_pages, None, vtab, None, 1, None, 0)
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_PAGE_ID)
    assert np.all(out.float().cpu().numpy()[1] == 0)
    vtab = 2 * case.block_table.copy()
    vtab[0, 0] = 2 * case.num_pages                   # outside the pool
    _elastic_decode(ekv_lib, torch, ctx, case, case.v_pages, None, vtab, None, 1, None, 0)
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_PAGE_ID)
    # a located transition to a location outside the pool
    _transition(ekv_lib, torch, ctx, 1, case.v_pages, np.zeros(case.num_pages, np.uint8), [0], [0],
                [2 * case.num_pages + 1], None, None, 2, 64)
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_PAGE_ID)


def _gather(ekv_lib, torch, ctx, case, v_pages, page_mode, scales, scale_mode, vtab, bnd, has_base, pr):
    total = int(np.asarray(pr)[:, 2].sum())
    H, D = case.num_kv_heads, case.head_dim
    ws_k = torch.full((total, 16, H, D), float("nan"), dtype=torch.float16, device="cuda")
    ws_v = torch.full_like(ws_k, float("nan"))
    idx = torch.empty((total,), dtype=torch.int32, device="cuda")
    ekv_lib.ekv_gather_prefill_elastic(ctx.handle, _t(torch, case.k_pages), _t(torch, v_pages), v_pages.shape[1],
                                       case.num_pages, v_pages.shape[0], _t(torch, scales), scale_mode,
                                       _t(torch, page_mode), 0, _t(torch, case.block_table), _t(torch, vtab),
                                       case.block_table.shape[1], _t(torch, bnd), has_base, case.batch, pr,
                                       ws_k, ws_v, idx, total)
    torch.cuda.synchronize()
    return ws_k.cpu().numpy(), ws_v.cpu().numpy(), idx.cpu().numpy()


@pytest.mark.parametrize("op", [oe.OP_TO_BASE, oe.OP_TO_E4M3])
def test_gather_from_packed_pairs(ekv_lib, torch_cuda, op):
    torch = torch_cuda
    lens = [16 * 9, 16 * 7 + 5]
    hkv, d = 4, 128
    case = wl.make_decode_case(lens, 16, hkv, d, v_format="fp16", seed=140 + op, pool_pages=20, poison=False)
    P, H = case.num_pages, hkv
    ctx = ekv_lib.Context(16, hkv, d, len(lens))
    bt = case.block_table
    pairs = [(int(bt[b, j]), int(bt[b, j + 1])) for b in (0, 1) for j in (2, 4)]
    a = [x for x, _ in pairs]
    bb = [y for _, y in pairs]
    mode = np.zeros(P, np.uint8)
    scales = np.ones((P, H), np.float32)
    v1, m1, s1, _ = _transition(ekv_lib, torch, ctx, op, case.v_pages, mode, a, None, None, scales, None, H, d)
    v2, m2, s2, _ = _transition(ekv_lib, torch, ctx, op, v1, m1, bb, [2 * y for y in bb],
                                [2 * x + 1 for x in a], s1, None, H, d)
    vtab = 2 * bt.copy()
    for x, y in pairs:
        vtab[bt == y] = 2 * x + 1
    for y in bb:                                      # freed slots: garbage
        v2[y] = 0x7E
    pr = np.array([[0, 0, 9], [1, 1, 7]])
    gk, gv, gi = _gather(ekv_lib, torch, ctx, case, v2, m2, s2, 1, vtab, None, 1, pr)
    assert ctx.error() == (0, 0)
    rk, rv, ri = oe.gather_prefill_elastic(case.k_pages, v2, s2, 1, m2, 0, bt, vtab, None, 1, pr)
    assert np.array_equal(gk.view(np.uint16), rk.view(np.uint16))
    assert np.array_equal(gv.view(np.uint16), rv.view(np.uint16)) and np.array_equal(gi, ri)


def test_gather_boundaries_has_base_and_bad_location(ekv_lib, torch_cuda):
    torch = torch_cuda
    lens = [16 * 8, 16 * 6 - 3]
    hkv, d = 4, 64
    case = wl.make_decode_case(lens, 8, hkv, d, v_format="fp16", seed=150, pool_pages=16, poison=False)
    P = case.num_pages
    bt = case.block_table
    bnd = np.array([[2, 6], [1, 5]], np.int32)
    base_pages = [int(bt[b, j]) for b in range(2) for j in range(bnd[b, 0], bnd[b, 1])]
    ctx = ekv_lib.Context(8, hkv, d, 2)
    v1, _, _, _ = _transition(ekv_lib, torch, ctx, oe.OP_TO_BASE, case.v_pages, np.zeros(P, np.uint8), base_pages,
                              None, None, None, None, hkv, d)
    pr = np.array([[0, 0, 8], [1, 0, 6]])
    _, gv, _ = _gather(ekv_lib, torch, ctx, case, v1, None, None, 0, 2 * bt, bnd, 1, pr)
    assert ctx.error() == (0, 0)
    _, rv, _ = oe.gather_prefill_elastic(case.k_pages, v1, None, 0, None, 0, bt, 2 * bt, bnd, 1, pr)
    assert np.array_equal(gv.view(np.uint16), rv.view(np.uint16))
    # has_base = 0: the original TARGET pool, modes and boundaries ignored
    _, gv, _ = _gather(ekv_lib, torch, ctx, case, case.v_pages, np.full(P, 2, np.uint8), None, 0, 2 * bt, bnd, 0, pr)
    assert ctx.error() == (0, 0)
    _, rv, _ = oe.gather_prefill_elastic(case.k_pages, case.v_pages, None, 0, np.full(P, 2, np.uint8), 0, bt,
                                         2 * bt, bnd, 0, pr)
    assert np.array_equal(gv.view(np.uint16), rv.view(np.uint16))
    # an odd location for a TARGET page: reported, that workspace page zeroed
    vtab = 2 * bt.copy()
    vtab[1, 0] += 1
    gk, gv, _ = _gather(ekv_lib, torch, ctx, case, case.v_pages, None, None, 0, vtab, None, 1, pr)
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_PAGE_ID)
    assert np.all(gv[8] == 0) and np.all(gk[8] == 0)
