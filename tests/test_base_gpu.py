"""GPU parity of the ElasticKV BASE value mode through the C ABI, against the oracle:
decode over pages in all three modes and over a uniform BASE pool (attention
tolerance), gather of BASE pages, TARGET -> BASE demotion and exact promotion (bit for
bit), and demote-then-decode / promote-then-decode round trips."""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl
from oracle import base as ob
from oracle import gather as og

from _helpers import assert_close, gpu_decode, oracle_decode, to_device

pytestmark = pytest.mark.gpu
VARIANTS = [0, 1]


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


CASES = [  # (lens, Hq, Hkv, D, scale_mode)
    ([37, 100, 1, 16, 250], 8, 2, 64, 1),
    ([33, 700, 129], 32, 8, 128, 0),
    ([5, 64, 99, 1500], 32, 4, 128, 1),
    ([48, 1, 77, 31], 8, 1, 64, 0),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("ci", range(len(CASES)))
def test_decode_three_modes(ekv_lib, torch_cuda, variant, ci):
    lens, hq, hkv, d, sm = CASES[ci]
    case = wl.make_decode_case(lens, hq, hkv, d, v_format="mixed", scale_mode=sm, seed=80 + ci,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 7, p_compact=0.35, p_base=0.35)
    assert set(np.unique(case.page_mode)) == {0, 1, 2}
    ctx = ekv_lib.Context(hq, hkv, d, len(lens), variant=variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    assert ctx.error() == (0, 0)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("hkv,d", [(2, 64), (8, 128)])
def test_decode_uniform_base_pool(ekv_lib, torch_cuda, variant, hkv, d):
    lens = [37, 300, 16]
    case = wl.make_decode_case(lens, 4 * hkv, hkv, d, v_format="base", seed=90, pool_pages=40)
    assert case.page_mode is None and case.uniform_mode == ekv_lib.EKV_MODE_BASE
    case.v_scales = None                                  # BASE needs no scales
    ctx = ekv_lib.Context(4 * hkv, hkv, d, len(lens), variant=variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    assert ctx.error() == (0, 0)


def test_gather_base_pages_bit_exact(ekv_lib, torch_cuda):
    import torch
    lens = [100, 260, 33]
    case = wl.make_decode_case(lens, 8, 4, 128, v_format="mixed", scale_mode=1, seed=91, pool_pages=40,
                               poison=False, p_compact=0.3, p_base=0.4)
    d = to_device(case)
    page_range = np.array([[0, 0, 7], [1, 2, 10], [2, 0, 3]])
    total = int(page_range[:, 2].sum())
    P, H, D = case.num_pages, case.num_kv_heads, case.head_dim
    ws_k = torch.empty((total, 16, H, D), dtype=torch.float16, device="cuda")
    ws_v = torch.empty_like(ws_k)
    idx = torch.empty((total,), dtype=torch.int32, device="cuda")
    ctx = ekv_lib.Context(8, H, D, 1)
    ekv_lib.ekv_gather_prefill(ctx.handle, d.k_pages, d.v_pages, case.v_page_stride, P, d.v_scales, 1,
                               d.page_mode, 0, d.block_table, case.block_table.shape[1], len(lens),
                               page_range, ws_k, ws_v, idx, total)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    rk, rv, ri = og.gather_prefill(case.k_pages, case.v_pages, case.v_scales, 1, case.page_mode, 0,
                                   case.block_table, page_range)
    assert np.array_equal(ws_k.cpu().numpy().view(np.uint16), rk.view(np.uint16))
    assert np.array_equal(ws_v.cpu().numpy().view(np.uint16), rv.view(np.uint16))


def _demote_base(ekv_lib, torch, vb, ids, mode, H, D, with_low=True):
    v = torch.from_numpy(vb.copy()).cuda()
    m = torch.from_numpy(mode.copy()).cuda()
    n = 16 * H * D
    low = torch.full((len(ids), n), 0xAB, dtype=torch.uint8, device="cuda") if with_low else None
    pid = torch.from_numpy(np.asarray(ids, dtype=np.int32)).cuda()
    ctx = ekv_lib.Context(H, H, D, 1)
    ekv_lib.ekv_demote_pages_base(ctx.handle, v, vb.shape[1], vb.shape[0], pid, len(ids), m, low)
    torch.cuda.synchronize()
    err = ctx.error()
    return v, m, low, err, ctx


@pytest.mark.parametrize("P,n,hkv,d", [(40, 22, 8, 128), (30, 30, 2, 64), (4096, 4000, 4, 128)])
def test_demote_to_base_and_promote_bit_exact(ekv_lib, torch_cuda, P, n, hkv, d):
    torch = torch_cuda
    rng = np.random.default_rng(95)
    x = (rng.standard_normal((P, 16, hkv, d)) * 3).astype(np.float16)
    x[1, 2, 0, 5] = np.inf                             # non-finite: left TARGET, reported
    vb = x.reshape(P, -1).view(np.uint8).copy()
    mode = np.zeros(P, np.uint8)
    mode[rng.choice(P, size=max(1, P // 10), replace=False)] = 1   # compact: skipped
    mode[1] = 0
    ids = rng.permutation(P)[:n]
    if 1 not in ids:
        ids[0] = 1
    v, m, low, err, ctx = _demote_base(ekv_lib, torch, vb, ids, mode, hkv, d)
    rv, rm, rlow, bad = ob.demote_to_base(vb, ids, mode, hkv, d)
    assert err == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_NONFINITE_PAGE) and bad == [1]
    assert np.array_equal(m.cpu().numpy(), rm)
    assert np.array_equal(v.cpu().numpy(), rv)
    lo = low.cpu().numpy()
    for i, p in enumerate(ids):
        if rm[p] == ob.MODE_BASE:
            assert np.array_equal(lo[i], rlow[p])
        else:
            assert np.all(lo[i] == 0xAB)                  # untouched row
    # exact promotion with the rows the demotion wrote
    pid = torch.from_numpy(np.asarray(ids, dtype=np.int32)).cuda()
    ekv_lib.ekv_promote_pages(ctx.handle, v, vb.shape[1], P, pid, len(ids), m, low)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    back = v.cpu().numpy()
    mm = m.cpu().numpy()
    for p in range(P):
        if rm[p] == ob.MODE_BASE:
            assert np.array_equal(back[p], vb[p]) and mm[p] == 0
        else:
            assert np.array_equal(back[p], rv[p]) and mm[p] == rm[p]


def test_demote_to_base_without_backing_then_decode(ekv_lib, torch_cuda):
    torch = torch_cuda
    lens = [300, 77, 1200]
    case = wl.make_decode_case(lens, 16, 4, 128, v_format="fp16", seed=96, pool_pages=120, poison=False)
    P = case.num_pages
    ids = np.random.default_rng(0).permutation(P)[: P // 2]
    v, m, _, err, _ = _demote_base(ekv_lib, torch, case.v_pages, ids, np.zeros(P, np.uint8), 4, 128,
                                   with_low=False)
    assert err == (0, 0)
    rv, rm, _, _ = ob.demote_to_base(case.v_pages, ids, np.zeros(P, np.uint8), 4, 128)
    assert np.array_equal(v.cpu().numpy(), rv) and np.array_equal(m.cpu().numpy(), rm)
    case.v_pages, case.page_mode, case.v_scales = rv, rm, None
    ctx = ekv_lib.Context(16, 4, 128, len(lens))
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    assert ctx.error() == (0, 0)


def test_bad_mode_byte_and_missing_scale(ekv_lib, torch_cuda):
    case = wl.make_decode_case([40, 70], 8, 2, 64, v_format="mixed", scale_mode=1, seed=97, pool_pages=12,
                               p_compact=0.0, p_base=0.5)
    case.page_mode = case.page_mode.copy()
    case.page_mode[case.block_table[1, 1]] = 3         # not a mode
    ctx = ekv_lib.Context(8, 2, 64, 2)
    out, lse = gpu_decode(ctx, to_device(case))
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_PAGE_MODE)
    assert np.all(out.float().cpu().numpy()[1] == 0)
    # a compact page in a mixed pool passed without scales: reported, not read
    case2 = wl.make_decode_case([40, 70], 8, 2, 64, v_format="mixed", scale_mode=1, seed=98, pool_pages=12)
    case2.v_scales = None
    out, lse = gpu_decode(ctx, to_device(case2))
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_SCALE)
