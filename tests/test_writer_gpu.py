"""GPU parity of ekv_append_kv (the K16/V8 cache writer) against the oracle: the pools
after each append are bit-identical to the oracle's, over pages in all three value
modes and uniform pools, across page boundaries and over many steps; a decode after
the appends matches the oracle's decode of its own pools; bad positions, page ids,
mode bytes and scales are reported and write nothing."""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl
from oracle import writer as ow

from _helpers import assert_close, gpu_decode, oracle_decode, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _append(ekv_lib, torch, ctx, case, d, kn, vn, pos):
    k_new = torch.from_numpy(kn).cuda()
    v_new = torch.from_numpy(vn).cuda()
    p = torch.from_numpy(np.asarray(pos, np.int32)).cuda()
    ekv_lib.ekv_append_kv(ctx.handle, k_new, v_new, d.k_pages, d.v_pages, case.v_page_stride, case.num_pages,
                          d.v_scales, case.scale_mode, d.page_mode, case.uniform_mode, d.block_table,
                          case.block_table.shape[1], p, len(pos))
    torch.cuda.synchronize()


FORMATS = [("mixed", 1, dict(p_compact=0.35, p_base=0.35)), ("mixed", 0, {}), ("e4m3", 0, {}),
           ("e4m3", 1, {}), ("fp16", 0, {}), ("base", 0, {})]


@pytest.mark.parametrize("fi", range(len(FORMATS)))
@pytest.mark.parametrize("hkv,d", [(2, 64), (8, 128)])
def test_appends_are_bit_exact_over_many_steps(ekv_lib, torch_cuda, fi, hkv, d):
    torch = torch_cuda
    fmt, sm, kw = FORMATS[fi]
    final = np.array([40, 33, 100, 17, 64], np.int32)
    steps = 20
    case = wl.make_decode_case(final, 4 * hkv, hkv, d, v_format=fmt, scale_mode=sm, seed=100 + fi,
                               pool_pages=40, poison=False, **kw)
    dev = to_device(case)
    ctx = ekv_lib.Context(4 * hkv, hkv, d, len(final))
    k_ref, v_ref = case.k_pages.copy(), case.v_pages.copy()
    rng = np.random.default_rng(7)
    for s in range(steps):                               # positions final - steps .. final - 1
        pos = final - steps + s
        pos[3] = pos[3] if s % 3 else -1                 # a sequence with no token some steps
        kn = rng.standard_normal((len(final), hkv, d)).astype(np.float16)
        vn = (rng.standard_normal((len(final), hkv, d)) * 0.8).astype(np.float16)
        _append(ekv_lib, torch, ctx, case, dev, kn, vn, pos)
        k_ref, v_ref = ow.append_token(k_ref, v_ref, case.v_scales, case.scale_mode, case.page_mode,
                                       case.uniform_mode, case.block_table, pos, kn, vn)
    assert ctx.error() == (0, 0)
    assert np.array_equal(dev.k_pages.cpu().numpy().view(np.uint16), k_ref.view(np.uint16))
    assert np.array_equal(dev.v_pages.cpu().numpy(), v_ref)
    # decode over the written pools
    case.k_pages, case.v_pages = k_ref, v_ref
    out, lse = gpu_decode(ctx, dev)
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)


def test_bad_inputs_write_nothing(ekv_lib, torch_cuda):
    torch = torch_cuda
    case = wl.make_decode_case([40, 40, 40], 8, 2, 64, v_format="mixed", scale_mode=1, seed=110,
                               pool_pages=12, poison=False, p_compact=1.0)
    dev = to_device(case)
    ctx = ekv_lib.Context(8, 2, 64, 3)
    kn = np.ones((3, 2, 64), np.float16)
    before_k, before_v = dev.k_pages.clone(), dev.v_pages.clone()
    _append(ekv_lib, torch, ctx, case, dev, kn, kn, [case.block_table.shape[1] * 16, -1, -1])
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_SEQ_LEN)
    dev.block_table[1, 0] = case.num_pages + 3
    _append(ekv_lib, torch, ctx, case, dev, kn, kn, [-1, 5, -1])
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_PAGE_ID)
    assert torch.equal(dev.k_pages, before_k) and torch.equal(dev.v_pages, before_v)
    # a compact page with a bad scale for one KV head: K written, that head's V kept
    p = int(case.block_table[2, 0])
    dev.v_scales[p, 1] = float("nan")
    _append(ekv_lib, torch, ctx, case, dev, kn, kn, [-1, -1, 3])
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_SCALE)
    sc = case.v_scales.copy()
    sc[p, 1] = np.nan
    k_ref, v_ref = ow.append_token(case.k_pages, case.v_pages, sc, 1, case.page_mode, 0, case.block_table,
                                   np.array([-1, -1, 3]), kn, kn)
    assert np.array_equal(dev.v_pages.cpu().numpy(), v_ref)
    assert np.array_equal(dev.k_pages.cpu().numpy().view(np.uint16), k_ref.view(np.uint16))
