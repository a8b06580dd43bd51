"""Errors made on the host, detected by the host checks or by the kernels' own bounds
checks (which record the fault and skip the access; no test traps or hangs the GPU)."""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl

from _helpers import gpu_decode, oracle_decode, to_device, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def base_case(fmt="e4m3", scale_mode=0):
    return wl.make_decode_case([40, 70, 20], 8, 2, 64, v_format=fmt, scale_mode=scale_mode,
                               pool_pages=12, seed=41)


def test_bad_page_id_is_reported_and_zeroes_only_that_sequence(ekv_lib, torch_cuda):
    case = base_case()
    case.block_table = case.block_table.copy()
    case.block_table[1, 2] = case.num_pages + 5           # outside the pool
    ctx = ekv_lib.Context(8, 2, 64, 3)
    out, lse = gpu_decode(ctx, to_device(case))
    code, detail = ctx.error()
    assert code == ekv_lib.EKV_ERR_DEVICE_CHECK and detail == ekv_lib.EKV_DETAIL_PAGE_ID
    o = out.float().cpu().numpy()
    assert np.all(o[1] == 0) and np.all(np.isneginf(lse.cpu().numpy()[1]))
    ref_out, ref_lse = oracle_decode(case, batch_indices=[0, 2])
    assert_close(out, lse, ref_out, ref_lse, rows=[0, 2])
    assert ctx.error() == (0, 0)                          # cleared by the read
    out2, _ = gpu_decode(ctx, to_device(base_case()))     # the context stays usable
    assert ctx.error() == (0, 0)


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), 0.0, -1.0])
def test_bad_scale_is_reported(ekv_lib, torch_cuda, bad):
    case = base_case("mixed", 1)
    case.v_scales = case.v_scales.copy()
    p = int(np.nonzero(case.page_mode == 1)[0][0])
    case.v_scales[p, 1] = bad
    ctx = ekv_lib.Context(8, 2, 64, 3)
    gpu_decode(ctx, to_device(case))
    code, detail = ctx.error()
    used = p in set(case.block_table[b, j] for b in range(3) for j in range((case.seq_lens[b] + 15) // 16))
    if used:
        assert (code, detail) == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_SCALE)


@pytest.mark.parametrize("lens", [[40, 70, 20], [700, 33, 1500, 5, 260]])
def test_bad_scale_zeroes_only_the_heads_of_its_kv_head(ekv_lib, torch_cuda, lens):
    """A bad per-(page, KV head) scale zeroes the G query heads of that KV head in the
    sequences that read the page; every other output matches the oracle. The longer
    length mix splits sequences over many CTAs, so the mark travels through the merge."""
    case = wl.make_decode_case(lens, 8, 2, 64, v_format="mixed", scale_mode=1, pool_pages=260, seed=43)
    good_scales = case.v_scales.copy()
    B, G = len(lens), 4
    bl = int(np.argmax(case.seq_lens))                     # a compact page of the longest sequence
    p = next(int(case.block_table[bl, j]) for j in range((case.seq_lens[bl] + 15) // 16)
             if case.page_mode[case.block_table[bl, j]] == 1)
    ref_out, ref_lse = oracle_decode(case)                 # with the good scales
    case.v_scales = good_scales.copy()
    case.v_scales[p, 1] = float("nan")
    ctx = ekv_lib.Context(8, 2, 64, B)
    out, lse = gpu_decode(ctx, to_device(case))
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_SCALE)
    users = [b for b in range(B) if p in set(case.block_table[b, :(case.seq_lens[b] + 15) // 16])]
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        for hq in range(8):
            if b in users and hq // G == 1:
                assert np.all(o[b, hq] == 0) and np.isneginf(l[b, hq]), (b, hq)
            else:
                assert np.abs(o[b, hq] - ref_out[b, hq]).max() <= 2e-3, (b, hq)
                assert abs(l[b, hq] - ref_lse[b, hq]) <= 1e-3, (b, hq)


def test_seq_len_above_capacity_is_reported(ekv_lib, torch_cuda):
    case = base_case()
    case.seq_lens = case.seq_lens.copy()
    case.seq_lens[2] = case.block_table.shape[1] * 16 + 1
    ctx = ekv_lib.Context(8, 2, 64, 3)
    out, lse = gpu_decode(ctx, to_device(case))
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_SEQ_LEN)
    assert np.all(out.float().cpu().numpy()[2] == 0)


def test_bad_page_mode_byte_is_reported(ekv_lib, torch_cuda):
    case = base_case("mixed", 1)
    case.page_mode = case.page_mode.copy()
    case.page_mode[case.block_table[0, 0]] = 7
    ctx = ekv_lib.Context(8, 2, 64, 3)
    gpu_decode(ctx, to_device(case))
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_PAGE_MODE)


def test_host_checks(ekv_lib, torch_cuda):
    import torch
    case = base_case()
    d = to_device(case)
    ctx = ekv_lib.Context(8, 2, 64, 2)
    out = torch.empty((3, 8, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(ekv_lib.EkvError) as e:       # batch 3 > max_batch 2
        ctx.decode(d, out)
    assert e.value.status == ekv_lib.EKV_ERR_CAPACITY
    ctx = ekv_lib.Context(8, 2, 64, 3)
    with pytest.raises(ekv_lib.EkvError) as e:       # misaligned q
        ekv_lib.ekv_paged_decode(ctx.handle, d.q.data_ptr() + 2, d.k_pages, d.v_pages, case.v_page_stride,
                                 case.num_pages, d.v_scales, 0, None, 1, d.block_table,
                                 case.block_table.shape[1], d.seq_lens, 3, 0.0, out)
    assert e.value.status == ekv_lib.EKV_ERR_INVALID_ARG
    with pytest.raises(ekv_lib.EkvError) as e:       # compact pool without scales
        ekv_lib.ekv_paged_decode(ctx.handle, d.q, d.k_pages, d.v_pages, case.v_page_stride,
                                 case.num_pages, None, 0, None, 1, d.block_table,
                                 case.block_table.shape[1], d.seq_lens, 3, 0.0, out)
    assert e.value.status == ekv_lib.EKV_ERR_INVALID_ARG
    with pytest.raises(ekv_lib.EkvError) as e:       # stride too small for TARGET pages
        ekv_lib.ekv_paged_decode(ctx.handle, d.q, d.k_pages, d.v_pages, case.v_page_stride,
                                 case.num_pages, d.v_scales, 0, None, 0, d.block_table,
                                 case.block_table.shape[1], d.seq_lens, 3, 0.0, out)
    assert e.value.status == ekv_lib.EKV_ERR_INVALID_ARG
    ws = torch.empty((2, 16, 2, 64), dtype=torch.float16, device="cuda")
    idx = torch.empty((2,), dtype=torch.int32, device="cuda")
    with pytest.raises(ekv_lib.EkvError) as e:       # workspace overflow
        ekv_lib.ekv_gather_prefill(ctx.handle, d.k_pages, d.v_pages, case.v_page_stride, case.num_pages,
                                   d.v_scales, 0, None, 1, d.block_table, case.block_table.shape[1],
                                   3, np.array([[1, 0, 3]]), ws, ws, idx, 2)
    assert e.value.status == ekv_lib.EKV_ERR_CAPACITY
    with pytest.raises(ekv_lib.EkvError) as e:       # range past the block table
        ekv_lib.ekv_gather_prefill(ctx.handle, d.k_pages, d.v_pages, case.v_page_stride, case.num_pages,
                                   d.v_scales, 0, None, 1, d.block_table, case.block_table.shape[1],
                                   3, np.array([[1, 4, 2]]), ws, ws, idx, 2)
    assert e.value.status == ekv_lib.EKV_ERR_INVALID_ARG
    with pytest.raises(ekv_lib.EkvError) as e:       # D = 96 unsupported
        ekv_lib.Context(8, 2, 96, 3)
    assert e.value.status == ekv_lib.EKV_ERR_UNSUPPORTED


def test_demote_bad_page_id_and_nonfinite(ekv_lib, torch_cuda):
    import torch
    P, H, D = 4, 2, 64
    x = np.random.default_rng(5).standard_normal((P, 16, H, D)).astype(np.float16)
    x[1, 3, 1, 9] = np.nan
    vb = torch.from_numpy(x.reshape(P, -1).view(np.uint8).copy()).cuda()
    mode = torch.zeros(P, dtype=torch.uint8, device="cuda")
    sc = torch.zeros((P, H), dtype=torch.float32, device="cuda")
    ctx = ekv_lib.Context(H, H, D, 1)
    ids = torch.tensor([1], dtype=torch.int32, device="cuda")
    before = vb.clone()
    ekv_lib.ekv_demote_pages(ctx.handle, vb, vb.shape[1], P, ids, 1, mode, sc)
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_NONFINITE_PAGE)
    assert torch.equal(vb, before) and int(mode[1]) == 0
    ids = torch.tensor([9], dtype=torch.int32, device="cuda")
    ekv_lib.ekv_demote_pages(ctx.handle, vb, vb.shape[1], P, ids, 1, mode, sc)
    assert ctx.error() == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_PAGE_ID)
