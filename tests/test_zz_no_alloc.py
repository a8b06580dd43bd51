"""The allocation-free decode entry point against the context-based one and the oracle.

ekv_paged_decode_noalloc is for callers that may not allocate device memory on the
decode path (a runtime whose memory pool owns the GPU, a framework hook where
allocation is forbidden, a fixed start-up budget): it keeps its split-K scratch in a
fixed array compiled into the library instead of a context's cudaMalloc'd buffers.
Here it must give the same outputs as ekv_paged_decode and as the float64 oracle, within
the attention tolerance, on two calls in a row (the second call reuses the array the
first one left behind), report data errors through err_out and clear them on the next
call, and refuse a batch whose scratch would not fit. This file is collected last on
purpose.
"""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl

from _helpers import LSE_ATOL, OUT_ATOL, assert_close, oracle_decode, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _noalloc(ekv_lib, torch, case, d):
    B, Hq, D = case.batch, case.num_q_heads, case.head_dim
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    ekv_lib.ekv_paged_decode_noalloc(Hq, case.num_kv_heads, D, d.q, d.k_pages, d.v_pages,
                                     case.v_page_stride, case.num_pages, d.v_scales,
                                     case.scale_mode, d.page_mode, case.uniform_mode,
                                     d.block_table, case.block_table.shape[1], d.seq_lens, B, 0.0,
                                     out, lse, err)
    torch.cuda.synchronize()
    return out, lse, err


def _with_context(ekv_lib, torch, case, d):
    B, Hq, D = case.batch, case.num_q_heads, case.head_dim
    ctx = ekv_lib.Context(Hq, case.num_kv_heads, D, B)
    out = torch.empty((B, Hq, D), dtype=torch.float16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    ctx.decode(d, out, lse)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    ctx.close()
    return out, lse


def _same(a, la, b, lb):
    assert (a.float() - b.float()).abs().max().item() <= OUT_ATOL
    fa, fb = la.cpu().numpy(), lb.cpu().numpy()
    assert np.array_equal(np.isfinite(fa), np.isfinite(fb))
    fin = np.isfinite(fa)
    if fin.any():
        assert np.abs(fa[fin] - fb[fin]).max() <= LSE_ATOL


def test_no_alloc_matches_context_decode_twice(ekv_lib, torch_cuda):
    torch = torch_cuda
    cases = [
        wl.make_decode_case([2000, 37, 0, 1500, 16], 32, 8, 128, v_format="e4m3", scale_mode=0,
                            pool_pages=260, seed=71),
        wl.make_decode_case([300, 1, 900, 45, 610, 77, 3], 32, 4, 128, v_format="mixed",
                            scale_mode=1, pool_pages=130, seed=72),
    ]
    for case in cases:                      # two calls in a row on different inputs
        d = to_device(case)
        ref_out, ref_lse = _with_context(ekv_lib, torch, case, d)
        out, lse, err = _noalloc(ekv_lib, torch, case, d)
        assert err.cpu().tolist() == [0, 0, 0, 0]
        _same(out, lse, ref_out, ref_lse)
        o_ref, l_ref = oracle_decode(case)
        assert_close(out, lse, o_ref, l_ref)
    # the same call again right after: results do not depend on what the array held
    out2, lse2, err2 = _noalloc(ekv_lib, torch, cases[1], to_device(cases[1]))
    assert err2.cpu().tolist() == [0, 0, 0, 0]
    _same(out2, lse2, ref_out, ref_lse)
    assert_close(out2, lse2, o_ref, l_ref)


@pytest.mark.parametrize("fmt", ["fp16", "base"])
def test_no_alloc_head_dim_64_uniform_pools(ekv_lib, torch_cuda, fmt):
    """Head dim 64 and the uniform FP16 (native) and BASE pools of the same entry point."""
    torch = torch_cuda
    case = wl.make_decode_case([1200, 3, 0, 700, 64], 16, 2, 64, v_format=fmt, pool_pages=140, seed=74)
    d = to_device(case)
    ref_out, ref_lse = _with_context(ekv_lib, torch, case, d)
    for _ in range(2):
        out, lse, err = _noalloc(ekv_lib, torch, case, d)
        assert err.cpu().tolist() == [0, 0, 0, 0]
        _same(out, lse, ref_out, ref_lse)
    o_ref, l_ref = oracle_decode(case)
    assert_close(out, lse, o_ref, l_ref)


def test_no_alloc_reports_data_errors_in_err_out(ekv_lib, torch_cuda):
    """A page id outside the pool zeroes its sequence; a bad per-(page, KV head) scale
    zeroes the query heads of that KV head in the sequences that read the page. Both are
    reported through err_out as {EKV_ERR_DEVICE_CHECK, detail, index, 0}; the next clean
    call starts from a zeroed err_out and matches the oracle."""
    torch = torch_cuda
    lens = [700, 40, 1500, 20]
    case = wl.make_decode_case(lens, 32, 8, 128, v_format="mixed", scale_mode=1, pool_pages=150, seed=75)
    o_ref, l_ref = oracle_decode(case)
    # a page id outside the pool in sequence 1
    bad = wl.DecodeCase(**{**case.__dict__})
    bad.block_table = case.block_table.copy()
    bad.block_table[1, 1] = case.num_pages + 3
    out, lse, err = _noalloc(ekv_lib, torch, bad, to_device(bad))
    assert err.cpu().tolist() == [ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_PAGE_ID, 1, 0]
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(o[1] == 0) and np.all(np.isneginf(l[1]))
    assert_close(out, lse, o_ref, l_ref, rows=[0, 2, 3])
    # a bad scale of KV head 3 on a compact page of the longest sequence
    bad = wl.DecodeCase(**{**case.__dict__})
    bad.v_scales = case.v_scales.copy()
    p = next(int(case.block_table[2, j]) for j in range((lens[2] + 15) // 16)
             if case.page_mode[case.block_table[2, j]] == 1)
    bad.v_scales[p, 3] = float("nan")
    out, lse, err = _noalloc(ekv_lib, torch, bad, to_device(bad))
    e = err.cpu().tolist()
    assert e[:2] == [ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_SCALE] and e[3] == 0
    users = {b for b in range(len(lens)) if p in set(case.block_table[b, :(lens[b] + 15) // 16])}
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    G = 4
    for b in range(len(lens)):
        for hq in range(32):
            if b in users and hq // G == 3:
                assert np.all(o[b, hq] == 0) and np.isneginf(l[b, hq])
            else:
                assert np.abs(o[b, hq] - o_ref[b, hq]).max() <= OUT_ATOL
    # a clean call right after: err_out zeroed by the call, outputs match the oracle
    out, lse, err = _noalloc(ekv_lib, torch, case, to_device(case))
    assert err.cpu().tolist() == [0, 0, 0, 0]
    assert_close(out, lse, o_ref, l_ref)


def test_no_alloc_refuses_batches_beyond_its_scratch(ekv_lib, torch_cuda):
    torch = torch_cuda
    case = wl.make_decode_case([20], 8, 1, 128, v_format="fp16", pool_pages=2, seed=73)
    d = to_device(case)
    B = 4096                                 # (4096 + #SMs) * 8 * 8 * 130 floats > 16 MiB
    bt = torch.zeros((B, 2), dtype=torch.int32, device="cuda")
    sl = torch.zeros((B,), dtype=torch.int32, device="cuda")
    q = torch.zeros((B, 8, 128), dtype=torch.float16, device="cuda")
    out = torch.empty((B, 8, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(ekv_lib.EkvError) as e:
        ekv_lib.ekv_paged_decode_noalloc(8, 1, 128, q, d.k_pages, d.v_pages, case.v_page_stride,
                                         case.num_pages, None, 0, None, 0, bt, 2, sl, B, 0.0, out)
    assert e.value.status == ekv_lib.EKV_ERR_CAPACITY
