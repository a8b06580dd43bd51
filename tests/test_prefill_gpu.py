"""GPU parity of ekv_prefill_attention (FP16 causal prefill over the gathered workspace)
against the float64 oracle, for both kernels (variant 0: tcgen05 tensor cores with
tensor-memory accumulators; variant 1: warp-level mma.sync): small ragged prompts compared
on every row (a one-token prompt, page-, key-block- and query-tile-boundary lengths, GQA
at several shapes), scores that grow along the prompt (forcing the running max to be
re-based), long prompts on sampled rows, the gather -> prefill chain on a mixed-fidelity
cache, and a prompt longer than max_len reported and cut there."""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl
from oracle import gather as og
from oracle import prefill as op

from _helpers import LSE_ATOL, OUT_ATOL

pytestmark = pytest.mark.gpu
VARIANTS = [0, 1]


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _case(lens, H_q, H_kv, D, seed, slack=2):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    npages = [(l + 15) // 16 for l in lens]
    page_off = (np.concatenate([[0], np.cumsum(npages)[:-1]]) + 1).astype(np.int32)   # page 0 unused
    W = sum(npages) + slack + 1
    q = rng.standard_normal((int(cu[-1]), H_q, D)).astype(np.float16)
    ws_k = rng.standard_normal((W, 16, H_kv, D)).astype(np.float16)
    ws_v = rng.standard_normal((W, 16, H_kv, D)).astype(np.float16)
    return q, ws_k, ws_v, cu, page_off


def _run(ekv_lib, torch, q, ws_k, ws_v, cu, po, H_q, H_kv, D, max_len=None, variant=0):
    T = q.shape[0]
    ctx = ekv_lib.Context(H_q, H_kv, D, 1, variant=variant)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = torch.full((T, H_q, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((T, H_q), float("nan"), dtype=torch.float32, device="cuda")
    lens = np.diff(cu)
    ekv_lib.ekv_prefill_attention(ctx.handle, t(q), t(ws_k), t(ws_v), ws_k.shape[0], t(cu), t(po), len(lens),
                                  int(lens.max()) if max_len is None else max_len, 0.0, out, lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), ctx.error()


def _check(out, lse, ref_out, ref_lse, rows):
    e = np.abs(out[rows] - ref_out[rows]).max()
    assert e <= OUT_ATOL, f"max-abs error {e:.3e}"
    le = np.abs(lse[rows] - ref_lse[rows]).max()
    assert le <= LSE_ATOL, f"lse error {le:.3e}"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("H_q,H_kv,D", [(8, 2, 64), (32, 8, 128), (12, 4, 128), (4, 4, 64)])
def test_small_prompts_every_row(ekv_lib, torch_cuda, H_q, H_kv, D, variant):
    lens = [1, 17, 64, 65, 130, 200]
    q, k, v, cu, po = _case(lens, H_q, H_kv, D, 140 + D + H_q)
    out, lse, err = _run(ekv_lib, torch_cuda, q, k, v, cu, po, H_q, H_kv, D, variant=variant)
    assert err == (0, 0)
    ref_out, ref_lse = op.prefill_attention(q, k, v, cu, po)
    _check(out, lse, ref_out, ref_lse, np.arange(q.shape[0]))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("D", [64, 128])
def test_tile_boundaries_every_row(ekv_lib, torch_cuda, D, variant):
    # 64-key blocks, 128-row query tiles and 256-row CTAs: lengths on and around each
    lens = [63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 385, 513]
    H_q, H_kv = 4, 2
    q, k, v, cu, po = _case(lens, H_q, H_kv, D, 160 + D)
    out, lse, err = _run(ekv_lib, torch_cuda, q, k, v, cu, po, H_q, H_kv, D, variant=variant)
    assert err == (0, 0)
    ref_out, ref_lse = op.prefill_attention(q, k, v, cu, po)
    _check(out, lse, ref_out, ref_lse, np.arange(q.shape[0]))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("lens", [[512], [256, 384], [128, 100, 256]])
def test_query_tiles_ending_at_the_last_row(ekv_lib, torch_cuda, lens, variant):
    # a 128-row query tile inside its prompt comes in by one TMA box; here the last prompt
    # ends on a tile boundary, so the last box ends exactly at q's last row
    H_q, H_kv, D = 8, 2, 128
    q, k, v, cu, po = _case(lens, H_q, H_kv, D, 190 + len(lens))
    out, lse, err = _run(ekv_lib, torch_cuda, q, k, v, cu, po, H_q, H_kv, D, variant=variant)
    assert err == (0, 0)
    ref_out, ref_lse = op.prefill_attention(q, k, v, cu, po)
    _check(out, lse, ref_out, ref_lse, np.arange(q.shape[0]))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("D", [64, 128])
def test_many_ragged_prompts_every_row(ekv_lib, torch_cuda, D, variant):
    # 48 prompts of random lengths (an empty one included): many work items per CTA, items
    # past their prompt's end, partial query tiles, the last prompt's last tile at q's end
    rng = np.random.default_rng(200 + D)
    lens = [int(x) for x in rng.integers(0, 700, size=48)]
    lens[7] = 0
    lens[-1] = 257
    H_q, H_kv = 8, 2
    q, k, v, cu, po = _case(lens, H_q, H_kv, D, 210 + D)
    out, lse, err = _run(ekv_lib, torch_cuda, q, k, v, cu, po, H_q, H_kv, D, variant=variant)
    assert err == (0, 0)
    ref_out, ref_lse = op.prefill_attention(q, k, v, cu, po)
    _check(out, lse, ref_out, ref_lse, np.arange(q.shape[0]))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("D", [64, 128])
def test_growing_scores_rebase_the_max(ekv_lib, torch_cuda, D, variant):
    # keys grow along the prompt, so each row's running max climbs by many powers of two
    # across its key blocks (the lazy re-basing of O and l must run, repeatedly)
    lens = [700, 300]
    H_q, H_kv = 4, 1
    q, k, v, cu, po = _case(lens, H_q, H_kv, D, 170 + D)
    q = np.abs(q.astype(np.float32)).astype(np.float16)
    ramp = (0.1 * np.arange(k.shape[0] * 16, dtype=np.float32) / 16).reshape(k.shape[0], 16, 1, 1)
    k = (np.abs(k.astype(np.float32)) * ramp).astype(np.float16)
    out, lse, err = _run(ekv_lib, torch_cuda, q, k, v, cu, po, H_q, H_kv, D, variant=variant)
    assert err == (0, 0)
    ref_out, ref_lse = op.prefill_attention(q, k, v, cu, po)
    assert np.all(np.isfinite(ref_lse))
    _check(out, lse, ref_out, ref_lse, np.arange(q.shape[0]))


@pytest.mark.parametrize("variant", VARIANTS)
def test_long_prompts_sampled_rows(ekv_lib, torch_cuda, variant):
    lens = [2048, 1500, 3000]
    H_q, H_kv, D = 32, 8, 128
    q, k, v, cu, po = _case(lens, H_q, H_kv, D, 150)
    out, lse, err = _run(ekv_lib, torch_cuda, q, k, v, cu, po, H_q, H_kv, D, variant=variant)
    assert err == (0, 0)
    sample = {0: [0, 63, 64, 1000, 2047], 1: [5, 1499], 2: [127, 128, 2999]}
    ref_out, ref_lse = op.prefill_attention(q, k, v, cu, po, rows=sample)
    rows = np.array([cu[i] + s for i, ss in sample.items() for s in ss])
    _check(out, lse, ref_out, ref_lse, rows)


@pytest.mark.parametrize("variant", VARIANTS)
def test_gather_then_prefill(ekv_lib, torch_cuda, variant):
    torch = torch_cuda
    lens = [300, 97, 500]
    H_q, H_kv, D = 32, 8, 128
    case = wl.make_decode_case(lens, H_q, H_kv, D, v_format="mixed", scale_mode=1, seed=151, pool_pages=70,
                               poison=False, p_compact=0.4, p_base=0.3)
    pr = np.array([[b, 0, (l + 15) // 16] for b, l in enumerate(lens)])
    total = int(pr[:, 2].sum())
    t = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()
    ws_k = torch.empty((total, 16, H_kv, D), dtype=torch.float16, device="cuda")
    ws_v = torch.empty_like(ws_k)
    idx = torch.empty((total,), dtype=torch.int32, device="cuda")
    ctx = ekv_lib.Context(H_q, H_kv, D, len(lens), variant=variant)
    ekv_lib.ekv_gather_prefill(ctx.handle, t(case.k_pages), t(case.v_pages), case.v_page_stride, case.num_pages,
                               t(case.v_scales), 1, t(case.page_mode), 0, t(case.block_table),
                               case.block_table.shape[1], len(lens), pr, ws_k, ws_v, idx, total)
    rng = np.random.default_rng(152)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    po = np.concatenate([[0], np.cumsum(pr[:, 2])[:-1]]).astype(np.int32)
    q = rng.standard_normal((int(cu[-1]), H_q, D)).astype(np.float16)
    out = torch.empty((q.shape[0], H_q, D), dtype=torch.float16, device="cuda")
    lse = torch.empty((q.shape[0], H_q), dtype=torch.float32, device="cuda")
    ekv_lib.ekv_prefill_attention(ctx.handle, t(q), ws_k, ws_v, total, t(cu), t(po), len(lens), int(max(lens)),
                                  0.0, out, lse)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    rk, rv, _ = og.gather_prefill(case.k_pages, case.v_pages, case.v_scales, 1, case.page_mode, 0,
                                  case.block_table, pr)
    assert np.array_equal(ws_v.cpu().numpy().view(np.uint16), rv.view(np.uint16))
    sample = {0: [0, 150, 299], 1: [96], 2: [0, 255, 256, 499]}
    ref_out, ref_lse = op.prefill_attention(q, rk, rv, cu, po, rows=sample)
    rows = np.array([cu[i] + s for i, ss in sample.items() for s in ss])
    _check(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, rows)


@pytest.mark.parametrize("variant", VARIANTS)
def test_prompt_longer_than_max_len_is_reported(ekv_lib, torch_cuda, variant):
    q, k, v, cu, po = _case([40, 200], 8, 2, 64, 153)
    out, lse, err = _run(ekv_lib, torch_cuda, q, k, v, cu, po, 8, 2, 64, max_len=64, variant=variant)
    assert err == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_SEQ_LEN)
    ref_out, ref_lse = op.prefill_attention(q, k, v, cu, po)
    _check(out, lse, ref_out, ref_lse, np.arange(40 + 64))   # the short prompt whole, the long one's first 64
    assert np.all(np.isnan(out[40 + 64:]))                    # its later rows untouched


@pytest.mark.parametrize("variant", VARIANTS)
def test_prompt_longer_than_max_len_first(ekv_lib, torch_cuda, variant):
    # the cut prompt comes first: the next prompt's rows start past n * max_len
    q, k, v, cu, po = _case([700, 40, 90], 8, 2, 128, 155)
    out, lse, err = _run(ekv_lib, torch_cuda, q, k, v, cu, po, 8, 2, 128, max_len=256, variant=variant)
    assert err == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_SEQ_LEN)
    ref_out, ref_lse = op.prefill_attention(q, k, v, cu, po)
    rows = np.r_[0:256, 700:830]
    _check(out, lse, ref_out, ref_lse, rows)
    assert np.all(np.isnan(out[256:700]))


@pytest.mark.parametrize("variant", VARIANTS)
def test_prompt_outside_the_workspace_is_reported(ekv_lib, torch_cuda, variant):
    # prompt 1's pages would run past the workspace: reported (page id), its rows left
    # untouched, the prompts before and after it computed as usual
    lens = [100, 300, 50]
    q, k, v, cu, po = _case(lens, 8, 2, 128, 157)
    po = po.copy()
    po[1] = k.shape[0] - 3                      # 19 pages from 3 before the end
    out, lse, err = _run(ekv_lib, torch_cuda, q, k, v, cu, po, 8, 2, 128, variant=variant)
    assert err == (ekv_lib.EKV_ERR_DEVICE_CHECK, ekv_lib.EKV_DETAIL_PAGE_ID)
    keep = np.r_[0:100, 400:450]
    ref_out, ref_lse = op.prefill_attention(q[keep], k, v, np.array([0, 100, 150], np.int32),
                                            np.array([po[0], po[2]], np.int32))
    _check(out[keep], lse[keep], ref_out, ref_lse, np.arange(150))
    assert np.all(np.isnan(out[100:400]))


@pytest.mark.parametrize("variant", VARIANTS)
def test_explicit_scale_empty_prompts_and_no_lse(ekv_lib, torch_cuda, variant):
    torch = torch_cuda
    lens = [0, 37, 0, 130, 1]
    H_q, H_kv, D = 8, 2, 128
    rng = np.random.default_rng(160)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    npages = [(l + 15) // 16 for l in lens]
    po = np.concatenate([[0], np.cumsum(npages)[:-1]]).astype(np.int32)
    W = sum(npages)
    q = rng.standard_normal((int(cu[-1]), H_q, D)).astype(np.float16)
    k = rng.standard_normal((W, 16, H_kv, D)).astype(np.float16)
    v = rng.standard_normal((W, 16, H_kv, D)).astype(np.float16)
    ctx = ekv_lib.Context(H_q, H_kv, D, 1, variant=variant)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = torch.full((q.shape[0], H_q, D), float("nan"), dtype=torch.float16, device="cuda")
    ekv_lib.ekv_prefill_attention(ctx.handle, t(q), t(k), t(v), W, t(cu), t(po), len(lens), max(lens), 0.07, out, None)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    ref_out, _ = op.prefill_attention(q, k, v, cu, po, sm_scale=0.07)
    e = np.abs(out.float().cpu().numpy() - ref_out).max()
    assert e <= OUT_ATOL, f"max-abs error {e:.3e}"
