"""GPU parity of ekv_paged_decode (through the C ABI) against the float64 oracle.

Tolerance: max-abs 2e-3 on the fp16 output, 1e-3 on lse. Inputs are seeded; unused
pool pages and tail rows are NaN-poisoned, so a stray read fails the test.
"""

import math

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl

from _helpers import assert_close, gpu_decode, oracle_decode, to_device

pytestmark = pytest.mark.gpu

VARIANTS = [0, 1]          # 0 tensor-core consumer, 1 CUDA-core consumer


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def make_ctx(ekv_lib, case, variant, max_batch=None):
    return ekv_lib.Context(case.num_q_heads, case.num_kv_heads, case.head_dim,
                           max_batch or max(1, case.batch), variant=variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_config(ekv_lib, torch_cuda, variant):
    case = wl.tiny_config()
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    assert ctx.error() == (0, 0)


SHAPES = [  # (lens, Hq, Hkv, D)
    ([1, 2, 15, 16, 17], 8, 8, 128),
    ([33, 100], 32, 8, 128),
    ([5, 64, 99], 32, 4, 128),
    ([37, 100], 4, 2, 64),
    ([48, 1, 77, 31], 8, 1, 64),
    ([90], 2, 2, 128),
    ([16, 32], 16, 2, 64),
    ([70, 3], 6, 2, 128),
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("fmt,scale_mode", [("e4m3", 0), ("e4m3", 1), ("fp16", 0), ("mixed", 1), ("mixed", 0)])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_small_shapes(ekv_lib, torch_cuda, variant, fmt, scale_mode, shape):
    lens, hq, hkv, d = SHAPES[shape]
    pages = sum((l + 15) // 16 for l in lens)
    case = wl.make_decode_case(lens, hq, hkv, d, v_format=fmt, scale_mode=scale_mode,
                               pool_pages=pages + 5, seed=100 + shape)
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    assert ctx.error() == (0, 0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_long_sequences_split_across_many_ctas(ekv_lib, torch_cuda, variant):
    # 6 sequences of up to ~5000 tokens: every sequence spans several CTAs, several CTAs
    # span sequence boundaries, and the last pages are ragged.
    lens = [5000, 1, 3333, 17, 4096, 2500]
    case = wl.make_decode_case(lens, 32, 8, 128, v_format="mixed", scale_mode=1,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 3, seed=7)
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("lens,hq,hkv,d", [([4000], 8, 1, 128), ([3000, 5], 16, 2, 64)])
def test_one_long_sequence_over_hundreds_of_ranges(ekv_lib, torch_cuda, variant, lens, hq, hkv, d):
    # with few KV heads every warp streams its own page range (#SMs * 8 / H_kv ranges of
    # about one page here), so one sequence is split into hundreds of records and its
    # merge runs in many waves of staged records
    case = wl.make_decode_case(lens, hq, hkv, d, v_format="mixed", scale_mode=1,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 3, seed=11 + hkv)
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    assert ctx.error() == (0, 0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_many_short_sequences(ekv_lib, torch_cuda, variant):
    rng = np.random.default_rng(8)
    lens = list(rng.integers(0, 40, size=300))
    lens[0] = 0
    lens[-1] = 0
    case = wl.make_decode_case(lens, 32, 4, 128, v_format="e4m3", scale_mode=0,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 1, seed=9)
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    o = out.float().cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[-1] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[[0, -1]]))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("hkv", [1, 8])
def test_ranges_over_empty_sequences(ekv_lib, torch_cuda, variant, hkv):
    # every sequence, empty ones included, weighs a fixed cost in the page stream that is cut
    # into equal ranges, so with hundreds of empty and one-token sequences whole ranges hold
    # no page at all, and one long sequence at the end is still split over many ranges
    rng = np.random.default_rng(30 + hkv)
    lens = [int(x) for x in rng.choice([0, 0, 0, 1, 2], size=700)] + [3000]
    lens[350] = 0
    case = wl.make_decode_case(lens, 8 * hkv, hkv, 128, v_format="mixed", scale_mode=1,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 2, seed=40 + hkv,
                               p_base=0.25)
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    empty = np.array(lens) == 0
    assert np.all(out.float().cpu().numpy()[empty] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[empty]))
    assert ctx.error() == (0, 0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_batch_larger_than_the_range_count(ekv_lib, torch_cuda, variant):
    # 1,200 short sequences with 8 KV heads: fewer ranges than sequences, so each range
    # holds many whole sequences and writes them without a merge
    rng = np.random.default_rng(33)
    lens = [int(x) for x in rng.integers(0, 50, size=1200)]
    case = wl.make_decode_case(lens, 16, 8, 64, v_format="mixed", scale_mode=0,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 2, seed=34)
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    assert ctx.error() == (0, 0)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("offset", [-1, 0, 1, 7, "2nv-1"])
def test_cost_stream_around_the_range_count(ekv_lib, torch_cuda, variant, offset):
    # The cost stream (T positions: pages + 2 per sequence start) is cut into one range per
    # (CTA, page group) of ceil(T / nv) positions, so around T = nv the last ranges hold
    # one position or none. Lengths are drawn so that T lands just around nv.
    ctx0 = make_ctx(ekv_lib, wl.make_decode_case([16], 8, 8, 64, seed=1), variant)
    _, nv = ekv_lib.ekv_query(ctx0.handle)              # 8 KV heads: one page group per CTA
    batch = 24
    target = 2 * nv - 1 if offset == "2nv-1" else nv + offset
    pages = target - 2 * batch
    rng = np.random.default_rng(70 + (0 if offset == "2nv-1" else offset + 2))
    cuts = np.sort(rng.integers(0, pages + 1, size=batch - 1))
    per_seq = np.diff(np.concatenate([[0], cuts, [pages]]))
    lens = [int(n * 16 - (rng.integers(0, 16) if n > 0 else 0)) for n in per_seq]
    assert sum((l + 15) // 16 for l in lens) + 2 * batch == target
    case = wl.make_decode_case(lens, 32, 8, 64, v_format="mixed", scale_mode=1,
                               pool_pages=pages + 3, seed=71)
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    assert ctx.error() == (0, 0)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("fmt,scale_mode", [("fp16", 0), ("mixed", 1), ("e4m3", 0)])
def test_scores_growing_along_the_sequence(ekv_lib, torch_cuda, variant, fmt, scale_mode):
    # keys scaled up page by page, so the page max of the scores keeps passing the running
    # reference and the lazy re-base (FP16 / mixed pools) fires every few pages, mid-segment
    lens = [900, 37, 1600]
    case = wl.make_decode_case(lens, 32, 8, 128, v_format=fmt, scale_mode=scale_mode,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 3, seed=60,
                               p_base=0.25 if fmt == "mixed" else 0.0)
    k = case.k_pages.astype(np.float32)
    for b, L in enumerate(lens):
        for j in range((L + 15) // 16):
            k[case.block_table[b, j]] *= 1.0 + 0.25 * j
    case.k_pages = k.astype(np.float16)
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)
    assert ctx.error() == (0, 0)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("fmt", ["fp16", "mixed"])
def test_one_late_dominant_token(ekv_lib, torch_cuda, variant, fmt):
    # one key far along the sequence aligned with the query: its score is ~40 (log2 units)
    # above the rest, so the reference jumps once by far more than the re-base threshold and
    # the output is essentially that token's value
    lens = [700, 333]
    case = wl.make_decode_case(lens, 8, 2, 128, v_format=fmt, scale_mode=1, seed=61,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 3)
    for b, t in [(0, 650), (1, 100)]:
        page, row = case.block_table[b, t // 16], t % 16
        for hk in range(2):
            qd = case.q[b, hk * 4].astype(np.float32)
            case.k_pages[page, row, hk] = (qd * (30.0 / np.linalg.norm(qd))).astype(np.float16)
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    ref_out, ref_lse = oracle_decode(case)
    assert_close(out, lse, ref_out, ref_lse)


@pytest.fixture(scope="module")
def max_batch_case():
    rng = np.random.default_rng(35)
    lens = [int(x) for x in rng.integers(0, 40, size=4096)]
    return lens, wl.make_decode_case(lens, 32, 8, 128, v_format="mixed", scale_mode=1, seed=36,
                                     pool_pages=sum((l + 15) // 16 for l in lens) + 2, p_base=0.2)


@pytest.mark.parametrize("variant", VARIANTS)
def test_maximum_batch(ekv_lib, torch_cuda, variant, max_batch_case):
    # the largest batch a context takes (4,096 sequences: the prefix sums fill 16 KiB of
    # shared memory beside FP16-sized ring slots), short mixed-pool sequences, some empty;
    # sampled sequences against the oracle, every empty one checked for zeros
    lens, case = max_batch_case
    ctx = make_ctx(ekv_lib, case, variant)
    out, lse = gpu_decode(ctx, to_device(case))
    assert ctx.error() == (0, 0)
    idx = np.concatenate([np.arange(0, 4096, 97), [4095]])
    ref_out, ref_lse = oracle_decode(case, batch_indices=idx)
    assert_close(out[idx], lse[idx], ref_out[idx], ref_lse[idx])
    empty = np.array(lens) == 0
    assert np.all(out.float().cpu().numpy()[empty] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[empty]))


@pytest.mark.parametrize("variant", VARIANTS)
def test_single_token_returns_value_times_scale(ekv_lib, torch_cuda, variant):
    case = wl.make_decode_case([1, 1, 1], 16, 4, 128, v_format="mixed", scale_mode=1,
                               pool_pages=6, seed=11)
    ctx = make_ctx(ekv_lib, case, variant)
    out, _ = gpu_decode(ctx, to_device(case))
    ref, _ = oracle_decode(case)
    o = out.float().cpu().numpy().astype(np.float64)
    # fp32 product then one fp16 rounding: within one fp16 ulp of the exact value
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -14))) - 10)
    assert np.all(np.abs(o - ref) <= ulp)


@pytest.mark.parametrize("variant", VARIANTS)
def test_block_table_permutation_is_bit_identical(ekv_lib, torch_cuda, variant):
    import torch
    lens = [200, 37, 513]
    case = wl.make_decode_case(lens, 32, 8, 128, v_format="mixed", scale_mode=1,
                               pool_pages=60, seed=12)
    ctx = make_ctx(ekv_lib, case, variant)
    out0, lse0 = gpu_decode(ctx, to_device(case))
    perm = np.random.default_rng(13).permutation(case.num_pages)
    c2 = wl.DecodeCase(**{**case.__dict__})
    c2.k_pages = np.empty_like(case.k_pages); c2.k_pages[perm] = case.k_pages
    c2.v_pages = np.empty_like(case.v_pages); c2.v_pages[perm] = case.v_pages
    c2.v_scales = np.empty_like(case.v_scales); c2.v_scales[perm] = case.v_scales
    c2.page_mode = np.empty_like(case.page_mode); c2.page_mode[perm] = case.page_mode
    c2.block_table = perm[case.block_table].astype(np.int32)
    out1, lse1 = gpu_decode(ctx, to_device(c2))
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_variants_agree(ekv_lib, torch_cuda):
    case = wl.make_decode_case([300, 7, 1000], 32, 8, 128, v_format="mixed", scale_mode=1,
                               pool_pages=90, seed=14)
    a, la = gpu_decode(make_ctx(ekv_lib, case, 0), to_device(case))
    b, lb = gpu_decode(make_ctx(ekv_lib, case, 1), to_device(case))
    assert (a.float() - b.float()).abs().max().item() <= 2e-3
    assert (la - lb).abs().max().item() <= 1e-3


def test_launch_floor(ekv_lib, torch_cuda):
    # the empty launch of the split kernel's shape: a few microseconds between its events,
    # far below one decode launch; bad repetition counts are refused
    ctx = ekv_lib.Context(32, 8, 128, 32)
    ms = ekv_lib.ekv_profile_launch_floor(ctx.handle, 16)
    assert 0.0 < ms < 0.1
    for reps in (0, 1025):
        with pytest.raises(RuntimeError):
            ekv_lib.ekv_profile_launch_floor(ctx.handle, reps)
    assert ctx.error() == (0, 0)


def test_explicit_sm_scale(ekv_lib, torch_cuda):
    case = wl.make_decode_case([50, 20], 8, 2, 64, v_format="e4m3", pool_pages=6, seed=15)
    ctx = make_ctx(ekv_lib, case, 0)
    out, lse = gpu_decode(ctx, to_device(case), sm_scale=0.3)
    ref_out, ref_lse = oracle_decode(case, sm_scale=0.3)
    assert_close(out, lse, ref_out, ref_lse)


def test_all_target_mixed_template_matches_native(ekv_lib, torch_cuda):
    """An all-TARGET pool through the per-page-mode template equals the native path."""
    import torch
    lens = [400, 90]
    case = wl.make_decode_case(lens, 32, 8, 128, v_format="fp16", pool_pages=32, seed=16)
    ctx = make_ctx(ekv_lib, case, 0)
    native, _ = gpu_decode(ctx, to_device(case))
    mixed = wl.DecodeCase(**{**case.__dict__})
    mixed.page_mode = np.zeros(case.num_pages, dtype=np.uint8)
    out, _ = gpu_decode(ctx, to_device(mixed))
    assert torch.equal(native, out)
