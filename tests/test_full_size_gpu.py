"""Parity at the full workload sizes, in the launch configuration the benchmark times.

Decode: for each benchmark workload (pages' shape, the mixed-fidelity batch, its all-FP16
control, the TARGET/BASE mix, high concurrency) two layers' pools are drawn on the device
with the benchmark's recipe and seeds, the two layer calls run back to back under
programmatic dependent launch, and every sequence of both layers is checked against the
float64 oracle, computed on the pages that sequence reads (one spawn worker per host core).

Gather and demotion (32 prompts x 8192 tokens, 16,384 pages, 8 KV heads, head dim 128;
knlp.io "What changes in vLLM's prefill routing?": at most 4,096 pages, a 256 MiB FP16
workspace; ElasticKV Sec. 3.4 "Transition protocols"): the benchmark's inputs, gathered
in 4 chunks of 4,096 pages into one 4,096-page workspace, and 8,192 of the 16,384 FP16
value pages demoted; every workspace page, every code, scale and mode byte is compared
bit for bit with the oracle, in chunks of pages so that host memory stays bounded.

Prefill (8 prompts x 8192 tokens, 32/8 heads, head dim 128, the benchmark's shape): rows on
and around the query-tile and key-block boundaries of every prompt, and random ones, every
query head, against the float64 oracle.
"""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl

from _helpers import assert_close, oracle_decode_sequences, sequence_subcases

pytestmark = pytest.mark.gpu

WORKLOADS = [  # name, lengths, Hq, Hkv, value format, scale mode, p(compact), p(BASE)
    ("pages_shape", wl.pages_shape_lens, 32, 8, "e4m3", 0, 0.5, 0.0),
    ("mixed", wl.mixed_lens, 32, 8, "mixed", 1, 0.5, 0.0),
    ("mixed_fp16_control", wl.mixed_lens, 32, 8, "fp16", 0, 0.5, 0.0),
    ("mixed_base", wl.mixed_lens, 32, 8, "mixed", 1, 0.0, 0.5),
    ("high_concurrency", wl.high_concurrency_lens, 32, 4, "e4m3", 0, 0.5, 0.0),
]


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.mark.parametrize("wi", range(len(WORKLOADS)), ids=[w[0] for w in WORKLOADS])
def test_full_size_layers_back_to_back(ekv_lib, torch_cuda, wi):
    torch = torch_cuda
    name, lens_fn, hq, hkv, fmt, scale_mode, p_compact, p_base = WORKLOADS[wi]
    lens = lens_fn()
    B = len(lens)
    layers = [wl.device_decode_case(lens, hq, hkv, 128, v_format=fmt, scale_mode=scale_mode,
                                    seed=1002 + 7919 * l, p_compact=p_compact, p_base=p_base)
              for l in range(2)]
    ctx = ekv_lib.Context(hq, hkv, 128, B, pdl=True)
    outs = [torch.empty((B, hq, 128), dtype=torch.float16, device="cuda") for _ in layers]
    lses = [torch.empty((B, hq), dtype=torch.float32, device="cuda") for _ in layers]
    for d, o, l in zip(layers, outs, lses):
        ctx.decode(d, o, l)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    for d, o, l in zip(layers, outs, lses):                    # every sequence of both layers
        ref_out, ref_lse = oracle_decode_sequences(sequence_subcases(d, range(B)))
        assert_close(o, l, ref_out, ref_lse)
    ctx.close()
    del layers, outs, lses
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def gather_demote_inputs(torch_cuda):
    case = wl.device_gather_demote_case(seed=1004)      # the benchmark's inputs
    yield case
    del case
    torch_cuda.cuda.empty_cache()


def test_gather_full_size_bit_exact(ekv_lib, torch_cuda, gather_demote_inputs):
    """16,384 K16/V8 pages gathered in 4 chunks of 4,096 into one 4,096-page FP16
    workspace, as the benchmark runs them; every workspace page of every chunk equals the
    oracle's bit for bit (K copied, V = fp16(fp32(E4M3 x scale)), indices w)."""
    from oracle import gather as og
    torch = torch_cuda
    gd = gather_demote_inputs
    P, S, H, D = gd.k_pages.shape
    ws_k = torch.empty((gd.ws_pages, S, H, D), dtype=torch.float16, device="cuda")
    ws_v = torch.empty_like(ws_k)
    idx = torch.empty((gd.ws_pages,), dtype=torch.int32, device="cuda")
    ctx = ekv_lib.Context(H, H, D, 1)
    bt = gd.block_table.cpu().numpy()
    assert len(gd.chunks) == 4 and all(int(c[:, 2].sum()) == gd.ws_pages for c in gd.chunks)
    for pr in gd.chunks:
        ws_k.fill_(float("nan"))
        ws_v.fill_(float("nan"))
        idx.fill_(-1)
        ekv_lib.ekv_gather_prefill(ctx.handle, gd.k_pages, gd.v8_pages, gd.v8_pages.shape[1], P, gd.v_scales, 1,
                                   None, 1, gd.block_table, bt.shape[1], bt.shape[0], pr, ws_k, ws_v, idx,
                                   gd.ws_pages)
        torch.cuda.synchronize()
        assert ctx.error() == (0, 0)
        # the oracle on the chunk's pages only: a compact pool in page_range order
        pages = np.concatenate([bt[s, f:f + n] for s, f, n in pr]).astype(np.int64)
        pid = torch.from_numpy(pages).cuda()
        sub_bt = np.arange(len(pages), dtype=np.int32)[None, :]
        rk, rv, ri = og.gather_prefill(gd.k_pages[pid].cpu().numpy(), gd.v8_pages[pid].cpu().numpy(),
                                       gd.v_scales[pid].cpu().numpy(), 1, None, 1, sub_bt,
                                       np.array([[0, 0, len(pages)]]))
        assert np.array_equal(ws_k.cpu().numpy().view(np.uint16), rk.view(np.uint16))
        assert np.array_equal(ws_v.cpu().numpy().view(np.uint16), rv.view(np.uint16))
        assert np.array_equal(idx.cpu().numpy(), ri)
    ctx.close()


def test_demote_full_size_bit_exact(ekv_lib, torch_cuda, gather_demote_inputs):
    """8,192 of the 16,384 FP16 value pages (values N(0, 2)) demoted to E4M3 in one call,
    as the benchmark runs it: codes, scales and mode bytes of every demoted page equal the
    oracle's bit for bit, and every other byte of the pool is untouched."""
    from oracle import demote as odm
    torch = torch_cuda
    gd = gather_demote_inputs
    P = gd.v16_pages.shape[0]
    H, D = gd.k_pages.shape[2], gd.k_pages.shape[3]
    n = 16 * H * D
    work = gd.v16_pages.clone()
    mode = torch.zeros(P, dtype=torch.uint8, device="cuda")
    scale_out = torch.zeros((P, H), dtype=torch.float32, device="cuda")
    ctx = ekv_lib.Context(H, H, D, 1)
    ids = gd.demote_ids
    ekv_lib.ekv_demote_pages(ctx.handle, work, work.shape[1], P, ids, ids.numel(), mode, scale_out)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    ids_np = ids.cpu().numpy()
    assert ids_np.size == P // 2 and np.unique(ids_np).size == ids_np.size
    m = mode.cpu().numpy()
    assert np.array_equal(np.nonzero(m)[0], np.sort(ids_np)) and set(np.unique(m)) == {0, 1}
    others = np.setdiff1d(np.arange(P), ids_np)
    po = torch.from_numpy(others).cuda()
    assert torch.equal(work[po], gd.v16_pages[po])             # pages not listed: untouched
    assert torch.equal(scale_out[po], torch.zeros_like(scale_out[po]))
    for c0 in range(0, ids_np.size, 1024):                     # the oracle in chunks of pages
        chunk = ids_np[c0:c0 + 1024].astype(np.int64)
        pc = torch.from_numpy(chunk).cuda()
        sub_v = gd.v16_pages[pc].cpu().numpy()
        k = len(chunk)
        rv, rm, rs = odm.demote_pages(sub_v, np.arange(k), np.zeros(k, np.uint8), np.zeros((k, H), np.float32),
                                      H, D)
        assert np.all(rm == 1)
        got = work[pc].cpu().numpy()
        assert np.array_equal(got[:, :n], rv[:, :n])           # the codes
        assert np.array_equal(got[:, n:], sub_v[:, n:])        # the second half of the slot unchanged
        assert np.array_equal(scale_out[pc].cpu().numpy().view(np.uint32), rs.view(np.uint32))
    ctx.close()


def test_prefill_full_size_sampled_rows(ekv_lib, torch_cuda):
    # the benchmark's prefill: 8 prompts x 8192 tokens, 32/8 heads, head dim 128, over a
    # workspace of exactly their 4,096 pages, in the persistent tcgen05 form; rows on and
    # around the query-tile and key-block boundaries (and random ones) of every prompt,
    # every query head, against the float64 oracle
    from oracle import prefill as op
    torch = torch_cuda
    n, L, H_q, H_kv, D = 8, 8192, 32, 8, 128
    pages = L // 16
    g = torch.Generator(device="cuda")
    g.manual_seed(1002)
    ws_k = torch.randn((n * pages, 16, H_kv, D), generator=g, device="cuda").to(torch.float16)
    ws_v = torch.randn((n * pages, 16, H_kv, D), generator=g, device="cuda").to(torch.float16)
    q = torch.randn((n * L, H_q, D), generator=g, device="cuda").to(torch.float16)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((n * L, H_q), float("nan"), dtype=torch.float32, device="cuda")
    cu = torch.arange(0, (n + 1) * L, L, dtype=torch.int32, device="cuda")
    po = torch.arange(0, n * pages, pages, dtype=torch.int32, device="cuda")
    ctx = ekv_lib.Context(H_q, H_kv, D, 1)
    ekv_lib.ekv_prefill_attention(ctx.handle, q, ws_k, ws_v, n * pages, cu, po, n, L, 0.0, out, lse)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    rng = np.random.default_rng(77)
    fixed = [0, 1, 127, 128, 255, 256, 4095, 4096, 8064, 8191]
    sample = {i: sorted(set(fixed + [int(x) for x in rng.integers(0, L, size=6)])) for i in range(n)}
    ref_out, ref_lse = op.prefill_attention(q.cpu().numpy(), ws_k.cpu().numpy(), ws_v.cpu().numpy(),
                                            cu.cpu().numpy(), po.cpu().numpy(), rows=sample)
    rows = np.array([i * L + s for i, ss in sample.items() for s in ss])
    o = out.float().cpu().numpy()[rows]
    e = np.abs(o - ref_out[rows]).max()
    assert e <= 2e-3, f"max-abs error {e:.3e}"
    le = np.abs(lse.cpu().numpy()[rows] - ref_lse[rows]).max()
    assert le <= 1e-3, f"lse error {le:.3e}"
