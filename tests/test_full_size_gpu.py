"""Parity at the full workload sizes, in the launch configuration the benchmark times.

For each benchmark workload (pages' shape, the mixed-fidelity batch, its all-FP16 control,
the TARGET/BASE mix, high concurrency) two layers' pools are drawn on the device with the
benchmark's recipe and seeds, the two layer calls run back to back under programmatic
dependent launch, and sampled sequences (first, last, shortest, longest) of both layers are
checked against the float64 oracle, computed on the pages those sequences read.
"""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl

from _helpers import assert_close, oracle_decode

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


def sampled_subcase(d, idx):
    """Host case holding only the pages the sequences `idx` of device case `d` read, in a
    compact pool with the block table renumbered (the oracle then reads the same data)."""
    import torch
    bt = d.block_table.cpu().numpy()
    sl = d.seq_lens.cpu().numpy()
    rows = [bt[b, :(int(sl[b]) + 15) // 16] for b in idx]
    uniq = np.unique(np.concatenate(rows).astype(np.int64))
    where = {int(p): i for i, p in enumerate(uniq)}
    pid = torch.from_numpy(uniq).to(d.k_pages.device)
    nbt = np.zeros((len(idx), max(1, max(len(r) for r in rows))), np.int32)
    for i, r in enumerate(rows):
        nbt[i, :len(r)] = [where[int(p)] for p in r]
    per_page_scales = d.v_scales is not None and d.v_scales.dim() == 2
    return wl.DecodeCase(
        q=d.q[torch.as_tensor(idx, device=d.q.device)].cpu().numpy(),
        k_pages=d.k_pages[pid].cpu().numpy(), v_pages=d.v_pages[pid].cpu().numpy(),
        v_scales=None if d.v_scales is None else (d.v_scales[pid] if per_page_scales else d.v_scales).cpu().numpy(),
        scale_mode=d.scale_mode, page_mode=None if d.page_mode is None else d.page_mode[pid].cpu().numpy(),
        uniform_mode=d.uniform_mode, block_table=nbt, seq_lens=sl[idx].astype(np.int32),
        num_q_heads=d.num_q_heads, num_kv_heads=d.num_kv_heads, head_dim=d.head_dim)


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
    L = np.asarray(lens)
    idx = sorted({0, B - 1, int(L.argmin()), int(L.argmax())})
    for d, o, l in zip(layers, outs, lses):
        ref_out, ref_lse = oracle_decode(sampled_subcase(d, idx))
        assert_close(o[idx], l[idx], ref_out, ref_lse)
    ctx.close()
    del layers, outs, lses
    torch.cuda.empty_cache()
