"""The hot calls are CUDA-graph capturable: no host planning, no device-to-host read, no
allocation, and the split merge's tickets return to zero inside each launch. A decode and a
prefill are captured once, the inputs are then changed in place (new queries, new sequence
lengths, a page moved to another slot through the block table), and every
replay is checked against the float64 oracle."""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl
from oracle import prefill as op

from _helpers import assert_close, oracle_decode, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def test_decode_graph_replays_with_new_inputs(ekv_lib, torch_cuda):
    torch = torch_cuda
    lens = [300, 17, 900, 5, 64]
    case = wl.make_decode_case(lens, 32, 8, 128, v_format="mixed", scale_mode=1, seed=170,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 40, p_compact=0.5)
    d = to_device(case)
    ctx = ekv_lib.Context(32, 8, 128, len(lens))
    out = torch.empty((len(lens), 32, 128), dtype=torch.float16, device="cuda")
    lse = torch.empty((len(lens), 32), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ctx.decode(d, out, lse)                          # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ctx.decode(d, out, lse)
    rng = np.random.default_rng(171)
    for rep in range(4):
        if rep > 0:
            # new queries, new lengths within the block table, one page moved to a free slot
            case.q = rng.standard_normal(case.q.shape).astype(np.float16)
            # (at most the original lengths: table entries past them point at poisoned pages)
            case.seq_lens = np.array([rng.integers(1, l + 1) for l in lens], np.int32)
            used = set(case.block_table[b, j] for b in range(len(lens))
                       for j in range((int(case.seq_lens[b]) + 15) // 16))
            free = [p for p in range(case.num_pages) if p not in used]
            b = rep % len(lens)
            if free:
                j = 0
                case.k_pages[free[0]] = case.k_pages[case.block_table[b, j]]
                case.v_pages[free[0]] = case.v_pages[case.block_table[b, j]]
                if case.page_mode is not None:
                    case.page_mode[free[0]] = case.page_mode[case.block_table[b, j]]
                if case.v_scales is not None and case.scale_mode == 1:
                    case.v_scales[free[0]] = case.v_scales[case.block_table[b, j]]
                case.block_table[b, j] = free[0]
            for name in ("q", "seq_lens", "block_table", "k_pages", "v_pages", "page_mode", "v_scales"):
                src = getattr(case, name)
                if src is not None:
                    getattr(d, name).copy_(torch.from_numpy(np.ascontiguousarray(src)))
            torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert ctx.error() == (0, 0)
        ref_out, ref_lse = oracle_decode(case)
        assert_close(out, lse, ref_out, ref_lse)


def test_prefill_graph_replays_with_new_queries(ekv_lib, torch_cuda):
    torch = torch_cuda
    lens = [200, 64, 513]
    H_q, H_kv, D = 8, 2, 128
    rng = np.random.default_rng(172)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    npages = [(l + 15) // 16 for l in lens]
    po = np.concatenate([[0], np.cumsum(npages)[:-1]]).astype(np.int32)
    W = sum(npages)
    k = rng.standard_normal((W, 16, H_kv, D)).astype(np.float16)
    v = rng.standard_normal((W, 16, H_kv, D)).astype(np.float16)
    q = rng.standard_normal((int(cu[-1]), H_q, D)).astype(np.float16)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    qd, kd, vd, cud, pod = t(q), t(k), t(v), t(cu), t(po)
    ctx = ekv_lib.Context(H_q, H_kv, D, 1)
    out = torch.empty((q.shape[0], H_q, D), dtype=torch.float16, device="cuda")
    lse = torch.empty((q.shape[0], H_q), dtype=torch.float32, device="cuda")
    ekv_lib.ekv_prefill_attention(ctx.handle, qd, kd, vd, W, cud, pod, len(lens), max(lens), 0.0, out, lse)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ekv_lib.ekv_prefill_attention(ctx.handle, qd, kd, vd, W, cud, pod, len(lens), max(lens), 0.0, out, lse)
    for rep in range(3):
        if rep > 0:
            q = rng.standard_normal(q.shape).astype(np.float16)
            qd.copy_(torch.from_numpy(q))
            torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert ctx.error() == (0, 0)
        rows = {0: [0, 199], 1: [63], 2: [0, 255, 256, 512]}
        ref_out, ref_lse = op.prefill_attention(q, k, v, cu, po, rows=rows)
        idx = np.array([cu[i] + s for i, ss in rows.items() for s in ss])
        o = out.float().cpu().numpy()
        assert np.abs(o[idx] - ref_out[idx]).max() <= 2e-3
        assert np.abs(lse.cpu().numpy()[idx] - ref_lse[idx]).max() <= 1e-3
