"""Shared helpers of the GPU tests: moving a host case to the device, running the
C-ABI decode, and the attention tolerance."""

import numpy as np

from mixed_precision_paged_gb300 import workloads as wl

# Attention tolerance: max-abs error of the fp16 output against the float64 oracle
# (FP32 accumulation); lse in natural-log units.
OUT_ATOL = 2e-3
LSE_ATOL = 1e-3


def to_device(case, device="cuda"):
    import torch

    def t(x):
        return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(device)
    return wl.DecodeCase(q=t(case.q), k_pages=t(case.k_pages), v_pages=t(case.v_pages),
                         v_scales=t(case.v_scales), scale_mode=case.scale_mode,
                         page_mode=t(case.page_mode), uniform_mode=case.uniform_mode,
                         block_table=t(case.block_table), seq_lens=t(case.seq_lens),
                         num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads,
                         head_dim=case.head_dim)


def gpu_decode(ctx, dcase, sm_scale=0.0, with_lse=True):
    import torch
    B, Hq, D = dcase.batch, dcase.num_q_heads, dcase.head_dim
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    ctx.decode(dcase, out, lse, sm_scale=sm_scale)
    torch.cuda.synchronize()
    return out, lse


def oracle_decode(case, batch_indices=None, sm_scale=None):
    from oracle import decode as od
    return od.paged_decode(case.q, case.k_pages, case.v_pages, case.v_scales, case.scale_mode,
                           case.page_mode, case.uniform_mode, case.block_table, case.seq_lens,
                           sm_scale=sm_scale, batch_indices=batch_indices)


def assert_close(out_gpu, lse_gpu, out_ref, lse_ref, rows=None):
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        o = o[rows]
        out_ref = out_ref[rows]
    err = np.abs(o - out_ref)
    assert np.all(np.isfinite(o)), "non-finite attention output"
    assert err.max() <= OUT_ATOL, f"max-abs error {err.max():.3e} > {OUT_ATOL}"
    if lse_gpu is not None:
        l = lse_gpu.cpu().numpy().astype(np.float64)
        if rows is not None:
            l = l[rows]
            lse_ref = lse_ref[rows]
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(l), fin)
        if fin.any():
            le = np.abs(l[fin] - lse_ref[fin]).max()
            assert le <= LSE_ATOL, f"lse error {le:.3e} > {LSE_ATOL}"
    return float(err.max())


# -------------------------------------------------------- the oracle over many sequences

def sequence_subcases(d, idx):
    """One host case per sequence of device case ``d`` in ``idx``, each holding only the
    pages that sequence reads, in a compact pool with its block table renumbered (the
    oracle then reads the same data as the kernel did)."""
    import torch
    bt = d.block_table.cpu().numpy()
    sl = d.seq_lens.cpu().numpy()
    per_page_scales = d.v_scales is not None and d.v_scales.dim() == 2
    q = d.q.cpu().numpy()
    out = []
    for b in idx:
        n = (int(sl[b]) + 15) // 16
        pages = bt[b, :n].astype(np.int64)
        pid = torch.from_numpy(pages).to(d.k_pages.device)
        out.append(wl.DecodeCase(
            q=q[b:b + 1], k_pages=d.k_pages[pid].cpu().numpy(), v_pages=d.v_pages[pid].cpu().numpy(),
            v_scales=None if d.v_scales is None else
            (d.v_scales[pid] if per_page_scales else d.v_scales).cpu().numpy(),
            scale_mode=d.scale_mode, page_mode=None if d.page_mode is None else d.page_mode[pid].cpu().numpy(),
            uniform_mode=d.uniform_mode, block_table=np.arange(max(n, 1), dtype=np.int32)[None, :],
            seq_lens=sl[b:b + 1].astype(np.int32), num_q_heads=d.num_q_heads,
            num_kv_heads=d.num_kv_heads, head_dim=d.head_dim))
    return out


def _oracle_one(case):
    out, lse = oracle_decode(case)
    return out[0], lse[0]


def oracle_decode_sequences(subcases):
    """The float64 oracle over single-sequence cases, one single-threaded spawn worker per
    host core (a pool started by spawn is safe after CUDA has been initialised)."""
    import multiprocessing as mp
    import os
    n = max(1, min(len(subcases), os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_oracle_one, subcases, chunksize=1)
    return np.stack([r[0] for r in res]), np.stack([r[1] for r in res])
