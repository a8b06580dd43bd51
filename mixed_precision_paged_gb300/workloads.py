"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws inputs. It holds none of the attention, gather or demotion
arithmetic: value pages are given to both the CUDA path and the oracle as E4M3 codes
plus scales. Codes are produced with PyTorch's own float8_e4m3fn cast (a library
routine) of the drawn values divided by a calibration scale; the scale is absmax/448
over the values it covers, the plain reading of "calibrated static scales" for
synthetic data.

Shapes follow the pages: page size 16, NHD page layout [16][H_kv][D], FP16 keys, FP16
(TARGET) or FP8 E4M3 (compact) values; 32 query / 8 KV heads and head dim 128 for the
8K-token, batch-32 Qwen3-8B-like decode (knlp.io "What changes in vLLM's prefill
routing?"). Tokens past a sequence's length in its last page and pool pages no
sequence maps are poisoned with NaN (FP16 0x7E00 pattern for K and FP16 V, E4M3 0x7F
for codes) so that a stray read shows up in the output.
"""

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

PAGE_SIZE = 16
MODE_TARGET_FP16 = 0
MODE_COMPACT_E4M3 = 1
MODE_BASE = 2
SCALE_PER_TENSOR = 0
SCALE_PER_PAGE_HEAD = 1
E4M3_NAN = 0x7F
BASE_NAN = 0x7E             # high byte of the fp16 NaN 0x7E00


@dataclass
class DecodeCase:
    """Host (numpy) or device (torch) arrays of one decode call."""
    q: object                 # fp16 [B][H_q][D]
    k_pages: object           # fp16 [P][16][H_kv][D]
    v_pages: object           # uint8 [P][v_page_stride_bytes]
    v_scales: object          # fp32 [1] or [P][H_kv]
    scale_mode: int
    page_mode: object         # uint8 [P] or None
    uniform_mode: int
    block_table: object       # int32 [B][max_pages]
    seq_lens: object          # int32 [B]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    extra: dict = field(default_factory=dict)

    @property
    def batch(self):
        return int(self.seq_lens.shape[0])

    @property
    def num_pages(self):
        return int(self.k_pages.shape[0])

    @property
    def v_page_stride(self):
        return int(self.v_pages.shape[1])


def _e4m3_codes(values_f32: torch.Tensor) -> torch.Tensor:
    """Library cast to float8_e4m3fn, returned as raw uint8 codes. Values are clamped
    to +-448 first (rows outside the calibrated range saturate instead of becoming
    NaN)."""
    return values_f32.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def _nan_fp16_bytes(n):
    return np.frombuffer(np.full(n // 2, 0x7E00, dtype=np.uint16).tobytes(), dtype=np.uint8)


def make_decode_case(seq_lens, num_q_heads, num_kv_heads, head_dim, *, v_format="e4m3",
                     scale_mode=SCALE_PER_TENSOR, pool_pages=None, seed=0,
                     p_compact=0.5, v_std=1.0, poison=True, q_zero=False,
                     uniform_v=None, explicit_page_mode=None, p_base=0.0):
    """Host-side decode case.

    v_format: 'e4m3' (uniform compact pool, stride S*H_kv*D), 'fp16' (uniform TARGET
    pool, stride S*H_kv*D*2), 'mixed' (FP16-sized slots, each page compact with
    probability ``p_compact``, BASE with probability ``p_base``, else TARGET;
    ``page_mode`` returned) or 'base' (uniform BASE pool with FP16-sized slots).
    A BASE page holds the high bytes of the FP16 values (ElasticKV's BASE state).
    Pages are placed at a random permutation of a pool of ``pool_pages`` pages.
    """
    rng = np.random.default_rng(seed)
    S, H, D = PAGE_SIZE, num_kv_heads, head_dim
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = seq_lens.size
    pages_per_seq = (seq_lens.astype(np.int64) + S - 1) // S
    live = int(pages_per_seq.sum())
    max_pages = max(1, int(pages_per_seq.max()) if B else 1)
    P = int(pool_pages) if pool_pages is not None else max(live, 1)
    assert P >= live
    perm = rng.permutation(P)
    block_table = np.zeros((B, max_pages), dtype=np.int32)
    owner = np.full(P, -1, dtype=np.int64)         # sequence owning each pool page
    tail = np.zeros(P, dtype=np.int64)             # valid tokens of each live page
    k = 0
    for b in range(B):
        for j in range(int(pages_per_seq[b])):
            p = int(perm[k]); k += 1
            block_table[b, j] = p
            owner[p] = b
            tail[p] = min(S, int(seq_lens[b]) - j * S)
    # unused block-table entries point at page 0 (never read for j >= pages_per_seq)

    q = rng.standard_normal((B, num_q_heads, D)).astype(np.float16)
    if q_zero:
        q[:] = 0
    k_pages = rng.standard_normal((P, S, H, D)).astype(np.float16)
    v_true = (rng.standard_normal((P, S, H, D)) * v_std).astype(np.float32)
    if uniform_v is not None:
        v_true[:] = np.asarray(uniform_v, dtype=np.float32)
    valid = np.zeros((P, S), dtype=bool)
    for p in range(P):
        valid[p, : tail[p]] = True
    n_elem = S * H * D

    if v_format == "mixed":
        r = rng.random(P)
        modes = (r < p_compact).astype(np.uint8)
        if p_base > 0:
            modes[(r >= p_compact) & (r < p_compact + p_base)] = MODE_BASE
        if explicit_page_mode is not None:
            modes = np.asarray(explicit_page_mode, dtype=np.uint8)
        stride = 2 * n_elem
    elif v_format == "e4m3":
        modes = np.full(P, MODE_COMPACT_E4M3, dtype=np.uint8)
        stride = n_elem
    elif v_format == "fp16":
        modes = np.full(P, MODE_TARGET_FP16, dtype=np.uint8)
        stride = 2 * n_elem
    elif v_format == "base":
        modes = np.full(P, MODE_BASE, dtype=np.uint8)
        stride = 2 * n_elem
    else:
        raise ValueError(v_format)

    # calibration scales over the live values they cover
    vabs = np.abs(v_true) * valid[:, :, None, None]
    if scale_mode == SCALE_PER_TENSOR:
        a = float(vabs[modes == MODE_COMPACT_E4M3].max()) if np.any(modes == 1) else 1.0
        v_scales = np.array([a / 448.0 if a > 0 else 1.0], dtype=np.float32)
        scale_of = np.broadcast_to(v_scales[0], (P, H)).astype(np.float32)
    else:
        a = vabs.max(axis=(1, 3))
        v_scales = np.where(a > 0, a / 448.0, 1.0).astype(np.float32)
        scale_of = v_scales

    v_pages = np.zeros((P, stride), dtype=np.uint8)
    codes = _e4m3_codes(torch.from_numpy(v_true / scale_of[:, None, :, None])).numpy()
    fp16_bytes = v_true.astype(np.float16).view(np.uint8).reshape(P, -1)
    for p in range(P):
        if modes[p] == MODE_COMPACT_E4M3:
            c = codes[p].copy()
            if poison:
                c[~valid[p]] = E4M3_NAN
            v_pages[p, :n_elem] = c.reshape(-1)
            if stride > n_elem:
                v_pages[p, n_elem:] = E4M3_NAN if poison else 0
        elif modes[p] == MODE_BASE:
            hb = fp16_bytes[p].reshape(S, -1)[:, 1::2].copy()     # high byte of each value
            if poison:
                hb[~valid[p]] = BASE_NAN
            v_pages[p, :n_elem] = hb.reshape(-1)
            v_pages[p, n_elem:] = BASE_NAN if poison else 0
        else:
            fb = fp16_bytes[p].reshape(S, -1).copy()
            if poison:
                fb[~valid[p]] = _nan_fp16_bytes(fb.shape[1])
            v_pages[p, : 2 * n_elem] = fb.reshape(-1)
    if poison:
        for p in range(P):
            k_pages[p, ~valid[p]] = np.float16(np.nan)
    page_mode = modes if v_format == "mixed" else None
    uniform_mode = {"e4m3": MODE_COMPACT_E4M3, "base": MODE_BASE}.get(v_format, MODE_TARGET_FP16)
    return DecodeCase(q=q, k_pages=k_pages, v_pages=v_pages, v_scales=v_scales,
                      scale_mode=scale_mode, page_mode=page_mode, uniform_mode=uniform_mode,
                      block_table=block_table, seq_lens=seq_lens, num_q_heads=num_q_heads,
                      num_kv_heads=num_kv_heads, head_dim=head_dim,
                      extra={"modes": modes, "v_true": v_true})


# ---------------------------------------------------------------------------- configs

def tiny_config(seed=1001):
    """Tiny paged decode: 2 sequences of context 37 and 100, 4 query / 2 KV heads,
    head dim 64, K FP16 / V E4M3 with one per-tensor scale, 10 live pages at a random
    permutation of a 32-page pool (the other 22 pages and the tail rows poisoned)."""
    return make_decode_case([37, 100], 4, 2, 64, v_format="e4m3",
                            scale_mode=SCALE_PER_TENSOR, pool_pages=32, seed=seed)


def pages_shape_lens(batch=32, seed=1002):
    """Context 8192 + U{0..127} per sequence (knlp.io 8,192-token prompts, batch 32)."""
    rng = np.random.default_rng(seed)
    return (8192 + rng.integers(0, 128, size=batch)).astype(np.int32)


def mixed_lens(batch=64, seed=1003):
    """Context uniform in [512, 32768]."""
    rng = np.random.default_rng(seed)
    return rng.integers(512, 32769, size=batch).astype(np.int32)


def high_concurrency_lens(batch=256, seed=1005):
    """20% of sequences (51 of 256) at U[1, 63]; the rest ceil(LogNormal(ln 2048, 1.0))
    clamped to [1, 32768]."""
    rng = np.random.default_rng(seed)
    n_short = int(round(0.2 * batch))
    longs = np.ceil(rng.lognormal(mean=math.log(2048.0), sigma=1.0, size=batch - n_short))
    longs = np.clip(longs, 1, 32768)
    shorts = rng.integers(1, 64, size=n_short)
    lens = np.concatenate([shorts, longs]).astype(np.int32)
    return lens[rng.permutation(batch)]


def gather_demote_shape():
    """32 prompts of 8192 tokens, 8 KV heads, head dim 128: 16,384 pages gathered into a
    4,096-page workspace in 4 chunks of 8 prompts; 50% of the FP16 value pages demoted."""
    return dict(prompts=32, tokens=8192, num_kv_heads=8, head_dim=128, ws_pages=4096,
                chunk_prompts=8, demote_fraction=0.5, demote_std=math.sqrt(2.0))


# ------------------------------------------------------------ device-side generation

@dataclass
class GatherDemoteCase:
    """Device tensors of the gather/demotion workload (32 prompts x 8192 tokens)."""
    k_pages: object           # fp16 [P][16][H_kv][D]
    v8_pages: object          # uint8 [P][16*H_kv*D] E4M3 codes (uniform compact pool)
    v_scales: object          # fp32 [P][H_kv] per-(page, KV head) scales
    block_table: object       # int32 [prompts][pages per prompt], a permutation of the pool
    chunks: list              # host int32 [n][3] page ranges {seq, first, num}, one per chunk
    ws_pages: int
    v16_pages: object         # uint8 [P][16*H_kv*D*2]: the FP16 pool given to demotion
    demote_ids: object        # int32 [P * fraction] distinct page ids to demote


def device_gather_demote_case(seed=1004, device="cuda", prompts=32, tokens=8192, num_kv_heads=8,
                              head_dim=128, ws_pages=4096, chunk_prompts=8, demote_fraction=0.5,
                              demote_std=math.sqrt(2.0)):
    """The gather/demotion workload on the device: K ~ N(0, 1) fp16; V ~ N(0, 1) stored as
    E4M3 codes with absmax/448 scales per (page, KV head); prompts' pages at a random
    permutation of the pool; gather ranges of ``chunk_prompts`` whole prompts per chunk;
    a separate FP16 value pool ~ N(0, demote_std^2) and a random ``demote_fraction`` of
    its page ids for demotion."""
    S, H, D = PAGE_SIZE, num_kv_heads, head_dim
    per = (tokens + S - 1) // S
    P = prompts * per
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    k = torch.randn((P, S, H, D), generator=g, device=device).to(torch.float16)
    vv = torch.randn((P, S, H, D), generator=g, device=device)
    a = vv.abs().amax(dim=(1, 3))
    sc = torch.where(a > 0, a / 448.0, torch.ones_like(a)).contiguous()
    v8 = _e4m3_codes(vv / sc[:, None, :, None]).reshape(P, -1)
    del vv
    bt = torch.randperm(P, generator=g, device=device).to(torch.int32).reshape(prompts, per)
    chunks = [np.array([[s, 0, per] for s in range(c, min(prompts, c + chunk_prompts))], dtype=np.int32)
              for c in range(0, prompts, chunk_prompts)]
    v16 = (torch.randn((P, S, H, D), generator=g, device=device) * demote_std).to(torch.float16)
    ids = torch.randperm(P, generator=g, device=device)[: int(P * demote_fraction)].to(torch.int32)
    return GatherDemoteCase(k_pages=k, v8_pages=v8, v_scales=sc, block_table=bt, chunks=chunks,
                            ws_pages=ws_pages, v16_pages=v16.view(torch.uint8).reshape(P, -1), demote_ids=ids)


def device_decode_case(seq_lens, num_q_heads, num_kv_heads, head_dim, *, v_format="e4m3",
                       scale_mode=SCALE_PER_TENSOR, seed=0, device="cuda", p_compact=0.5,
                       pool_slack=0, poison_tail=True, p_base=0.0):
    """Same recipe as ``make_decode_case`` drawn on the device (for the full-size
    workloads, whose pools are hundreds of MB to tens of GB). Returns torch tensors."""
    S, H, D = PAGE_SIZE, num_kv_heads, head_dim
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    lens = torch.as_tensor(np.asarray(seq_lens, dtype=np.int32))
    B = lens.numel()
    pages_per_seq = (lens.to(torch.int64) + S - 1) // S
    live = int(pages_per_seq.sum())
    P = live + int(pool_slack)
    max_pages = max(1, int(pages_per_seq.max()))
    perm = torch.randperm(P, generator=gen, device=device).to(torch.int32)
    bt = torch.zeros((B, max_pages), dtype=torch.int32, device=device)
    cu = torch.zeros(B + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(pages_per_seq, 0)
    for b in range(B):
        n = int(pages_per_seq[b])
        bt[b, :n] = perm[int(cu[b]): int(cu[b]) + n]
    n_elem = S * H * D
    q = torch.randn((B, num_q_heads, D), generator=gen, device=device).to(torch.float16)
    k_pages = torch.randn((P, S, H, D), generator=gen, device=device).to(torch.float16)
    if v_format == "mixed":
        r = torch.rand(P, generator=gen, device=device)
        modes = (r < p_compact).to(torch.uint8)
        if p_base > 0:
            modes[(r >= p_compact) & (r < p_compact + p_base)] = MODE_BASE
        stride = 2 * n_elem
    elif v_format == "e4m3":
        modes = torch.ones(P, dtype=torch.uint8, device=device)
        stride = n_elem
    else:
        modes = torch.zeros(P, dtype=torch.uint8, device=device)
        stride = 2 * n_elem
    v_pages = torch.empty((P, stride), dtype=torch.uint8, device=device)
    chunk = 4096
    v_scales_pp = torch.empty((P, H), dtype=torch.float32, device=device)
    amax_all = torch.zeros((), dtype=torch.float32, device=device)
    v_chunks = []
    for p0 in range(0, P, chunk):
        p1 = min(P, p0 + chunk)
        v = torch.randn((p1 - p0, S, H, D), generator=gen, device=device)
        v_chunks.append((p0, p1, v.to(torch.float16)))
        a = v.abs().amax(dim=(1, 3))
        v_scales_pp[p0:p1] = torch.where(a > 0, a / 448.0, torch.ones_like(a))
        amax_all = torch.maximum(amax_all, a.max())
    per_tensor = torch.where(amax_all > 0, amax_all / 448.0,
                             torch.ones_like(amax_all)).reshape(1).to(torch.float32)
    for p0, p1, v16 in v_chunks:
        v = v16.float()
        m = modes[p0:p1]
        if scale_mode == SCALE_PER_TENSOR:
            codes = _e4m3_codes(v / per_tensor)
        else:
            codes = _e4m3_codes(v / v_scales_pp[p0:p1, None, :, None])
        codes = codes.reshape(p1 - p0, -1)
        fb = v16.reshape(p1 - p0, -1).view(torch.uint8)
        if stride == n_elem:
            v_pages[p0:p1] = codes
        else:
            sel = (m == MODE_COMPACT_E4M3)[:, None]
            comp = torch.cat([codes, torch.full_like(codes, E4M3_NAN)], dim=1)
            v_pages[p0:p1] = torch.where(sel, comp, fb)
            if p_base > 0:                             # BASE: the high bytes, then filler
                hb = fb[:, 1::2]
                basep = torch.cat([hb, torch.full_like(hb, BASE_NAN)], dim=1)
                v_pages[p0:p1] = torch.where((m == MODE_BASE)[:, None], basep, v_pages[p0:p1])
    if poison_tail:
        for b in range(B):
            L = int(lens[b])
            n = int(pages_per_seq[b])
            r = L - (n - 1) * S
            if n and r < S:
                p = int(bt[b, n - 1])
                k_pages[p, r:] = float("nan")
                if modes[p] == MODE_COMPACT_E4M3:
                    v_pages[p, r * H * D: n_elem] = E4M3_NAN
                elif modes[p] == MODE_BASE:
                    v_pages[p, r * H * D: n_elem] = BASE_NAN
                else:
                    v_pages[p].view(torch.float16)[r * H * D: n_elem] = float("nan")
    v_scales = per_tensor if scale_mode == SCALE_PER_TENSOR else v_scales_pp
    page_mode = modes if v_format == "mixed" else None
    uniform_mode = MODE_COMPACT_E4M3 if v_format == "e4m3" else MODE_TARGET_FP16
    return DecodeCase(q=q, k_pages=k_pages, v_pages=v_pages, v_scales=v_scales,
                      scale_mode=scale_mode, page_mode=page_mode, uniform_mode=uniform_mode,
                      block_table=bt, seq_lens=lens.to(device), num_q_heads=num_q_heads,
                      num_kv_heads=num_kv_heads, head_dim=head_dim,
                      extra={"modes": modes})


def host_copy(case: DecodeCase, batch_indices=None) -> DecodeCase:
    """Numpy copy of a device case (optionally only what ``batch_indices`` read:
    all arrays are copied whole; the oracle then reads the selected sequences)."""
    def n(x):
        return None if x is None else x.detach().cpu().numpy()
    return DecodeCase(q=n(case.q), k_pages=n(case.k_pages), v_pages=n(case.v_pages),
                      v_scales=n(case.v_scales), scale_mode=case.scale_mode,
                      page_mode=n(case.page_mode), uniform_mode=case.uniform_mode,
                      block_table=n(case.block_table), seq_lens=n(case.seq_lens),
                      num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads,
                      head_dim=case.head_dim)
