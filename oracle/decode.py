"""Paged GQA decode attention over a mixed-fidelity KV cache, in float64. Oracle only.

Plain definition (no blocking, no split, no online softmax):

* Paged layout: a request's tokens live in fixed-size physical pages reached through
  its block table, logical page j -> physical page block_table[b][j] (ElasticKV
  Sec. 2.1 "Paged KV Cache Management"); page size 16 and NHD layout, i.e. a page
  is [16 tokens][H_kv heads][D] (knlp.io "What changes in vLLM's prefill routing?",
  the measured-route paragraph).
* Keys are FP16. Each value page is TARGET (FP16) or compact (FP8 E4M3 codes times a
  scale); "existing value scales still apply in attention" (knlp.io, same section).
  Page mode is per physical page (ElasticKV Sec. 3.2: TARGET and BASE pages are
  loaded with different semantics behind one attention interface).
* GQA: query head h_q reads KV head floor(h_q / G), G = H_q / H_kv.
* One decode query per sequence attends to all L_b cached tokens; no mask.
* z_t = sm_scale * <q, k_t>, out = sum_t softmax(z)_t v_t, lse = log sum_t exp z_t.
"""

import math

import numpy as np

from . import base, e4m3

PAGE_SIZE = 16
MODE_TARGET_FP16 = 0
MODE_COMPACT_E4M3 = 1
SCALE_PER_TENSOR = 0
SCALE_PER_PAGE_HEAD = 1


def dequant_value_page(v_page_bytes, mode, scale_row, H_kv, D, S=PAGE_SIZE):
    """Float64 [S][H_kv][D] values of one physical value page.

    ``v_page_bytes``: the page's uint8 slot. TARGET reads its first S*H_kv*D*2 bytes
    as little-endian FP16; compact reads its first S*H_kv*D bytes as E4M3 codes and
    multiplies by the scale of each KV head (``scale_row``: float[H_kv]).
    """
    n = S * H_kv * D
    if mode == MODE_TARGET_FP16:
        raw = np.ascontiguousarray(v_page_bytes[: 2 * n])
        return raw.view("<f2").astype(np.float64).reshape(S, H_kv, D)
    if mode == MODE_COMPACT_E4M3:
        codes = v_page_bytes[:n].reshape(S, H_kv, D)
        s = np.asarray(scale_row, dtype=np.float64).reshape(1, H_kv, 1)
        return e4m3.decode(codes) * s
    if mode == base.MODE_BASE:
        return base.base_value(v_page_bytes[:n]).reshape(S, H_kv, D)
    raise ValueError(f"unknown page mode {mode}")


def _scale_row(v_scales, scale_mode, page, H_kv):
    if scale_mode == SCALE_PER_TENSOR:
        return np.full(H_kv, float(np.asarray(v_scales).reshape(-1)[0]))
    if scale_mode == SCALE_PER_PAGE_HEAD:
        return np.asarray(v_scales, dtype=np.float64).reshape(-1, H_kv)[page]
    raise ValueError(f"unknown scale mode {scale_mode}")


def sequence_kv(b, k_pages, v_pages, v_scales, scale_mode, page_mode, uniform_mode,
                block_table, seq_lens):
    """Contiguous float64 K [L][H_kv][D] and V [L][H_kv][D] of sequence ``b``."""
    S, H_kv, D = k_pages.shape[1:]
    L = int(seq_lens[b])
    n_pages = (L + S - 1) // S
    ks, vs = [], []
    for j in range(n_pages):
        p = int(block_table[b][j])
        mode = uniform_mode if page_mode is None else int(page_mode[p])
        ks.append(k_pages[p].astype(np.float64))
        srow = _scale_row(v_scales, scale_mode, p, H_kv) if mode == MODE_COMPACT_E4M3 else None
        vs.append(dequant_value_page(v_pages[p], mode, srow, H_kv, D, S))
    if n_pages == 0:
        return np.zeros((0, H_kv, D)), np.zeros((0, H_kv, D))
    K = np.concatenate(ks, axis=0)[:L]
    V = np.concatenate(vs, axis=0)[:L]
    return K, V


def attend(q_b, K, V, sm_scale):
    """Softmax attention of one sequence's queries q_b [H_q][D] over K, V [L][H_kv][D].

    Returns (out [H_q][D], lse [H_q]) in float64. L == 0 gives zeros and -inf.
    """
    H_q, D = q_b.shape
    L, H_kv, _ = K.shape
    G = H_q // H_kv
    out = np.zeros((H_q, D))
    lse = np.full(H_q, -np.inf)
    if L == 0:
        return out, lse
    for hq in range(H_q):
        h = hq // G
        z = (K[:, h, :] @ q_b[hq].astype(np.float64)) * sm_scale
        m = z.max()
        w = np.exp(z - m)
        out[hq] = (w @ V[:, h, :]) / w.sum()
        lse[hq] = m + math.log(w.sum())
    return out, lse


def paged_decode(q, k_pages, v_pages, v_scales, scale_mode, page_mode, uniform_mode,
                 block_table, seq_lens, sm_scale=None, batch_indices=None):
    """Oracle of ``ekv_paged_decode``.

    q: float16 [B][H_q][D]; k_pages: float16 [P][16][H_kv][D];
    v_pages: uint8 [P][v_page_stride_bytes]; v_scales: float32 [1] or [P][H_kv];
    page_mode: uint8 [P] or None (then every page has ``uniform_mode``);
    block_table: int32 [B][max_pages]; seq_lens: int32 [B].
    ``sm_scale`` None or <= 0 means 1/sqrt(D). ``batch_indices`` restricts the work to
    some sequences (the others are left zero / -inf).
    Returns out float64 [B][H_q][D], lse float64 [B][H_q] (natural log).
    """
    B, H_q, D = q.shape
    if sm_scale is None or sm_scale <= 0:
        sm_scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, H_q, D))
    lse = np.full((B, H_q), -np.inf)
    for b in (range(B) if batch_indices is None else batch_indices):
        K, V = sequence_kv(b, k_pages, v_pages, v_scales, scale_mode, page_mode,
                           uniform_mode, block_table, seq_lens)
        out[b], lse[b] = attend(q[b], K, V, sm_scale)
    return out, lse
