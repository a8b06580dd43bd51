"""ElasticKV pair-structured value layout and structured dispatch. Oracle only.

ElasticKV ("Does Execution Require Target KV Fidelity?"), Sec. 3.1 "Pair-Structured
Elastic KV Layout", Sec. 3.2 and App. B.3:

* Physical value slots hold one TARGET page (fp16) or two compact halves: two demoted
  pages of a pair packed into one slot free the other slot for the allocator. A value
  *location* is a half-slot index e: a TARGET page fills slot e // 2 (e even); a compact
  or BASE page's 16*H_kv*D bytes are half e % 2 of slot e // 2. A separate value block
  table gives each logical page's location (keys stay at the logical page id).
* Structured dispatch: a sequence whose modes form TARGET-BASE-TARGET is described by
  two boundaries (pages b0 <= j < b1 BASE, the others TARGET) with no per-page mode
  lookup; a batch-level indicator (has_base = 0) sends TARGET-only batches down the
  native path.
* Transitions with locations: demotion reads a TARGET page from its slot and writes its
  compact half to a destination location; promotion reads a BASE half and writes the
  TARGET page to a destination slot. Packing a pair (A, B) into A's slot is two
  transitions: A in place (half 0 of its slot), then B into half 1 of A's slot.

* The compact-prefill gather reads each page's values at its location with the same
  mode rules (``gather_prefill_elastic``).

Pins: ``tests/test_oracle_elastic.py``.
"""

import numpy as np

from . import decode, demote

PAGE_SIZE = 16
MODE_TARGET_FP16 = 0
MODE_COMPACT_E4M3 = 1
MODE_BASE = 2
OP_TO_E4M3 = 0
OP_TO_BASE = 1
OP_PROMOTE = 2


def half_bytes(v_pages, loc, n):
    """The n bytes of half-slot ``loc``."""
    loc = int(loc)
    off = (loc & 1) * n
    return v_pages[loc >> 1][off: off + n]


def slot_bytes(v_pages, loc, n):
    """The 2n bytes of the slot of an even location ``loc`` (a TARGET page)."""
    loc = int(loc)
    if loc & 1:
        raise ValueError("a TARGET page needs an even location")
    return v_pages[loc >> 1][: 2 * n]


def page_mode_of(b, j, page, page_mode, uniform_mode, boundaries, has_base):
    if not has_base:
        return MODE_TARGET_FP16
    if boundaries is not None:
        b0, b1 = int(boundaries[b][0]), int(boundaries[b][1])
        return MODE_BASE if b0 <= j < b1 else MODE_TARGET_FP16
    return uniform_mode if page_mode is None else int(page_mode[page])


def paged_decode_elastic(q, k_pages, v_pages, v_scales, scale_mode, page_mode, uniform_mode,
                         block_table, v_block_table, boundaries, has_base, seq_lens,
                         sm_scale=None, batch_indices=None):
    """Oracle of ``ekv_paged_decode_elastic``: the plain decode definition with each
    logical page's values read at its location and its mode from the boundaries, the
    mode table or the batch indicator."""
    B, H_q, D = q.shape
    S, H_kv = k_pages.shape[1], k_pages.shape[2]
    n = S * H_kv * D
    if sm_scale is None or sm_scale <= 0:
        sm_scale = 1.0 / np.sqrt(D)
    out = np.zeros((B, H_q, D))
    lse = np.full((B, H_q), -np.inf)
    for b in (range(B) if batch_indices is None else batch_indices):
        L = int(seq_lens[b])
        ks, vs = [], []
        for j in range((L + S - 1) // S):
            p = int(block_table[b][j])
            loc = int(v_block_table[b][j])
            mode = page_mode_of(b, j, p, page_mode, uniform_mode, boundaries, has_base)
            ks.append(k_pages[p].astype(np.float64))
            if mode == MODE_TARGET_FP16:
                raw = np.ascontiguousarray(slot_bytes(v_pages, loc, n))
                vs.append(decode.dequant_value_page(raw, mode, None, H_kv, D, S))
            else:
                raw = np.ascontiguousarray(half_bytes(v_pages, loc, n))
                srow = decode._scale_row(v_scales, scale_mode, p, H_kv) if mode == MODE_COMPACT_E4M3 else None
                vs.append(decode.dequant_value_page(raw, mode, srow, H_kv, D, S))
        if vs:
            K = np.concatenate(ks, axis=0)[:L]
            V = np.concatenate(vs, axis=0)[:L]
        else:
            K = V = np.zeros((0, H_kv, D))
        out[b], lse[b] = decode.attend(q[b], K, V, sm_scale)
    return out, lse


def transition(op, v_pages, page_ids, src, dst, page_mode, scale_out, low, H_kv, D, S=PAGE_SIZE):
    """Oracle of ``ekv_transition_pages``; returns updated copies of (v_pages, page_mode,
    scale_out, low). ``src`` / ``dst`` None mean in place: a TARGET page at slot
    page_ids[i] (location 2 * page_ids[i]), a BASE half at location 2 * page_ids[i].
    Demotions: src = the TARGET page's even location, dst = the half it goes to.
    Promotion: src = the BASE half, dst = the even location of the slot it fills.
    ``low``: [n][S*H_kv*D] rows (kToBase output, kPromote input), or None."""
    v = np.array(v_pages, dtype=np.uint8, copy=True)
    m = np.array(page_mode, dtype=np.uint8, copy=True)
    sc = None if scale_out is None else np.array(scale_out, copy=True)
    lw = None if low is None else np.array(low, dtype=np.uint8, copy=True)
    n = S * H_kv * D
    want = MODE_BASE if op == OP_PROMOTE else MODE_TARGET_FP16
    for i, p in enumerate(np.asarray(page_ids).reshape(-1)):
        p = int(p)
        if m[p] != want:
            continue
        s_loc = 2 * p if src is None else int(src[i])
        d_loc = 2 * p if dst is None else int(dst[i])
        if op == OP_PROMOTE:
            high = half_bytes(v, s_loc, n).astype(np.uint16)                                 # a copy
            words = (high << np.uint16(8)) | lw[i].astype(np.uint16)
            v[d_loc >> 1][: 2 * n] = words.astype("<u2").view(np.uint8)
            m[p] = MODE_TARGET_FP16
            continue
        x = np.array(slot_bytes(v, s_loc, n), copy=True).view("<f2").reshape(S, H_kv, D)   # read before writing
        if not np.all(np.isfinite(x)):
            continue                                   # reported, left TARGET
        off = (d_loc & 1) * n
        if op == OP_TO_E4M3:
            s = demote.page_scales(x)
            codes = demote.quantise_page(x, s)
            v[d_loc >> 1][off: off + n] = codes.reshape(-1)
            sc[p] = s
            m[p] = MODE_COMPACT_E4M3
        else:
            words = x.reshape(-1).view("<u2")
            v[d_loc >> 1][off: off + n] = (words >> np.uint16(8)).astype(np.uint8)
            if lw is not None:
                lw[i] = (words & np.uint16(0xFF)).astype(np.uint8)
            m[p] = MODE_BASE
    return v, m, sc, lw


def gather_prefill_elastic(k_pages, v_pages, v_scales, scale_mode, page_mode, uniform_mode, block_table,
                           v_block_table, boundaries, has_base, page_range, apply_scale=True, S=PAGE_SIZE):
    """Oracle of ``ekv_gather_prefill_elastic``: the plain gather definition
    (``gather.gather_prefill``) applied to each page's values read at its location and its
    mode taken from the boundaries, the mode table or the batch indicator. Built as a
    plain pool of the gathered pages (page w = the w-th gathered page: its K page, its
    value bytes, its mode and its scale row) and the plain gather over it."""
    from . import gather
    P, _, H_kv, D = k_pages.shape
    n = S * H_kv * D
    pages = []
    for seq, first, num in np.asarray(page_range, dtype=np.int64).reshape(-1, 3):
        for j in range(int(first), int(first) + int(num)):
            pages.append((int(seq), j))
    W = len(pages)
    k_tmp = np.zeros((max(W, 1), S, H_kv, D), dtype=np.float16)
    v_tmp = np.zeros((max(W, 1), 2 * n), dtype=np.uint8)
    m_tmp = np.zeros(max(W, 1), dtype=np.uint8)
    s_tmp = None if scale_mode != 1 or v_scales is None else np.ones((max(W, 1), H_kv), dtype=np.float32)
    for w, (b, j) in enumerate(pages):
        p = int(block_table[b][j])
        loc = int(v_block_table[b][j])
        mode = page_mode_of(b, j, p, page_mode, uniform_mode, boundaries, has_base)
        k_tmp[w] = k_pages[p]
        m_tmp[w] = mode
        if mode == MODE_TARGET_FP16:
            v_tmp[w] = slot_bytes(v_pages, loc, n)
        else:
            v_tmp[w][:n] = half_bytes(v_pages, loc, n)
        if s_tmp is not None:
            s_tmp[w] = np.asarray(v_scales, dtype=np.float32).reshape(-1, H_kv)[p]
    scales = s_tmp if s_tmp is not None else v_scales
    ws_k, ws_v, idx = gather.gather_prefill(k_tmp, v_tmp, scales, scale_mode, m_tmp, 0,
                                            np.arange(max(W, 1), dtype=np.int32).reshape(1, -1),
                                            np.array([[0, 0, W]]), apply_scale)
    return ws_k, ws_v, idx
