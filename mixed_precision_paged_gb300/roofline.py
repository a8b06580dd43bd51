"""Byte accounting for the roofline: algorithmic bytes of each kernel call.

Host-side arithmetic only (no kernel math). The per-token KV payload formula is the
one the knlp.io page uses for its capacity and bandwidth examples ("A bandwidth
example with explicit assumptions": 28 layers x 4 KV heads x 128 x 4 B = 56 KiB per
token for K16/V16; "Physical storage": 42,948,624,384 B hold 291,264 K16/V16 or
388,352 K16/V8 token slots per layer for 36 layers x 8 KV heads x 128).
"""

import numpy as np

PAGE_SIZE = 16


def kv_bytes_per_token(layers, num_kv_heads, head_dim, k_bytes=2, v_bytes=2):
    """KV payload bytes of one cached token across ``layers`` layers."""
    return layers * num_kv_heads * head_dim * (k_bytes + v_bytes)


def token_slots(pool_bytes, layers, num_kv_heads, head_dim, k_bytes=2, v_bytes=2):
    """Token slots per layer that a KV byte pool holds (floor)."""
    return pool_bytes // kv_bytes_per_token(layers, num_kv_heads, head_dim, k_bytes, v_bytes)


def workspace_bytes(pages, num_kv_heads, head_dim, page_size=PAGE_SIZE):
    """FP16 K + FP16 V payload of a gather workspace of ``pages`` pages."""
    return pages * page_size * num_kv_heads * head_dim * (2 + 2)


def decode_bytes(seq_lens, num_q_heads, num_kv_heads, head_dim, v_bytes_per_page,
                 per_page_scales, with_lse=False):
    """Algorithmic bytes of one ``ekv_paged_decode`` call.

    sum_b L_b * H_kv * D * (2 + v_b) for the K and V tokens actually attended (partial
    pages count tokens, not whole pages) + q + out (fp16) + block-table entries +
    seq_lens + scales (4 B per KV head of each compact page in per-page mode, else one
    float) + lse (fp32) when requested. Split-K partials are overhead, not counted.

    ``v_bytes_per_page``: an int (1 or 2) when every page has the same V element size,
    or a per-sequence list of per-page codes: 2 (TARGET fp16), 1 (E4M3, scaled) or -1
    (BASE: one byte per value, no scale).
    Returns a dict with 'kv', 'split' (what the split kernel must read) and 'total'.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    B = seq_lens.size
    pages = (seq_lens + PAGE_SIZE - 1) // PAGE_SIZE
    row = num_kv_heads * head_dim
    if isinstance(v_bytes_per_page, (int, np.integer)):
        kv = int(seq_lens.sum()) * row * (2 + int(v_bytes_per_page))
        n_compact = int(pages.sum()) if int(v_bytes_per_page) == 1 else 0
    else:
        kv = 0
        n_compact = 0
        for b in range(B):
            L = int(seq_lens[b])
            for j, vb in enumerate(v_bytes_per_page[b][: int(pages[b])]):
                ntok = min(PAGE_SIZE, L - j * PAGE_SIZE)
                kv += ntok * row * (2 + abs(int(vb)))
                n_compact += int(vb) == 1
    q = B * num_q_heads * head_dim * 2
    out = B * num_q_heads * head_dim * 2
    meta = 4 * int(pages.sum()) + 4 * B
    scales = 4 * num_kv_heads * n_compact if per_page_scales else 4
    lse = 4 * B * num_q_heads if with_lse else 0
    split = kv + q + meta + scales
    return {"kv": kv, "split": split, "total": split + out + lse}


def gather_bytes(n_pages, n_compact, num_kv_heads, head_dim, per_page_scales,
                 page_size=PAGE_SIZE):
    """Bytes read and written by ``ekv_gather_prefill`` for ``n_pages`` pages."""
    elem = page_size * num_kv_heads * head_dim
    read = n_pages * elem * 2 + n_compact * elem + (n_pages - n_compact) * elem * 2
    read += 4 * n_pages                                   # block-table entries
    read += 4 * num_kv_heads * n_compact if per_page_scales else 4
    write = n_pages * elem * 4 + 4 * n_pages              # ws_k + ws_v + ws_indices
    return read + write


def demote_bytes(n_pages, num_kv_heads, head_dim, page_size=PAGE_SIZE):
    """Bytes read and written by ``ekv_demote_pages`` for ``n_pages`` pages."""
    elem = page_size * num_kv_heads * head_dim
    read = n_pages * (elem * 2 + 4 + 1)                   # FP16 page, page id, mode
    write = n_pages * (elem + 4 * num_kv_heads + 1)       # codes, scales, mode
    return read + write


def base_transition_bytes(n_pages, num_kv_heads, head_dim, page_size=PAGE_SIZE):
    """Bytes read and written by ``ekv_demote_pages_base`` (with a low-byte backing) or
    ``ekv_promote_pages`` for ``n_pages`` pages: either way the fp16 page (2 bytes per
    value) on one side and high + low bytes (1 + 1) on the other, plus id and mode."""
    elem = page_size * num_kv_heads * head_dim
    return n_pages * (elem * 2 + elem * 2 + 4 + 2)


def append_bytes(batch, num_kv_heads, head_dim, v_bytes):
    """Bytes of one ``ekv_append_kv`` call: new K and V read (fp16), the K row written
    (fp16) and the V row written (``v_bytes`` per value), plus position, block-table
    entry and (compact) the scale of each sequence."""
    row = num_kv_heads * head_dim
    return batch * (row * (2 + 2 + 2 + v_bytes) + 4 + 4 + (4 * num_kv_heads if v_bytes == 1 else 0))


def prefill_flops(prompt_lens, num_q_heads, head_dim):
    """Algorithmic FLOPs of ``ekv_prefill_attention``: per prompt, query head and query
    position s, 2 * (s + 1) * D for QK^T and the same for PV (causal: keys 0 .. s)."""
    total = 0
    for L in prompt_lens:
        L = int(L)
        total += 4 * head_dim * num_q_heads * (L * (L + 1) // 2)
    return total

