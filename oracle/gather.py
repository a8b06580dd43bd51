"""Compact-prefill gather of K16/V8 pages into an FP16 workspace. Oracle only, exact.

knlp.io "What changes in vLLM's prefill routing?": compact prefill gathers the stored
K16/V8 pages of the fresh prompts into one bounded FP16 workspace (at most 4,096
pages, a 256 MiB payload) for a native FP16 prefill, casting V8 -> FP16; the cast
keeps the quantisation error.

Definition used (each step exact or a single IEEE rounding):

* K page: copied bit for bit.
* TARGET value page: copied bit for bit.
* compact value page, scale applied: fp16_RN(fp32_RN(E4M3(code) * s)). The float64
  product of a 4-significant-bit value and a 24-bit float is exact, so rounding it to
  float32 equals an IEEE float32 multiply; a second rounding to float16 follows.
* compact value page, scale not applied: fp16(E4M3(code)), exact (every E4M3 value is
  an FP16 value).
* Pages are placed in consecutive workspace slots in ``page_range`` order;
  ``ws_indices[w] = w`` is the workspace page table the FP16 prefill reads.
"""

import numpy as np

from . import base, e4m3

PAGE_SIZE = 16
MODE_TARGET_FP16 = 0
MODE_COMPACT_E4M3 = 1
SCALE_PER_TENSOR = 0
SCALE_PER_PAGE_HEAD = 1


def gather_prefill(k_pages, v_pages, v_scales, scale_mode, page_mode, uniform_mode,
                   block_table, page_range, apply_scale=True):
    """Oracle of ``ekv_gather_prefill``.

    page_range: int [n][3] rows (seq, first_page, num_pages).
    Returns ws_k float16 [W][16][H_kv][D], ws_v float16 [W][16][H_kv][D],
    ws_indices int32 [W], with W the total number of gathered pages.
    """
    P, S, H_kv, D = k_pages.shape
    n_elem = S * H_kv * D
    slots = []
    for seq, first, num in np.asarray(page_range, dtype=np.int64).reshape(-1, 3):
        for j in range(int(num)):
            slots.append(int(block_table[int(seq)][int(first) + j]))
    W = len(slots)
    ws_k = np.zeros((W, S, H_kv, D), dtype=np.float16)
    ws_v = np.zeros((W, S, H_kv, D), dtype=np.float16)
    for w, p in enumerate(slots):
        ws_k[w] = k_pages[p]
        mode = uniform_mode if page_mode is None else int(page_mode[p])
        if mode == MODE_TARGET_FP16:
            ws_v[w] = np.ascontiguousarray(v_pages[p][: 2 * n_elem]).view("<f2").reshape(S, H_kv, D)
        elif mode == base.MODE_BASE:
            # ElasticKV BASE: high byte in place, low byte zero (exact, no scale)
            ws_v[w] = base.base_value(v_pages[p][:n_elem]).astype(np.float16).reshape(S, H_kv, D)
        else:
            vals = e4m3.decode(v_pages[p][:n_elem]).reshape(S, H_kv, D)
            if apply_scale:
                if scale_mode == SCALE_PER_TENSOR:
                    s = np.full(H_kv, np.float64(np.asarray(v_scales).reshape(-1)[0]))
                else:
                    s = np.asarray(v_scales, dtype=np.float64).reshape(-1, H_kv)[p]
                prod = vals * s.reshape(1, H_kv, 1)          # exact in float64
                ws_v[w] = prod.astype(np.float32).astype(np.float16)
            else:
                ws_v[w] = vals.astype(np.float16)
    return ws_k, ws_v, np.arange(W, dtype=np.int32)
