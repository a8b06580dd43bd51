"""K16/V8 cache writer: append one token per sequence. Oracle only.

knlp.io "Asymmetric K16/V8 KV cache", the implementation checks ("vLLM cache writer:
K bit-exact, V within FP8 noise") and the production list ("cache writer"): each decode
step stores the new token's key and value into the paged cache, the key as FP16 and
the value in the representation of its page. ElasticKV Sec. 3.2: newly appended KV is
written in TARGET form (the writer simply follows the page's mode; a page that the
caller keeps TARGET receives FP16 bits).

For sequence b with position t = positions[b] (t < 0: no token this step):
  page = block_table[b][t // 16], row = t % 16;
  K[page][row] = k_new[b] (bits);
  TARGET page:  V16[page][row] = v_new[b] (bits);
  E4M3 page:    V8[page][row][h][d] = E4M3_rn_satfinite(fp32_rn(v / s)), s the page's
                existing scale (per tensor, or per (page, KV head)); a KV head whose scale
                is not positive finite keeps its old bytes (reported on the GPU);
  BASE page:    the high bytes of the FP16 values.
fp32_rn(v / s) is computed in float64 then rounded to float32: double rounding is
innocuous for division here (53 >= 2*24 + 2), so this equals IEEE fp32 division.
"""

import numpy as np

from . import e4m3

PAGE_SIZE = 16
MODE_TARGET_FP16 = 0
MODE_COMPACT_E4M3 = 1
MODE_BASE = 2
SCALE_PER_TENSOR = 0


def append_token(k_pages, v_pages, v_scales, scale_mode, page_mode, uniform_mode, block_table,
                 positions, k_new, v_new):
    """Returns (k_pages', v_pages') with the new tokens written."""
    k = np.array(k_pages, copy=True)
    v = np.array(v_pages, dtype=np.uint8, copy=True)
    P, S, H, D = k.shape
    row_elems = H * D
    for b, t in enumerate(np.asarray(positions).reshape(-1)):
        t = int(t)
        if t < 0:
            continue
        page = int(block_table[b][t // S])
        row = t % S
        k[page, row] = np.asarray(k_new[b], dtype=np.float16)
        mode = uniform_mode if page_mode is None else int(page_mode[page])
        x = np.asarray(v_new[b], dtype=np.float16).reshape(H, D)
        if mode == MODE_TARGET_FP16:
            off = row * row_elems * 2
            v[page, off: off + row_elems * 2] = x.reshape(-1).view(np.uint8)
        elif mode == MODE_BASE:
            off = row * row_elems
            v[page, off: off + row_elems] = (x.reshape(-1).view("<u2") >> np.uint16(8)).astype(np.uint8)
        elif mode == MODE_COMPACT_E4M3:
            if scale_mode == SCALE_PER_TENSOR:
                s = np.full(H, float(np.asarray(v_scales).reshape(-1)[0]))
            else:
                s = np.asarray(v_scales, dtype=np.float64).reshape(-1, H)[page]
            ok = np.isfinite(s) & (s > 0)                   # per KV head
            s_safe = np.where(ok, s, 1.0)
            y = (x.astype(np.float64) / s_safe.reshape(H, 1)).astype(np.float32).astype(np.float64)
            nan = np.isnan(y)
            y = np.clip(np.where(nan, 0.0, y), -e4m3.E4M3_MAX, e4m3.E4M3_MAX)   # satfinite: +-inf -> +-448
            codes = e4m3.encode_rne_satfinite(y)
            codes[nan] = 0x7F                                                  # NaN stays NaN
            off = row * row_elems
            cur = v[page, off: off + row_elems].reshape(H, D)
            v[page, off: off + row_elems] = np.where(ok.reshape(H, 1), codes, cur).reshape(-1)
        else:
            raise ValueError(f"unknown page mode {mode}")
    return k, v
