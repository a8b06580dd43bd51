"""FP16 causal prefill over the gathered workspace, in float64. Oracle only.

knlp.io "Asymmetric K16/V8 KV cache", "What changes in vLLM's prefill routing?": the
stored K16/V8 pages of fresh prompts are gathered into one bounded FP16 workspace and a
native FP16 prefill runs over it: FP16 query, key and value, whole prompts with no
cached prefix, causal attention, no sliding window, sinks or soft caps.

Prompt i has len_i = cu_seqlens[i+1] - cu_seqlens[i] tokens; its queries are rows
cu_seqlens[i] .. of q [T][H_q][D]; its keys and values are the workspace pages
page_off[i], page_off[i] + 1, ... (token t at page page_off[i] + t // 16, row t % 16),
in the [W][16][H_kv][D] layout the gather writes. Query position s of prompt i, head
h_q, attends keys 0 .. s of KV head h_q // G:
  out = sum_{t <= s} softmax_t(sm_scale * <q_s, k_t>) v_t,  lse = log sum_{t <= s} e^(.)
"""

import math

import numpy as np

PAGE_SIZE = 16


def prefill_attention(q, ws_k, ws_v, cu_seqlens, page_off, sm_scale=None, prompts=None, rows=None):
    """Returns out float64 [T][H_q][D] and lse float64 [T][H_q] (natural log). ``prompts``
    restricts the work to some prompts and ``rows`` (a dict prompt -> list of query
    positions) to some of their query rows; the rest stays 0 / -inf."""
    T, H_q, D = q.shape
    H_kv = ws_k.shape[2]
    G = H_q // H_kv
    if sm_scale is None or sm_scale <= 0:
        sm_scale = 1.0 / math.sqrt(D)
    out = np.zeros((T, H_q, D))
    lse = np.full((T, H_q), -np.inf)
    n = len(cu_seqlens) - 1
    for i in (range(n) if prompts is None else prompts):
        L = int(cu_seqlens[i + 1]) - int(cu_seqlens[i])
        if L == 0:
            continue
        pages = int(page_off[i]) + np.arange((L + PAGE_SIZE - 1) // PAGE_SIZE)
        K = ws_k[pages].astype(np.float64).reshape(-1, H_kv, D)[:L]
        V = ws_v[pages].astype(np.float64).reshape(-1, H_kv, D)[:L]
        for s in (range(L) if rows is None or i not in rows else rows[i]):
            row = int(cu_seqlens[i]) + s
            for hq in range(H_q):
                h = hq // G
                z = (K[: s + 1, h, :] @ q[row, hq].astype(np.float64)) * sm_scale
                m = z.max()
                w = np.exp(z - m)
                out[row, hq] = (w @ V[: s + 1, h, :]) / w.sum()
                lse[row, hq] = m + math.log(w.sum())
    return out, lse
