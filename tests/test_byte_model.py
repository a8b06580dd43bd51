"""Byte accounting pinned to the numbers the knlp.io page prints (tests/golden)."""

import json
import os

import numpy as np

from mixed_precision_paged_gb300 import roofline as rf

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "byte_model.json")))


def test_token_slots_per_layer():
    g = GOLD["qwen3_8b_slots"]
    args = (g["pool_bytes"], g["layers"], g["num_kv_heads"], g["head_dim"])
    assert rf.token_slots(*args, k_bytes=2, v_bytes=2) == g["slots_k16v16"]
    assert rf.token_slots(*args, k_bytes=2, v_bytes=1) == g["slots_k16v8"]
    # the page's pool divides exactly in both layouts
    per16 = rf.kv_bytes_per_token(g["layers"], g["num_kv_heads"], g["head_dim"], 2, 2)
    per8 = rf.kv_bytes_per_token(g["layers"], g["num_kv_heads"], g["head_dim"], 2, 1)
    assert g["pool_bytes"] % per16 == 0 and g["pool_bytes"] % per8 == 0


def test_bandwidth_example():
    g = GOLD["qwen25_7b_bandwidth"]
    per = rf.kv_bytes_per_token(g["layers"], g["num_kv_heads"], g["head_dim"], 2, 2)
    assert per == g["bytes_per_token_k16v16"]
    for name, (kb, vb) in {"k16v16": (2, 2), "k16v8": (2, 1), "k8v8": (1, 1)}.items():
        total = g["tokens"] * rf.kv_bytes_per_token(g["layers"], g["num_kv_heads"],
                                                    g["head_dim"], kb, vb)
        assert total / 2 ** 30 == g["cache_gib"][name]
        assert round(total / 0.010 / 1e9, 1) == g["reread_10ms_gbs"][name]


def test_workspace_and_indices():
    g = GOLD["compact_workspace"]
    assert rf.workspace_bytes(g["pages"], g["num_kv_heads"], g["head_dim"]) == g["payload_bytes"]
    assert g["pages"] * 4 == g["index_bytes"]


def test_payload_ratios():
    g = GOLD["payload_ratio"]
    b = g["bytes_per_pair"]
    assert b["k16v8"] / b["k16v16"] == g["k16v8_payload_fraction"]
    for k in b:
        assert round(b["k16v16"] / b[k], 2) == g["capacity_vs_k16v16"][k]


def test_decode_bytes_counts_tokens_not_pages():
    d = rf.decode_bytes([37, 100], 4, 2, 64, 1, per_page_scales=False)
    assert d["kv"] == 137 * 2 * 64 * 3
    assert d["split"] == d["kv"] + 2 * 4 * 64 * 2 + 4 * (3 + 7) + 4 * 2 + 4
    assert d["total"] == d["split"] + 2 * 4 * 64 * 2
    mixed = rf.decode_bytes([20], 2, 1, 64, [[1, 2]], per_page_scales=True)
    assert mixed["kv"] == 16 * 64 * 3 + 4 * 64 * 4
    assert mixed["split"] == mixed["kv"] + 2 * 64 * 2 + 4 * 2 + 4 + 4 * 1
