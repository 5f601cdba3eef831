"""Figures printed on the pages pin the byte accounting (CPU).

The fixture ``tests/golden/kv_entry_sizes.json`` holds the numbers and the page
and section each comes from.
"""

import json
import os

from paged_mla_decode_gb300 import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_entry_sizes.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_entry_elements():
    assert accounting.D_ENTRY == _golden()["entry_elements"]["value"]


def test_bf16_bytes_per_token_over_61_layers():
    g = _golden()["bf16_bytes_per_token_all_layers"]
    assert accounting.kv_bytes_per_token("bf16") * g["layers"] == g["value"]
    # printed as "~72 KB"
    assert abs(g["value"] / 1000 - 72) < 2


def test_fp8_halves_bytes_and_doubles_capacity():
    g = _golden()["fp8_capacity_tokens"]
    ratio = accounting.kv_bytes_per_token("bf16") / accounting.kv_bytes_per_token("e4m3")
    assert ratio == 2
    assert abs(g["bf16_tokens"] * ratio - g["fp8_tokens"]) / g["fp8_tokens"] < 0.01
