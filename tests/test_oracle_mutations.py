"""Planted mistakes in the oracle must be caught by its pins (CPU).

Each case patches one plausible slip into the oracle (a dropped term, a wrong
sign, an off-by-one, a transposed index, a wrong exponent bias) and runs the
pin tests of ``test_oracle_attention`` / ``test_oracle_e4m3`` against it. At
least one pin has to fail for every mutation; otherwise the pins would not
be strong enough to trust the oracle.
"""

import numpy as np
import pytest

from oracle import attention as att
from oracle import e4m3
from tests import test_oracle_attention as pins
from tests import test_oracle_e4m3 as e4m3_pins

ATTN_PINS = [
    pins.test_bruteforce_matches_paged,
    pins.test_matches_scipy_softmax_dense,
    pins.test_one_token_context,
    pins.test_zero_query_gives_mean_value,
    pins.test_duplicating_tokens_adds_ln2,
    pins.test_page_permutation_invariance,
    lambda: pins.test_split_and_merge_equals_unsplit([0, 1, 2, 500]),
    pins.test_draft_queries_equal_prefix_decodes,
]


def _attend_no_rope(q_rows, k, sm_scale):
    k2 = k.copy()
    k2[:, 512:] = 0
    o, l = _ORIG_ATTEND(q_rows, k2, sm_scale)
    return o, l


def _attend_neg_sign(q_rows, k, sm_scale):
    return _ORIG_ATTEND(q_rows, k, -sm_scale)


def _attend_lse_without_max(q_rows, k, sm_scale):
    o, l = _ORIG_ATTEND(q_rows, k, sm_scale)
    if k.shape[0] == 0:
        return o, l
    s = np.float64(np.float32(sm_scale)) * (q_rows @ k.T)
    return o, l - s.max(axis=1)


def _attend_value_from_rope_side(q_rows, k, sm_scale):
    o, l = _ORIG_ATTEND(q_rows, k, sm_scale)
    if k.shape[0] == 0:
        return o, l
    s = np.float64(np.float32(sm_scale)) * (q_rows @ k.T)
    p = np.exp(s - l[:, None])
    return p @ k[:, 64:], l                     # value taken from the wrong 512 dims


def _gather_transposed(kv_pages, block_table_row, length):
    ps = kv_pages.shape[1]
    n_pages = (length + ps - 1) // ps
    phys = np.asarray(block_table_row[:n_pages], dtype=np.int64)
    return kv_pages[phys].transpose(1, 0, 2).reshape(-1, kv_pages.shape[2])[:length]


def _visible_off_by_one(seq_len, num_queries, j):
    return seq_len - num_queries + j


_ORIG_ATTEND = att.attend

MUTATIONS = {
    "scores drop the rope dims": ("attend", _attend_no_rope),
    "scores with flipped sign": ("attend", _attend_neg_sign),
    "lse missing the max shift": ("attend", _attend_lse_without_max),
    "value from the wrong dims": ("attend", _attend_value_from_rope_side),
    "token/page index transposed": ("gather_pages", _gather_transposed),
    "draft visibility off by one": ("visible_length", _visible_off_by_one),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_attention_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(att, attr, fn)
    failures = 0
    for pin in ATTN_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures >= 1, f"mutation {name!r} passed every pin"


def test_e4m3_bias_mutation_is_caught(monkeypatch):
    bad = np.array([e4m3.code_value(c) * 0.5 if c not in (0, 0x80) else 0.0
                    for c in range(256)])            # exponent bias 8 instead of 7
    monkeypatch.setattr(e4m3, "DECODE_TABLE", bad)
    with pytest.raises(AssertionError):
        e4m3_pins.test_decode_matches_torch_float8()


def test_e4m3_ties_away_mutation_is_caught(monkeypatch):
    def rint_away(x):
        return np.where(x >= 0, np.floor(x + 0.5), np.ceil(x - 0.5))
    monkeypatch.setattr(e4m3.np, "rint", rint_away)
    try:
        with pytest.raises(AssertionError):
            e4m3_pins.test_encode_exact_midpoints_go_to_even()
    finally:
        monkeypatch.undo()
