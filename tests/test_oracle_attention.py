"""Pins for the oracle's paged MLA attention (CPU).

Each test fixes the oracle against something other than its own code:

* brute force: the definition written with explicit loops and no paging;
* scipy's ``softmax`` / ``logsumexp`` (library routines) on a dense problem;
* closed forms: a one-token context returns that token's value and its score;
  a zero query (constant score) returns the mean of the values and ``ln L``;
  duplicating every token leaves ``out`` unchanged and adds ``ln 2`` to lse;
* invariances: permuting physical pages under a matching block table; split
  into pieces plus log-sum-exp merge equals the unsplit result ("vLLM x
  AgentX", section "Kimi K3": partial outputs and LSE merged with online
  softmax); a Q-draft request equals Q single-query requests at the matching
  prefix lengths ("How to serve trillions of tokens ...", section "Use custom
  speculative decoding ...": verification does not change the distribution).
"""

import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import attention as att
from oracle import e4m3
from paged_mla_decode_gb300 import workloads as wl

PS = 64


def _random_paged(rng, lengths, heads, nq=1, scale=None, dtype=att.KV_E4M3, spare=3):
    """A small paged problem with shuffled physical pages (spare pages unused)."""
    kv_scale = float(np.float32(scale if scale is not None else 4.0 / 448.0))
    n_pages = [-(-L // PS) for L in lengths]
    total = sum(n_pages) + spare
    perm = rng.permutation(total)
    table = np.full((len(lengths), max(n_pages)), -1, np.int32)
    cursor = 0
    for b, n in enumerate(n_pages):
        table[b, :n] = perm[cursor:cursor + n]
        cursor += n
    x = wl.f32_to_bf16_bits(rng.standard_normal((total, PS, att.D_ENTRY), dtype=np.float32) * 0.5)
    if dtype == att.KV_E4M3:
        pages = e4m3.encode(e4m3.bf16_bits_to_f64(x), kv_scale)
    else:
        pages = x
        kv_scale = 1.0
    q = wl.f32_to_bf16_bits(rng.standard_normal((len(lengths), nq, heads, att.D_ENTRY),
                                                dtype=np.float32))
    return q, pages, table, np.array(lengths, np.int32), kv_scale


def test_bruteforce_matches_paged():
    rng = np.random.default_rng(10)
    q, pages, table, lens, kv_scale = _random_paged(rng, [130, 64, 1], heads=3)
    out, lse = att.decode(q, pages, table, lens, wl.SM_SCALE, kv_scale)
    for b, L in enumerate(lens):
        # dense entries written out token by token, no block table arithmetic reuse
        k_rows = []
        for t in range(int(L)):
            page = int(table[b][t // PS])
            k_rows.append([e4m3.code_value(c) * kv_scale for c in pages[page, t % PS]])
        for h in range(3):
            qh = e4m3.bf16_bits_to_f64(q[b, 0, h])
            o_ref, l_ref = att.dense_bruteforce(qh, k_rows, wl.SM_SCALE)
            assert abs(lse[b, 0, h] - l_ref) < 1e-12
            assert np.max(np.abs(out[b, 0, h] - np.array(o_ref))) < 1e-12


def test_matches_scipy_softmax_dense():
    rng = np.random.default_rng(11)
    q, pages, table, lens, _ = _random_paged(rng, [300], heads=4, dtype=att.KV_BF16)
    out, lse = att.decode(q, pages, table, lens, wl.SM_SCALE, 1.0, kv_dtype=att.KV_BF16)
    k = e4m3.bf16_bits_to_f64(att.gather_pages(pages, table[0], 300))
    qf = e4m3.bf16_bits_to_f64(q[0, 0])
    s = np.float64(np.float32(wl.SM_SCALE)) * np.einsum("hd,td->ht", qf, k)
    assert np.allclose(lse[0, 0], logsumexp(s, axis=1), rtol=0, atol=1e-12)
    assert np.allclose(out[0, 0], softmax(s, axis=1) @ k[:, :512], rtol=0, atol=1e-12)


def test_one_token_context():
    rng = np.random.default_rng(12)
    q, pages, table, lens, kv_scale = _random_paged(rng, [1], heads=2)
    out, lse = att.decode(q, pages, table, lens, wl.SM_SCALE, kv_scale)
    v = e4m3.decode(pages[table[0, 0], 0]) * kv_scale
    assert np.array_equal(out[0, 0, 0], v[:512]) and np.array_equal(out[0, 0, 1], v[:512])
    qf = e4m3.bf16_bits_to_f64(q[0, 0])
    s0 = float(np.float32(wl.SM_SCALE)) * (qf @ v)
    assert np.allclose(lse[0, 0], s0, rtol=0, atol=1e-12)


def test_zero_query_gives_mean_value():
    rng = np.random.default_rng(13)
    q, pages, table, lens, kv_scale = _random_paged(rng, [777], heads=2)
    q[:] = 0
    out, lse = att.decode(q, pages, table, lens, wl.SM_SCALE, kv_scale)
    k = e4m3.decode(att.gather_pages(pages, table[0], 777)) * kv_scale
    assert np.allclose(out[0, 0, 0], k[:, :512].mean(axis=0), rtol=0, atol=1e-13)
    assert np.allclose(lse[0, 0], math.log(777), rtol=0, atol=1e-13)


def test_duplicating_tokens_adds_ln2():
    rng = np.random.default_rng(14)
    q, pages, table, lens, kv_scale = _random_paged(rng, [128], heads=2)
    out1, lse1 = att.decode(q, pages, table, lens, wl.SM_SCALE, kv_scale)
    k = att.gather_pages(pages, table[0], 128)
    doubled = np.concatenate([k, k], axis=0).reshape(4, PS, att.D_ENTRY)
    out2, lse2 = att.decode(q, doubled, np.array([[0, 1, 2, 3]], np.int32),
                            np.array([256], np.int32), wl.SM_SCALE, kv_scale)
    assert np.allclose(out1, out2, rtol=0, atol=1e-13)
    assert np.allclose(lse2 - lse1, math.log(2.0), rtol=0, atol=1e-12)


def test_page_permutation_invariance():
    rng = np.random.default_rng(15)
    q, pages, table, lens, kv_scale = _random_paged(rng, [200, 65], heads=2)
    out1, lse1 = att.decode(q, pages, table, lens, wl.SM_SCALE, kv_scale)
    perm = rng.permutation(pages.shape[0])        # new physical slot of each page
    moved = np.empty_like(pages)
    moved[perm] = pages
    table2 = np.where(table >= 0, perm[np.clip(table, 0, None)], -1).astype(np.int32)
    out2, lse2 = att.decode(q, moved, table2, lens, wl.SM_SCALE, kv_scale)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


@pytest.mark.parametrize("cuts", [[0, 1, 2, 500], [0, 0, 250, 250, 500], [0, 64, 65, 499, 500],
                                  [0, 500]])
def test_split_and_merge_equals_unsplit(cuts):
    rng = np.random.default_rng(16)
    q, pages, table, lens, kv_scale = _random_paged(rng, [500], heads=3)
    out, lse = att.decode(q, pages, table, lens, wl.SM_SCALE, kv_scale)
    k = att.dequant(att.gather_pages(pages, table[0], 500), att.KV_E4M3, kv_scale)
    qf = e4m3.bf16_bits_to_f64(q[0, 0])
    parts = [att.attend(qf, k[a:b], wl.SM_SCALE) for a, b in zip(cuts[:-1], cuts[1:])]
    m_out, m_lse = att.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.allclose(m_out, out[0, 0], rtol=0, atol=1e-12)
    assert np.allclose(m_lse, lse[0, 0], rtol=0, atol=1e-12)


def test_merge_all_empty():
    o, l = att.merge(np.zeros((3, 2, 512)), np.full((3, 2), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_draft_queries_equal_prefix_decodes():
    rng = np.random.default_rng(17)
    nq = 4
    q, pages, table, lens, kv_scale = _random_paged(rng, [131, 70], heads=2, nq=nq)
    out, lse = att.decode(q, pages, table, lens, wl.SM_SCALE, kv_scale)
    for j in range(nq):
        lens_j = lens - nq + j + 1
        o1, l1 = att.decode(q[:, j:j + 1], pages, table, lens_j, wl.SM_SCALE, kv_scale)
        assert np.array_equal(out[:, j], o1[:, 0]) and np.array_equal(lse[:, j], l1[:, 0])
    # and the drafts really see different prefixes
    assert not np.allclose(out[:, 0], out[:, 3])


def test_kv_scale_enters_linearly():
    rng = np.random.default_rng(18)
    q, pages, table, lens, kv_scale = _random_paged(rng, [90], heads=2)
    q[:] = 0                                   # constant scores: out = mean(V) * scale
    o1, _ = att.decode(q, pages, table, lens, wl.SM_SCALE, 1.0)
    o2, _ = att.decode(q, pages, table, lens, wl.SM_SCALE, 0.25)
    assert np.allclose(o2, 0.25 * o1, rtol=0, atol=1e-14)
