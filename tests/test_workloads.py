"""The seeded workload generator: determinism, page tables, sharing (CPU)."""

import numpy as np

from paged_mla_decode_gb300 import workloads as wl


def _check_tables(w):
    ps = w.page_size
    used = set()
    for b in range(w.batch):
        n = -(-int(w.seq_lens[b]) // ps)
        row = w.block_table[b]
        assert np.all(row[:n] >= 0) and np.all(row[:n] < w.num_pages)
        assert np.all(row[n:] == -1)
        used.update(int(p) for p in row[:n])
    assert used == set(range(w.num_pages))          # every allocated page is referenced


def test_tiny_config():
    w = wl.tiny()
    assert w.batch == 2 and w.num_heads == 16 and w.num_queries == 1
    assert list(w.seq_lens) == [1024, 777]
    assert w.num_pages == 16 + 13
    _check_tables(w)
    # pages come from a shuffled free list, not in order
    assert not np.array_equal(w.block_table[0, :16], np.arange(16))
    assert w.q_bits.shape == (2, 1, 16, 576)


def test_determinism_and_segment_regeneration():
    a, b = wl.tiny(), wl.tiny()
    assert np.array_equal(a.block_table, b.block_table)
    assert np.array_equal(a.q_bits, b.q_bits)
    assert np.array_equal(a.segment_latent(1), b.segment_latent(1))
    assert not np.array_equal(a.segment_latent(0)[:777], a.segment_latent(1))


def test_bf16_rounding_of_draws():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.0, 3.0e-39], np.float32)
    bits = wl.f32_to_bf16_bits(x)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert back[0] == 1.0 and back[1] == 1.0          # tie 1+2^-8 goes to even
    assert back[2] == np.float32(1.0078125)            # above the tie rounds up
    assert back[3] == -2.0


def test_prefix_shared_structure():
    w = wl.prefix_shared()
    assert w.batch == 64
    _check_tables(w)
    pre = 120_000 // 64
    for g in range(16):
        rows = w.block_table[4 * g:4 * g + 4, :pre]
        assert np.all(rows == rows[0])                  # forks share the prefix pages
    assert np.all(w.seq_lens >= 120_001) and np.all(w.seq_lens <= 140_000)
    assert w.unique_tokens < w.total_tokens


def test_large_config_shapes():
    c = wl.concurrent()
    assert c.batch == 32 and c.seq_lens.min() >= 60_000 and c.seq_lens.max() <= 140_000
    _check_tables(c)
    s = wl.speculative()
    assert s.batch == 32 and s.num_queries == 4
    assert s.seq_lens.min() >= 32_000 and s.seq_lens.max() <= 256_000
    l = wl.long_context()
    assert l.seq_lens.tolist() == [100_000] and l.num_pages == 1563


def test_fresh_tokens_and_copies():
    w = wl.make_lengths_workload("t", 5, [100, 65], num_heads=4, num_queries=2)
    slots = w.fresh_token_slots()
    lat = w.fresh_token_latent()
    assert slots.shape == (4,) and lat.shape == (4, 576)
    full0 = w.request_latent(0)
    assert np.array_equal(lat[:2], full0[98:100])
    maps, tables = w.cache_copies(3)
    assert len(tables) == 3
    allp = np.concatenate([t[t >= 0] for t in tables])
    assert len(set(allp.tolist())) == 3 * w.num_pages
