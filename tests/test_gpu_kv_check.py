"""mla_kv_check matches the integrity-check oracle bit for bit (GPU).

"Smaller, faster, safer: running Kimi and GLM at scale", section "Protecting a
shared KV cache". The block tables are those of the seeded workloads (full
size: the check reads only tables and tags), the page tags are random 32-bit
values, and a seeded share of the requests is corrupted: a used entry's
expected tag changed, a used entry pointing outside the cache, a length
outside the row, or an entry past the used pages changed (which must pass).
Expected values come from ``oracle.integrity`` only.
"""

import numpy as np
import pytest
import torch

from oracle import integrity as oig
from paged_mla_decode_gb300 import binding
from paged_mla_decode_gb300 import workloads as wl

from .gpu_util import (assert_close, gpu_decode, gpu_fill_cache, oracle_decode,
                       oracle_fill_cache)

pytestmark = pytest.mark.gpu


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a).astype(np.uint32).view(np.int32))


def _case(table, lens, num_pages, seed):
    """Random tags, matching expectations, then seeded corruptions."""
    rng = np.random.default_rng(seed)
    tags = rng.integers(0, 1 << 32, size=num_pages, dtype=np.uint64).astype(np.uint32)
    table = table.copy()
    lens = np.array(lens, dtype=np.int32)
    B, M = table.shape
    expected = rng.integers(0, 1 << 32, size=(B, M), dtype=np.uint64).astype(np.uint32)
    for b in range(B):
        used = min(-(-int(lens[b]) // 64), M)
        expected[b, :used] = tags[table[b, :used]]
    for b in range(B):
        used = min(-(-int(lens[b]) // 64), M)
        kind = rng.integers(0, 6)
        if used == 0:
            continue
        j = int(rng.integers(0, used))
        if kind == 0:
            expected[b, j] ^= np.uint32(1 << int(rng.integers(0, 32)))
        elif kind == 1:
            table[b, j] = num_pages + int(rng.integers(0, 3)) if rng.integers(0, 2) else -1
        elif kind == 2:
            lens[b] = M * 64 + 1
        elif kind == 3 and used < M:
            expected[b, used] ^= np.uint32(1)        # past the used pages: ignored
            table[b, M - 1] = -5
    return tags, table, expected, lens


def _run(tags, table, expected, lens, dev):
    B = table.shape[0]
    status = torch.full((B,), -123, dtype=torch.int32, device=dev)
    checked = torch.full((B,), -123, dtype=torch.int32, device=dev)
    binding.mla_kv_check(_i32(tags).to(dev), torch.from_numpy(table).to(dev),
                         _i32(expected).to(dev), torch.from_numpy(lens).to(dev), status, checked)
    torch.cuda.synchronize()
    return status.cpu().numpy().view(np.uint32), checked.cpu().numpy()


@pytest.mark.parametrize("make", [wl.tiny, wl.long_context, wl.concurrent, wl.prefix_shared,
                                  wl.speculative])
def test_workload_tables_bit_exact(cuda_device, make):
    w = make()
    for seed in range(3):
        tags, table, expected, lens = _case(w.block_table, w.seq_lens, w.num_pages, seed)
        got_s, got_c = _run(tags, table, expected, lens, cuda_device)
        ref_s, ref_c = oig.kv_check(tags, table, expected, lens)
        assert np.array_equal(got_s, ref_s.astype(np.uint32)), (w.name, seed)
        assert np.array_equal(got_c, ref_c), (w.name, seed)
        if seed == 0 and len(lens) > 1:
            assert (ref_s != 0).any() and (ref_s == 0).any()


def test_edges(cuda_device):
    rng = np.random.default_rng(7)
    # lengths 0 / 1 / page boundaries / a request longer than one pass of the
    # kernel's loads (4,096 pages) / out of range below and above
    lens = [0, 1, 63, 64, 65, 4096 * 64, 4096 * 64 + 1, 300_000, -1, 5000 * 64 + 1]
    M = 5000
    num_pages = 6000
    table = rng.integers(0, num_pages, size=(len(lens), M)).astype(np.int32)
    tags, table, expected, _ = _case(table, lens, num_pages, 11)
    got = _run(tags, table, expected, np.array(lens, np.int32), cuda_device)
    ref = oig.kv_check(tags, table, expected, lens)
    assert np.array_equal(got[0], ref[0].astype(np.uint32)) and np.array_equal(got[1], ref[1])
    # one corrupted entry at the very last used page of the long requests
    clean_table = rng.integers(0, num_pages, size=(len(lens), M)).astype(np.int32)
    clean = tags[clean_table]
    for b in (5, 7):
        used = -(-lens[b] // 64)
        e2 = clean.copy()
        e2[b, used - 1] ^= np.uint32(0x80000000)
        got = _run(tags, clean_table, e2, np.array(lens, np.int32), cuda_device)
        ref = oig.kv_check(tags, clean_table, e2, lens)
        assert got[0][b] == oig.TAG_MISMATCH and np.array_equal(got[0], ref[0].astype(np.uint32))
        assert np.array_equal(got[1], ref[1])
    # a cache with no pages: every used entry is out of range, empty requests pass
    got = _run(np.zeros(0, np.uint32), table[:3, :4].copy(), expected[:3, :4].copy(),
               np.array([0, 1, 256], np.int32), cuda_device)
    assert got[0].tolist() == [0, oig.PAGE_RANGE, oig.PAGE_RANGE]
    assert got[1].tolist() == [0, -1, -1]
    # rows with no table columns: only length 0 passes
    got = _run(tags, np.zeros((2, 0), np.int32), np.zeros((2, 0), np.uint32),
               np.array([0, 1], np.int32), cuda_device)
    assert got[0].tolist() == [0, oig.BAD_LENGTH] and got[1].tolist() == [0, -1]


def test_failed_requests_are_aborted_in_decode(cuda_device):
    """Checked lengths fed to mla_decode: failed requests read nothing and give
    out = 0, lse = -inf; the others match the oracle."""
    w = wl.make_lengths_workload("check", 41, [700, 1300, 65, 2000], num_heads=64)
    pages = gpu_fill_cache(w, cuda_device)
    ref_pages = oracle_fill_cache(w)
    rng = np.random.default_rng(3)
    tags = rng.integers(0, 1 << 32, size=w.num_pages, dtype=np.uint64).astype(np.uint32)
    expected = np.zeros(w.block_table.shape, np.uint32)
    lens = w.seq_lens
    for b in range(len(lens)):
        used = -(-int(lens[b]) // 64)
        expected[b, :used] = tags[w.block_table[b, :used]]
    expected[1, 3] += np.uint32(1)            # request 1: a page reallocated since
    tags_d = _i32(tags).to(cuda_device)
    status = torch.zeros(len(lens), dtype=torch.int32, device=cuda_device)
    checked = torch.zeros(len(lens), dtype=torch.int32, device=cuda_device)
    binding.mla_kv_check(tags_d, torch.from_numpy(w.block_table).to(cuda_device),
                         _i32(expected).to(cuda_device), torch.from_numpy(lens).to(cuda_device),
                         status, checked)
    assert status.cpu().tolist() == [0, oig.TAG_MISMATCH, 0, 0]
    # a block-table entry of the failed request now points outside the cache:
    # the decode must not read it (no bad-page report, only the length report)
    table = w.block_table.copy()
    table[1, 3] = w.num_pages + 10 ** 6
    out, lse, ws = gpu_decode(w, pages, cuda_device, seq_lens=checked.cpu().numpy(),
                              block_table=table)
    assert np.all(out[1] == 0) and np.all(lse[1] == -np.inf)
    ok_rows = [(b, 0) for b in (0, 2, 3)]
    ref_out, ref_lse = oracle_decode(w, ref_pages)
    assert_close(out, lse, ref_out, ref_lse, rows=ok_rows, what="checked decode")
    assert binding.read_device_status(ws) == binding.MLA_DEVICE_ERR_BAD_LENGTH
