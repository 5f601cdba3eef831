"""Pins of the KV-cache integrity check oracle (CPU).

"Smaller, faster, safer: running Kimi and GLM at scale", section "Protecting a
shared KV cache": each physical page carries a tag that changes when the page is
reallocated, the server keeps the (page, tag) pairs each request expects, and a
request whose pairs no longer match is aborted before decode reads the cache.

The expected results below do not come from the oracle's comparison code: they
follow from how each scenario is built (a small page allocator that bumps a
page's tag on every allocation, then frees and hands pages to other requests),
from the length rule written out by hand (a request of L tokens uses
ceil(L / 64) pages), or from brute force over every single-entry corruption.
The last test plants plausible slips in the oracle and checks that a pin fails
for each.
"""

import numpy as np
import pytest

from oracle import integrity as ig

PS = 64


class Allocator:
    """A page pool whose tag of a page changes every time the page is handed out."""

    def __init__(self, num_pages, seed):
        self.rng = np.random.default_rng(seed)
        self.free = list(self.rng.permutation(num_pages))
        self.tags = np.zeros(num_pages, np.uint32)
        self.counter = 0

    def alloc(self):
        page = int(self.free.pop(0))
        self.counter += 1
        self.tags[page] = np.uint32(0x9E3779B1 * self.counter & 0xFFFFFFFF)
        return page

    def release(self, page):
        self.free.append(page)


def _build(alloc, lens, max_pages):
    """Block table and expected tags of requests of the given lengths."""
    table = np.full((len(lens), max_pages), -7, np.int32)     # unused entries: junk
    expected = np.full((len(lens), max_pages), 12345, np.uint32)
    for b, n in enumerate(lens):
        for j in range(-(-n // PS)):
            page = alloc.alloc()
            table[b, j] = page
            expected[b, j] = alloc.tags[page]
    return table, expected


def test_fresh_mappings_all_pass():
    alloc = Allocator(200, seed=1)
    lens = [1, 64, 65, 777, 1024, 0]
    table, expected = _build(alloc, lens, 20)
    status, checked = ig.kv_check(alloc.tags, table, expected, lens)
    assert status.tolist() == [0] * len(lens)
    assert checked.tolist() == lens


def test_reallocated_page_aborts_only_its_old_owner():
    alloc = Allocator(64, seed=2)
    lens = [300, 200, 129]
    table, expected = _build(alloc, lens, 8)
    # request 1's third page is freed (the request is preempted, say) and handed
    # to a new request; request 1's stale mapping must now be rejected
    victim = int(table[1, 2])
    alloc.release(victim)
    while alloc.free[0] != victim:
        alloc.free.append(alloc.free.pop(0))
    assert alloc.alloc() == victim
    status, checked = ig.kv_check(alloc.tags, table, expected, lens)
    assert status.tolist() == [0, ig.TAG_MISMATCH, 0]
    assert checked.tolist() == [300, -1, 129]


def test_shared_prefix_pages_pass_for_every_fork():
    # forks of one session point at the same physical prefix pages with the
    # same tags; a private suffix page reallocated under one fork fails that fork
    alloc = Allocator(100, seed=3)
    prefix = [alloc.alloc() for _ in range(5)]
    table = np.zeros((3, 8), np.int32)
    expected = np.zeros((3, 8), np.uint32)
    for b in range(3):
        table[b, :5] = prefix
        expected[b, :5] = alloc.tags[prefix]
        page = alloc.alloc()
        table[b, 5] = page
        expected[b, 5] = alloc.tags[page]
    lens = [5 * PS + 10, 5 * PS + 1, 6 * PS]
    status, _ = ig.kv_check(alloc.tags, table, expected, lens)
    assert status.tolist() == [0, 0, 0]
    alloc.tags[table[2, 5]] += np.uint32(1)          # fork 2's own page reused
    status, _ = ig.kv_check(alloc.tags, table, expected, lens)
    assert status.tolist() == [0, 0, ig.TAG_MISMATCH]
    alloc.tags[prefix[3]] += np.uint32(1)            # the shared prefix reused: all fail
    status, checked = ig.kv_check(alloc.tags, table, expected, lens)
    assert status.tolist() == [ig.TAG_MISMATCH] * 3
    assert checked.tolist() == [-1, -1, -1]


@pytest.mark.parametrize("length,used", [(0, 0), (1, 1), (63, 1), (64, 1), (65, 2),
                                         (128, 2), (129, 3), (8 * PS, 8)])
def test_only_used_pages_are_looked_at(length, used):
    # every entry corrupted one at a time: a failure exactly for j < ceil(L / 64)
    num_pages = 16
    tags = np.arange(num_pages, dtype=np.uint32) * 3 + 1
    table = np.arange(8, dtype=np.int32)[None, :].copy()
    expected = tags[table].astype(np.uint32)
    for j in range(8):
        bad_tag = expected.copy()
        bad_tag[0, j] ^= 0x80000000
        bad_page = table.copy()
        bad_page[0, j] = num_pages + j
        st_tag, _ = ig.kv_check(tags, table, bad_tag, [length])
        st_page, _ = ig.kv_check(tags, bad_page, expected, [length])
        assert st_tag[0] == (ig.TAG_MISMATCH if j < used else 0), (length, j)
        assert st_page[0] == (ig.PAGE_RANGE if j < used else 0), (length, j)


def test_length_outside_the_row():
    tags = np.ones(10, np.uint32)
    table = np.zeros((3, 4), np.int32)
    expected = np.ones((3, 4), np.uint32)
    status, checked = ig.kv_check(tags, table, expected, [4 * PS, 4 * PS + 1, -1])
    assert status.tolist() == [0, ig.BAD_LENGTH, ig.BAD_LENGTH]
    assert checked.tolist() == [4 * PS, -1, -1]


def test_page_id_range_bounds():
    tags = np.zeros(5, np.uint32)
    expected = np.zeros((4, 1), np.uint32)
    table = np.array([[0], [4], [5], [-1]], np.int32)
    status, _ = ig.kv_check(tags, table, expected, [1, 1, 1, 1])
    assert status.tolist() == [0, 0, ig.PAGE_RANGE, ig.PAGE_RANGE]


def test_both_failures_in_one_request_or_together():
    tags = np.array([7, 8, 9], np.uint32)
    table = np.array([[0, 1, 5]], np.int32)
    expected = np.array([[7, 0, 9]], np.uint32)
    status, checked = ig.kv_check(tags, table, expected, [3 * PS])
    assert status[0] == ig.TAG_MISMATCH | ig.PAGE_RANGE
    assert checked[0] == -1


def test_tags_compare_as_unsigned_32_bit():
    # the same bit patterns given as int32 (negative) or uint32 compare equal
    tags_u = np.array([0xFFFFFFFF, 0x80000000, 5], np.uint32)
    tags_i = tags_u.view(np.int32)
    table = np.array([[0, 1, 2]], np.int32)
    exp_u = tags_u[None, :].copy()
    s1, _ = ig.kv_check(tags_u, table, exp_u.view(np.int32), [3 * PS])
    s2, _ = ig.kv_check(tags_i, table, exp_u, [3 * PS])
    assert s1[0] == 0 and s2[0] == 0
    s3, _ = ig.kv_check(tags_u, table, (exp_u ^ np.uint32(1 << 31)), [3 * PS])
    assert s3[0] == ig.TAG_MISMATCH


PINS = [
    test_fresh_mappings_all_pass,
    test_reallocated_page_aborts_only_its_old_owner,
    test_shared_prefix_pages_pass_for_every_fork,
    lambda: [test_only_used_pages_are_looked_at(L, u) for L, u in
             [(0, 0), (1, 1), (64, 1), (65, 2), (8 * PS, 8)]],
    test_length_outside_the_row,
    test_page_id_range_bounds,
    test_both_failures_in_one_request_or_together,
    test_tags_compare_as_unsigned_32_bit,
]


def _check_floor_pages(page_tags, block_row, expected_row, seq_len, page_size=64):
    if seq_len < 0 or seq_len > len(block_row) * page_size:
        return ig.BAD_LENGTH
    st = 0
    for j in range(seq_len // page_size):           # slip: a partial last page skipped
        page = int(block_row[j])
        if page < 0 or page >= len(page_tags):
            st |= ig.PAGE_RANGE
        elif int(page_tags[page]) != int(expected_row[j]):
            st |= ig.TAG_MISMATCH
    return st


def _check_logical_index(page_tags, block_row, expected_row, seq_len, page_size=64):
    if seq_len < 0 or seq_len > len(block_row) * page_size:
        return ig.BAD_LENGTH
    st = 0
    for j in range(-(-seq_len // page_size)):
        page = int(block_row[j])
        if page < 0 or page >= len(page_tags):
            st |= ig.PAGE_RANGE
        elif int(page_tags[j % len(page_tags)]) != int(expected_row[j]):   # slip: tag of j
            st |= ig.TAG_MISMATCH
    return st


def _check_upper_bound_inclusive(page_tags, block_row, expected_row, seq_len, page_size=64):
    if seq_len < 0 or seq_len > len(block_row) * page_size:
        return ig.BAD_LENGTH
    st = 0
    for j in range(-(-seq_len // page_size)):
        page = int(block_row[j])
        if page < 0 or page > len(page_tags):          # slip: page == num_pages accepted
            st |= ig.PAGE_RANGE
        elif int(page_tags[page % len(page_tags)]) != int(expected_row[j]):
            st |= ig.TAG_MISMATCH
    return st


def _check_signed_tags(page_tags, block_row, expected_row, seq_len, page_size=64):
    if seq_len < 0 or seq_len > len(block_row) * page_size:
        return ig.BAD_LENGTH
    st = 0
    for j in range(-(-seq_len // page_size)):
        page = int(block_row[j])
        if page < 0 or page >= len(page_tags):
            st |= ig.PAGE_RANGE
        elif int(page_tags[page]) & 0x7FFFFFFF != int(expected_row[j]) & 0x7FFFFFFF:  # slip
            st |= ig.TAG_MISMATCH
    return st


@pytest.mark.parametrize("slip", [_check_floor_pages, _check_logical_index,
                                  _check_upper_bound_inclusive, _check_signed_tags])
def test_planted_slips_are_caught(monkeypatch, slip):
    monkeypatch.setattr(ig, "check_request", slip)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, slip.__name__
