"""KV cache integrity check, written out from its definition.

TEST INFRASTRUCTURE ONLY (see the package docstring): only the tests, the smoke
check and the CPU-baseline leg of ``bench.py`` may use this module.

Source: [CF] "Smaller, faster, safer: running Kimi and GLM at scale", section
"Protecting a shared KV cache". Every physical cache page carries a tag that
changes whenever the page is reallocated; the server records which pages, with
which tags, each request expects to read; before decode reads the cache those
mappings are compared, and a request with any mismatch is aborted instead of
being allowed to return data computed from a page that is no longer its own.
The check runs as a separate batch pass, not inside the attention kernel.

Readings where the page gives no layout (this module's own choices):

* a tag is a 32-bit unsigned integer per physical page (``page_tags[p]``);
* a request's expected tags sit beside its block-table entries, one per logical
  page (``expected_tags[b][j]`` for ``block_table[b][j]``);
* a request of sequence length L uses logical pages 0 .. ceil(L / 64) - 1; later
  entries of its row are not looked at;
* the result is one status word per request, a bit set per kind of failure
  (tag mismatch, page id outside the cache, length outside the row), plus a
  copy of the lengths with -1 for every failed request, which a decode call
  turns into out = 0, lse = -inf without reading any of its pages.
"""

import numpy as np

TAG_MISMATCH = 1   # an in-range page whose tag differs from the expected one
PAGE_RANGE = 2     # a used block-table entry outside [0, num_pages)
BAD_LENGTH = 4     # L < 0 or L > max_pages * page_size: no page is looked at


def check_request(page_tags, block_row, expected_row, seq_len, page_size=64):
    """Status word of one request: the OR of its used pages' failures."""
    max_pages = len(block_row)
    if seq_len < 0 or seq_len > max_pages * page_size:
        return BAD_LENGTH
    status = 0
    used = (seq_len + page_size - 1) // page_size
    for j in range(used):
        page = int(block_row[j])
        if page < 0 or page >= len(page_tags):
            status |= PAGE_RANGE
        elif int(page_tags[page]) != int(expected_row[j]):
            status |= TAG_MISMATCH
    return status


def kv_check(page_tags, block_table, expected_tags, seq_lens, page_size=64):
    """Per-request status words and the checked lengths (-1 where a check failed).

    ``page_tags`` [num_pages] and ``expected_tags`` [batch][max_pages] hold
    unsigned 32-bit tags (any integer dtype; compared as uint32),
    ``block_table`` [batch][max_pages] int32, ``seq_lens`` [batch].
    """
    tags = np.asarray(page_tags).astype(np.int64) & 0xFFFFFFFF
    exp = np.asarray(expected_tags).astype(np.int64) & 0xFFFFFFFF
    table = np.asarray(block_table)
    lens = np.asarray(seq_lens)
    status = np.zeros(len(lens), np.int32)
    checked = np.zeros(len(lens), np.int32)
    for b in range(len(lens)):
        status[b] = check_request(tags, table[b], exp[b], int(lens[b]), page_size)
        checked[b] = -1 if status[b] else int(lens[b])
    return status, checked
