"""Algorithmic work of one paged MLA decode step (host-side bookkeeping).

These figures are what the method must move and compute, independent of how a
kernel does it; the benchmark divides them by measured time.

* Bytes: each cached entry is 576 elements ("How to serve trillions of tokens
  for trillion-parameter coding agents", section "Tensor parallel was the best
  parallelism strategy for maximum interactivity"), one byte each in FP8 e4m3
  or two in BF16 ("Smaller, faster, safer: running Kimi and GLM at scale",
  section "Quantizing the KV cache"). A decode step reads every unique page
  once, plus 4 bytes of block table per page, plus queries, and writes outputs.
* Flops: per cached token and query row, 2*576 for the score and 2*512 for the
  weighted value sum.
"""

from __future__ import annotations

import numpy as np

D_ENTRY = 576
D_LATENT = 512

KV_ELEMENT_BYTES = {"e4m3": 1, "bf16": 2}


def kv_bytes_per_token(kv_dtype: str) -> int:
    """Bytes of one cached token's latent entry for one layer."""
    return D_ENTRY * KV_ELEMENT_BYTES[kv_dtype]


def flops_per_token_row() -> int:
    """Flops per (cached token, query row): QK over 576 dims plus PV over 512."""
    return 2 * D_ENTRY + 2 * D_LATENT


def step_bytes(seq_lens, num_queries: int, num_heads: int, kv_dtype: str,
               page_size: int = 64, unique_tokens: int | None = None) -> dict:
    """Algorithmic bytes of one decode step over a batch.

    ``unique_tokens`` counts tokens of shared pages once (prefix sharing);
    by default every request's tokens are counted.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    tokens = int(seq_lens.sum()) if unique_tokens is None else int(unique_tokens)
    pages = int(np.sum(-(-seq_lens // page_size)))
    rows = len(seq_lens) * num_queries * num_heads
    kv = tokens * kv_bytes_per_token(kv_dtype)
    table = 4 * pages
    q = rows * D_ENTRY * 2
    out = rows * D_LATENT * 2 + rows * 4
    return {"kv": kv, "block_table": table, "q": q, "out": out,
            "total": kv + table + q + out}


def step_flops(seq_lens, num_queries: int, num_heads: int) -> int:
    """Flops of one decode step: every visible (token, draft, head) triple."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    visible = 0
    for j in range(num_queries):
        visible += int(np.sum(seq_lens - num_queries + j + 1))
    return visible * num_heads * flops_per_token_row()
