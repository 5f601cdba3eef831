"""Paged MLA decode attention in float64 (oracle; test infrastructure only).

What is computed, and where each step comes from:

* One cache entry per token is 576 elements ([K2.6] "How to serve trillions of
  tokens for trillion-parameter coding agents", section "Tensor parallel was the
  best parallelism strategy for maximum interactivity"). The model has no
  distinct keys and values (same page, section "First, understand the
  workload"): the value of a token is part of its key entry. We read the entry
  as 512 latent elements followed by 64 rotary elements; the key is all 576,
  the value is the first 512.
* MLA keeps a single latent head that every query head attends over
  ([vLLM] "vLLM x AgentX: Optimizing for Real-World Agentic Serving", section
  "Kimi K3").
* The cache is paged and shared: a request names its pages through a block
  table ([CF] "Smaller, faster, safer: running Kimi and GLM at scale", section
  "Protecting a shared KV cache"); entries are FP8 e4m3 and are converted as
  they are read (same page, section "Quantizing the KV cache").
* Speculative verification scores the drafted tokens in parallel without
  changing the target model's distribution ([K2.6], section "Use custom
  speculative decoding ..."). We read this as: ``seq_lens[b]`` counts the
  cached tokens including the ``Q`` drafts just appended, and draft ``j``
  sees positions ``t <= L_b - Q + j``.
* Partial outputs over disjoint pieces of the sequence are combined through
  their log-sum-exp statistics with online softmax ([vLLM], section "Kimi K3").
  ``lse`` is the natural logarithm of the sum of ``exp(score)``, where the
  score already includes ``sm_scale``.

Definition (per request b, draft j, head h):

    K[t]  = dequant(page[block_table[b, t // page_size]][t % page_size])
    n_j   = L_b - Q + j + 1
    s_t   = sm_scale * sum_d q[b, j, h, d] * K[t, d]        for t < n_j
    lse   = log(sum_t exp(s_t))
    out   = sum_t exp(s_t - lse) * K[t, 0:512]

Everything is float64; inputs (bf16 queries, e4m3 / bf16 cache codes) are
widened exactly. The brute-force function restates the same definition with
explicit Python loops and no paging, for tiny inputs only.
"""

from __future__ import annotations

import math

import numpy as np

from . import e4m3

D_LATENT = 512
D_ROPE = 64
D_ENTRY = D_LATENT + D_ROPE

KV_E4M3 = "e4m3"
KV_BF16 = "bf16"


def dequant(codes: np.ndarray, kv_dtype: str, kv_scale: float) -> np.ndarray:
    """Stored cache values -> float64 entries (value times the per-tensor scale)."""
    scale = np.float64(np.float32(kv_scale))
    if kv_dtype == KV_E4M3:
        return e4m3.decode(codes) * scale
    if kv_dtype == KV_BF16:
        return e4m3.bf16_bits_to_f64(codes) * scale
    raise ValueError(f"unknown kv dtype {kv_dtype!r}")


def gather_pages(kv_pages: np.ndarray, block_table_row: np.ndarray, length: int) -> np.ndarray:
    """Logical tokens 0..length-1 of one request, read through its block table.

    ``kv_pages`` is ``[num_pages, page_size, 576]``; logical page ``j`` of the
    request lives in physical page ``block_table_row[j]``.
    """
    page_size = kv_pages.shape[1]
    n_pages = (length + page_size - 1) // page_size
    phys = np.asarray(block_table_row[:n_pages], dtype=np.int64)
    if np.any(phys < 0) or np.any(phys >= kv_pages.shape[0]):
        raise IndexError("block table names a page outside the cache")
    return kv_pages[phys].reshape(n_pages * page_size, kv_pages.shape[2])[:length]


def visible_length(seq_len: int, num_queries: int, j: int) -> int:
    """Positions visible to draft j: the causal reading of parallel verification."""
    return seq_len - num_queries + j + 1


def attend(q_rows: np.ndarray, k: np.ndarray, sm_scale: float):
    """Softmax attention of query rows over one latent head, float64.

    ``q_rows`` is ``[H, 576]``, ``k`` is ``[n, 576]`` (already dequantised).
    Returns ``(out [H, 512], lse [H])``; an empty ``k`` gives zeros and -inf.
    """
    h = q_rows.shape[0]
    n = k.shape[0]
    if n == 0:
        return np.zeros((h, D_LATENT)), np.full(h, -np.inf)
    s = np.float64(np.float32(sm_scale)) * (q_rows @ k.T)    # [H, n]
    m = s.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
    p = np.exp(s - lse[:, None])
    out = p @ k[:, :D_LATENT]
    return out, lse


def decode(q_bits: np.ndarray, kv_pages: np.ndarray, block_table: np.ndarray,
           seq_lens: np.ndarray, sm_scale: float, kv_scale: float,
           kv_dtype: str = KV_E4M3, rows=None):
    """Paged MLA decode for a batch, float64.

    ``q_bits``: bf16 bit patterns ``[B, Q, H, 576]`` (uint16).
    ``kv_pages``: stored cache ``[num_pages, page_size, 576]`` (uint8 codes for
    e4m3, uint16 bf16 bits for bf16). ``block_table``: ``[B, max_pages]``.
    ``seq_lens``: ``[B]``. ``rows``: optional iterable of ``(b, j)`` to compute
    (others are left NaN) so that large batches can be sampled.

    Returns ``(out [B, Q, H, 512], lse [B, Q, H])`` in float64.
    """
    bsz, nq, nh, _ = q_bits.shape
    out = np.full((bsz, nq, nh, D_LATENT), np.nan)
    lse = np.full((bsz, nq, nh), np.nan)
    wanted = None if rows is None else set((int(b), int(j)) for b, j in rows)
    for b in range(bsz):
        if wanted is not None and not any(bb == b for bb, _ in wanted):
            continue
        length = int(seq_lens[b])
        k = dequant(gather_pages(kv_pages, block_table[b], length), kv_dtype, kv_scale)
        for j in range(nq):
            if wanted is not None and (b, j) not in wanted:
                continue
            n = visible_length(length, nq, j)
            q = e4m3.bf16_bits_to_f64(q_bits[b, j])
            out[b, j], lse[b, j] = attend(q, k[:max(n, 0)], sm_scale)
    return out, lse


def merge(part_out: np.ndarray, part_lse: np.ndarray):
    """Merge partial attention results through their log-sum-exp statistics.

    ``part_out``: ``[S, ..., 512]`` normalised partial outputs; ``part_lse``:
    ``[S, ...]``. A part with ``lse = -inf`` (an empty piece) contributes
    nothing; if every part is empty the result is zeros and ``-inf``.
    """
    part_out = np.asarray(part_out, dtype=np.float64)
    part_lse = np.asarray(part_lse, dtype=np.float64)
    m = part_lse.max(axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(part_lse - m_safe)                 # exp(-inf) = 0 for empty parts
    total = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, total, 1.0)), -np.inf)
    coef = np.where(finite, np.exp(part_lse - np.where(finite, lse, 0.0)), 0.0)
    out = (coef[..., None] * part_out).sum(axis=0)
    return out, lse


def dense_bruteforce(q_row, k_rows, sm_scale):
    """The definition with explicit loops, no paging, no numpy algebra.

    ``q_row``: sequence of 576 floats (one head's query); ``k_rows``: list of
    576-float entries. Returns ``(out list[512], lse float)``. Tiny inputs only.
    """
    scores = []
    for k in k_rows:
        acc = 0.0
        for d in range(D_ENTRY):
            acc += float(q_row[d]) * float(k[d])
        scores.append(float(np.float32(sm_scale)) * acc)
    if not scores:
        return [0.0] * D_LATENT, -math.inf
    m = max(scores)
    total = 0.0
    for s in scores:
        total += math.exp(s - m)
    lse = m + math.log(total)
    out = [0.0] * D_LATENT
    for s, k in zip(scores, k_rows):
        p = math.exp(s - lse)
        for d in range(D_LATENT):
            out[d] += p * float(k[d])
    return out, lse
