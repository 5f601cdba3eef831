"""Seeded synthetic workloads for paged MLA decode.

This module only draws inputs: request lengths, a shuffled page free list,
block tables (with shared prefix pages for forked sessions), bfloat16 latent
entries for every cached token, and bfloat16 queries. It holds none of the
attention arithmetic and none of the FP8 rounding; both the CUDA path and the
float64 oracle consume what it produces.

The workload shapes follow the traffic described on the pages: ~100k-142k
token contexts with short outputs, 64 query heads over one 576-element latent
entry per token, paged cache with page size 64, and subagent sessions forked
from a shared context ("vLLM x AgentX: Optimizing for Real-World Agentic
Serving", section "Characterizing agentic workloads: a second look": median
input 142K tokens, prefix hit rate above 96%, subagents forking from the parent
context). The synthetic draws stand in for those traces; no trace data is used.

Recipe (all draws from numpy PCG64, platform independent):

* ``rng = default_rng(seed)`` draws, in order: request lengths, the page
  permutation (the shuffled free list), then the queries ``q ~ N(0,1)`` rounded
  to bfloat16.
* Cached entries are drawn per *segment* (a private sequence, a shared prefix,
  or a private suffix) from ``default_rng([seed, 1, segment_id])`` as
  ``N(0,1) * 0.5`` in float32 rounded to bfloat16, so any request's tokens can
  be regenerated without drawing the whole batch.
* ``kv_scale`` is one float32 per cache: ``4 / 448`` (an 8-sigma range maps to
  the largest e4m3 magnitude); ``sm_scale = 1/sqrt(192)`` in float32.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PAGE_SIZE = 64
D_ENTRY = 576
D_LATENT = 512
KV_SIGMA = 0.5
KV_SCALE = float(np.float32(4.0 / 448.0))
SM_SCALE = float(np.float32(1.0 / math.sqrt(192.0)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


@dataclass
class Segment:
    """A run of cached tokens that starts on a page boundary."""

    seg_id: int
    length: int
    pages: np.ndarray  # physical page ids, ceil(length / page_size) of them


@dataclass
class Workload:
    name: str
    seed: int
    batch: int
    num_queries: int
    num_heads: int
    page_size: int
    seq_lens: np.ndarray            # int32 [B]
    block_table: np.ndarray         # int32 [B, max_pages]
    num_pages: int
    segments: list                  # list[Segment]
    request_segments: list          # per request: list of segment indices, in order
    q_bits: np.ndarray              # uint16 [B, Q, H, 576]
    kv_scale: float = KV_SCALE
    sm_scale: float = SM_SCALE
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.sum())

    @property
    def unique_tokens(self) -> int:
        return int(sum(s.length for s in self.segments))

    def segment_latent(self, seg_index: int) -> np.ndarray:
        """bf16 bits ``[length, 576]`` of one segment's cached entries."""
        seg = self.segments[seg_index]
        rng = np.random.default_rng([self.seed, 1, seg.seg_id])
        x = rng.standard_normal((seg.length, D_ENTRY), dtype=np.float32)
        x *= np.float32(KV_SIGMA)
        return f32_to_bf16_bits(x)

    def segment_slots(self, seg_index: int, table_map=None) -> np.ndarray:
        """Cache slot (physical_page * page_size + offset) of each token of a segment.

        ``table_map`` optionally renames physical pages (used for cache copies).
        """
        seg = self.segments[seg_index]
        pages = seg.pages if table_map is None else table_map[seg.pages]
        t = np.arange(seg.length, dtype=np.int64)
        return (pages[t // self.page_size].astype(np.int64) * self.page_size
                + t % self.page_size).astype(np.int32)

    def request_latent(self, b: int) -> np.ndarray:
        """bf16 bits ``[L_b, 576]`` of request b's logical tokens, in order."""
        parts = [self.segment_latent(i) for i in self.request_segments[b]]
        out = np.concatenate(parts, axis=0)
        assert out.shape[0] == int(self.seq_lens[b])
        return out

    def fresh_token_slots(self) -> np.ndarray:
        """Slots of the last Q tokens of every request (the step's new tokens), [B*Q]."""
        slots = []
        for b in range(self.batch):
            length = int(self.seq_lens[b])
            for t in range(length - self.num_queries, length):
                page = self.block_table[b, t // self.page_size]
                slots.append(int(page) * self.page_size + t % self.page_size)
        return np.asarray(slots, dtype=np.int32)

    def fresh_token_latent(self) -> np.ndarray:
        """bf16 bits ``[B*Q, 576]`` of the last Q tokens of every request."""
        rows = []
        for b in range(self.batch):
            length = int(self.seq_lens[b])
            segs = self.request_segments[b]
            last = self.segments[segs[-1]]
            # the last Q tokens always sit in the request's last segment
            assert last.length >= self.num_queries
            lat = self.segment_latent(segs[-1])
            rows.append(lat[last.length - self.num_queries:])
            del length
        return np.concatenate(rows, axis=0)

    def cache_copies(self, copies: int, seed: int = 12345):
        """Page renamings for ``copies`` independent copies of the cache.

        Returns ``(maps, tables)``: ``maps[r]`` sends a page id of this workload
        to a page id of a pool of ``copies * num_pages`` pages, ``tables[r]`` is
        the block table of copy r. Each copy uses its own shuffled pages.
        """
        rng = np.random.default_rng([seed, copies])
        maps, tables = [], []
        for r in range(copies):
            m = (rng.permutation(self.num_pages) + r * self.num_pages).astype(np.int64)
            maps.append(m)
            t = self.block_table.astype(np.int64)
            mapped = np.where(t >= 0, m[np.clip(t, 0, None)], -1)
            tables.append(mapped.astype(np.int32))
        return maps, tables


def _assemble(name, seed, rng, num_queries, num_heads, request_parts, description,
              page_size=PAGE_SIZE):
    """Build segments, a shuffled page assignment and block tables.

    ``request_parts[b]`` lists ``(segment_key, length)`` in order; equal keys
    denote one shared segment (same pages, same tokens).
    """
    seg_index = {}
    segments = []
    for parts in request_parts:
        for key, length in parts:
            if key not in seg_index:
                seg_index[key] = len(segments)
                segments.append(Segment(seg_id=len(segments), length=int(length),
                                        pages=np.empty(0, np.int64)))
    n_pages = [-(-s.length // page_size) for s in segments]
    num_pages = int(sum(n_pages))
    perm = rng.permutation(num_pages).astype(np.int64)   # the shuffled free list
    cursor = 0
    for s, n in zip(segments, n_pages):
        s.pages = perm[cursor:cursor + n]
        cursor += n
    batch = len(request_parts)
    req_segs = [[seg_index[k] for k, _ in parts] for parts in request_parts]
    seq_lens = np.array([sum(l for _, l in parts) for parts in request_parts], np.int32)
    max_pages = int(max(-(-int(L) // page_size) for L in seq_lens))
    table = np.full((batch, max_pages), -1, np.int32)
    for b, segs in enumerate(req_segs):
        col = 0
        for i, si in enumerate(segs):
            s = segments[si]
            if i + 1 < len(segs) and s.length % page_size:
                raise ValueError("only a request's last segment may end mid-page")
            table[b, col:col + len(s.pages)] = s.pages
            col += len(s.pages)
    q = rng.standard_normal((batch, num_queries, num_heads, D_ENTRY), dtype=np.float32)
    return Workload(name=name, seed=seed, batch=batch, num_queries=num_queries,
                    num_heads=num_heads, page_size=page_size, seq_lens=seq_lens,
                    block_table=table, num_pages=num_pages, segments=segments,
                    request_segments=req_segs, q_bits=f32_to_bf16_bits(q),
                    description=description)


def make_lengths_workload(name, seed, lengths, num_heads=64, num_queries=1, description=""):
    """Independent requests with the given lengths (no sharing)."""
    rng = np.random.default_rng(seed)
    parts = [[(("req", b), int(L))] for b, L in enumerate(lengths)]
    return _assemble(name, seed, rng, num_queries, num_heads, parts, description)


def tiny(seed: int = 0) -> Workload:
    """batch 2, 16 heads, seq_lens {1024, 777}, pages permuted."""
    return make_lengths_workload("tiny", seed, [1024, 777], num_heads=16,
                                 description="B=2 H=16 Q=1 L={1024,777}")


def long_context(seed: int = 1, seq_len: int = 100_000) -> Workload:
    """batch 1, 64 heads, one query token, 100,000 cached tokens."""
    return make_lengths_workload("long", seed, [seq_len], num_heads=64,
                                 description=f"B=1 H=64 Q=1 L={seq_len}")


def concurrent(seed: int = 2, batch: int = 32, lo: int = 60_000, hi: int = 140_000) -> Workload:
    """batch 32, 64 heads, lengths uniform in [60k, 140k]."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(lo, hi, size=batch, endpoint=True)
    parts = [[(("req", b), int(L))] for b, L in enumerate(lengths)]
    return _assemble("concurrent", seed, rng, 1, 64, parts,
                     f"B={batch} H=64 Q=1 L~U[{lo},{hi}]")


def prefix_shared(seed: int = 3, groups: int = 16, forks: int = 4, prefix: int = 120_000,
                  suffix_median: float = 2000.0, suffix_sigma: float = 1.0,
                  suffix_max: int = 20_000, num_queries: int = 1,
                  num_heads: int = 64) -> Workload:
    """16 groups x 4 forks; each group shares one physical 120k-token prefix.

    ``extra`` records the grouping: requests [g*forks, (g+1)*forks) share the
    ``prefix_pages`` first pages.
    """
    if prefix % PAGE_SIZE:
        raise ValueError("shared prefix must fill whole pages")
    rng = np.random.default_rng(seed)
    suffix = rng.lognormal(math.log(suffix_median), suffix_sigma, size=groups * forks)
    suffix = np.clip(np.rint(suffix), num_queries, suffix_max).astype(np.int64)
    parts = []
    for g in range(groups):
        for f in range(forks):
            b = g * forks + f
            parts.append([(("prefix", g), prefix), (("suffix", b), int(suffix[b]))])
    w = _assemble("prefix_shared", seed, rng, num_queries, num_heads, parts,
                  f"B={groups * forks} ({groups}x{forks} forks) H={num_heads} Q={num_queries} "
                  f"prefix={prefix} suffix~logN(median {suffix_median:g}, sigma {suffix_sigma})")
    w.extra = {"forks": forks, "prefix_pages": np.full(groups, prefix // PAGE_SIZE, np.int32)}
    return w


def speculative(seed: int = 4, batch: int = 32, num_queries: int = 4,
                median: float = 142_000.0, sigma: float = 0.5,
                lo: int = 32_000, hi: int = 256_000) -> Workload:
    """batch 32, 4 draft queries, lengths lognormal(median 142k) clipped to [32k, 256k]."""
    rng = np.random.default_rng(seed)
    lengths = rng.lognormal(math.log(median), sigma, size=batch)
    lengths = np.clip(np.rint(lengths), lo, hi).astype(np.int64)
    parts = [[(("req", b), int(L))] for b, L in enumerate(lengths)]
    return _assemble("speculative", seed, rng, num_queries, 64, parts,
                     f"B={batch} H=64 Q={num_queries} L~logN(median {median:g}, sigma {sigma}) "
                     f"clipped [{lo},{hi}]")


CONFIGS = {
    "tiny": tiny,
    "long": long_context,
    "concurrent": concurrent,
    "prefix_shared": prefix_shared,
    "speculative": speculative,
}
