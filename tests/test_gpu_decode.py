"""mla_decode matches the float64 oracle (GPU).

Tolerance (element by element): max|out - ref| <= 1e-2 * max|ref| + 1e-3 and
max|lse - ref| <= 1e-3. Every case runs through the C ABI. The cache is
written by mla_kv_append; the oracle reads its own e4m3 encoding of the same
draws, and the two caches are compared byte for byte first.
"""

import numpy as np
import pytest
import torch

from paged_mla_decode_gb300 import binding
from paged_mla_decode_gb300 import workloads as wl

from .gpu_util import (assert_close, gpu_decode, gpu_fill_cache, oracle_decode,
                       oracle_fill_cache)

pytestmark = pytest.mark.gpu


def _run(w, dev, kv_dtype="e4m3", num_ctas=0, **kw):
    pages = gpu_fill_cache(w, dev, kv_dtype)
    ref_pages = oracle_fill_cache(w, kv_dtype)
    got_pages = pages.cpu()
    if kv_dtype == "e4m3":
        assert np.array_equal(got_pages.numpy(), ref_pages)
    else:
        assert np.array_equal(got_pages.view(torch.int16).numpy().view(np.uint16), ref_pages)
    if kv_dtype == "bf16":
        kw.setdefault("kv_scale", 1.0)
    out, lse, ws = gpu_decode(w, pages, dev, num_ctas=num_ctas, **kw)
    ref_out, ref_lse = oracle_decode(w, ref_pages, kv_dtype, **{k: v for k, v in kw.items()
                                                                 if k in ("q_bits", "seq_lens")})
    return out, lse, ref_out, ref_lse, ws


def test_tiny_config(cuda_device):
    """batch 2, 16 heads, seq_lens {1024, 777}, pages permuted (seed 0)."""
    w = wl.tiny()
    out, lse, ref_out, ref_lse, ws = _run(w, cuda_device)
    assert_close(out, lse, ref_out, ref_lse, what="tiny")
    assert binding.read_device_status(ws) == 0


@pytest.mark.parametrize("heads", [16, 32, 64])
@pytest.mark.parametrize("num_ctas", [1, 3, 0, 400])
def test_ragged_lengths_and_splits(cuda_device, heads, num_ctas):
    lengths = [1, 2, 63, 64, 65, 129, 777, 1000]
    w = wl.make_lengths_workload("ragged", 20 + heads, lengths, num_heads=heads)
    out, lse, ref_out, ref_lse, _ = _run(w, cuda_device, num_ctas=num_ctas)
    assert_close(out, lse, ref_out, ref_lse, what=f"H={heads} G={num_ctas}")


@pytest.mark.parametrize("nq", [2, 3, 4])
def test_draft_queries(cuda_device, nq):
    w = wl.make_lengths_workload("drafts", 30 + nq, [nq, nq + 1, 64 + nq - 1, 300, 1031],
                                 num_heads=64, num_queries=nq)
    out, lse, ref_out, ref_lse, _ = _run(w, cuda_device, num_ctas=0)
    assert_close(out, lse, ref_out, ref_lse, what=f"Q={nq}")


def test_peaked_scores(cuda_device):
    """q scaled by 8: softmax concentrates, outputs are O(0.1-1), the relative term binds."""
    w = wl.make_lengths_workload("peaked", 40, [5000, 333], num_heads=64)
    q = w.q_bits.view(np.uint16).astype(np.uint32) << 16
    qf = q.view(np.float32) * np.float32(8.0)
    q8 = (qf.view(np.uint32) >> 16).astype(np.uint16)     # exact: power of two
    out, lse, ref_out, ref_lse, _ = _run(w, cuda_device, q_bits=q8)
    assert np.abs(ref_out).max() > 0.05
    err, tol, lerr = assert_close(out, lse, ref_out, ref_lse, what="peaked")
    assert err / np.abs(ref_out).max() < 5e-3


def test_bf16_cache(cuda_device):
    w = wl.make_lengths_workload("bf16", 41, [1500, 64, 7], num_heads=64)
    out, lse, ref_out, ref_lse, _ = _run(w, cuda_device, kv_dtype="bf16")
    assert_close(out, lse, ref_out, ref_lse, what="bf16 cache")


def test_prefix_shared_forks(cuda_device):
    """Forks whose block tables share prefix pages read the same physical pages."""
    from paged_mla_decode_gb300.workloads import _assemble
    rng = np.random.default_rng(42)
    parts = [[(("p", 0), 640), (("s", 0), 37)], [(("p", 0), 640), (("s", 1), 300)],
             [(("p", 1), 128), (("s", 2), 1)], [(("p", 1), 128), (("s", 3), 64)]]
    w = _assemble("forks", 42, rng, 1, 64, parts, "forks")
    assert np.array_equal(w.block_table[0, :10], w.block_table[1, :10])
    out, lse, ref_out, ref_lse, _ = _run(w, cuda_device)
    assert_close(out, lse, ref_out, ref_lse, what="forks")


def test_bad_page_id_marks_row(cuda_device):
    w = wl.make_lengths_workload("badpage", 43, [300, 200], num_heads=16)
    pages = gpu_fill_cache(w, cuda_device)
    ref_pages = oracle_fill_cache(w)
    table = w.block_table.copy()
    table[0, 2] = w.num_pages + 5          # outside the cache
    out, lse, ws = gpu_decode(w, pages, cuda_device, block_table=table)
    ref_out, ref_lse = oracle_decode(w, ref_pages)
    assert binding.read_device_status(ws) & binding.MLA_DEVICE_ERR_BAD_PAGE
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert_close(out[1:], lse[1:], ref_out[1:], ref_lse[1:], what="good row")


def test_bad_length_marks_row(cuda_device):
    w = wl.make_lengths_workload("badlen", 44, [300, 200, 100], num_heads=16, num_queries=2)
    pages = gpu_fill_cache(w, cuda_device)
    ref_pages = oracle_fill_cache(w)
    lens = w.seq_lens.copy()
    lens[0] = 1                            # fewer than the 2 draft tokens
    lens[2] = w.max_pages * 64 + 1         # longer than the block table
    out, lse, ws = gpu_decode(w, pages, cuda_device, seq_lens=lens)
    ref_out, ref_lse = oracle_decode(w, ref_pages)
    assert binding.read_device_status(ws) & binding.MLA_DEVICE_ERR_BAD_LENGTH
    for b in (0, 2):
        assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
    assert_close(out[1:2], lse[1:2], ref_out[1:2], ref_lse[1:2], what="good row")


def test_page_permutation_gives_same_result(cuda_device):
    w = wl.make_lengths_workload("perm", 45, [900, 130], num_heads=64)
    pages = gpu_fill_cache(w, cuda_device)
    out1, lse1, _ = gpu_decode(w, pages, cuda_device)
    perm = np.random.default_rng(1).permutation(w.num_pages)
    moved = torch.empty_like(pages)
    moved[torch.from_numpy(perm).to(cuda_device)] = pages
    table = np.where(w.block_table >= 0, perm[np.clip(w.block_table, 0, None)], -1).astype(np.int32)
    out2, lse2, _ = gpu_decode(w, moved, cuda_device, block_table=table)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_workspace_reuse_and_graph_replay(cuda_device):
    """The device-side planner lets one captured graph serve changing lengths."""
    w = wl.make_lengths_workload("graph", 46, [700, 500, 90], num_heads=64)
    pages = gpu_fill_cache(w, cuda_device)
    ref_pages = oracle_fill_cache(w)
    dev = cuda_device
    from .gpu_util import bf16_tensor
    q = bf16_tensor(w.q_bits, dev)
    table = torch.from_numpy(w.block_table).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    out = torch.empty((3, 1, 64, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((3, 1, 64), dtype=torch.float32, device=dev)
    ws = torch.zeros(binding.mla_decode_workspace_size(3, 1, 64), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.mla_decode(q, pages, table, lens, w.sm_scale, w.kv_scale, out, lse, ws)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.mla_decode(q, pages, table, lens, w.sm_scale, w.kv_scale, out, lse, ws)
    # each request keeps its pages (11, 8 and 2 of them): lengths stay within them
    for new_lens in ([700, 500, 90], [64, 1, 128], [699, 129, 2]):
        lens.copy_(torch.tensor(new_lens, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        lens_np = np.array(new_lens, np.int32)
        ref_out, ref_lse = oracle_decode(w, ref_pages, seq_lens=lens_np)
        assert_close(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse,
                     what=f"graph replay {new_lens}")


def test_invalid_arguments_raise(cuda_device):
    w = wl.make_lengths_workload("inv", 47, [100], num_heads=64)
    pages = gpu_fill_cache(w, cuda_device)
    with pytest.raises(binding.MlaError):
        gpu_decode(w, pages, cuda_device, workspace=torch.zeros(16, dtype=torch.uint8,
                                                                device=cuda_device))
