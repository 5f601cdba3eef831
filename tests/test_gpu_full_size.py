"""Full-size workloads, sampled against the oracle (GPU).

Each workload is built at its full size (100k-256k token contexts, 64 heads),
the cache is filled through mla_kv_append and decoded with the default launch
configuration (one CTA per SM, as bench.py runs it). For a few sampled
requests the oracle regenerates the same draws, encodes them, checks the
request's cache bytes bit for bit, and recomputes every head and draft of that
request in float64.
"""

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import e4m3 as oe4m3
from paged_mla_decode_gb300 import workloads as wl

from .gpu_util import assert_close, gpu_decode, gpu_fill_cache

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _check_sampled(w, pages, dev, samples, kv_dtype="e4m3", f16_operands=False):
    kv_scale = w.kv_scale if kv_dtype == "e4m3" else 1.0
    out, lse, ws = gpu_decode(w, pages, dev, kv_scale=kv_scale, f16_operands=f16_operands)
    path = "f16 operands" if f16_operands else kv_dtype
    flat = pages.view(-1, 576)
    for b in samples:
        bits = w.request_latent(b)
        L = int(w.seq_lens[b])
        t = np.arange(L)
        slots = (w.block_table[b, t // 64].astype(np.int64) * 64 + t % 64)
        got = flat[torch.from_numpy(slots).to(dev)].cpu()
        if kv_dtype == "e4m3":
            codes = oe4m3.encode(oe4m3.bf16_bits_to_f64(bits), w.kv_scale)
            assert np.array_equal(got.numpy(), codes), f"cache bytes of request {b}"
            k = oatt.dequant(codes, oatt.KV_E4M3, w.kv_scale)
        else:
            assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), bits)
            k = oatt.dequant(bits, oatt.KV_BF16, 1.0)
        for j in range(w.num_queries):
            n = oatt.visible_length(L, w.num_queries, j)
            q = oe4m3.bf16_bits_to_f64(w.q_bits[b, j])
            ref_out, ref_lse = oatt.attend(q, k[:n], w.sm_scale)
            _, _, lerr = assert_close(out[b, j], lse[b, j], ref_out, ref_lse,
                                      what=f"{w.name} b={b} j={j}")
            # the relative term on its own (the absolute one carries the combined
            # tolerance where a nearly flat softmax makes |out| ~ 1e-3)
            rel = float(np.abs(out[b, j] - ref_out).max() / np.abs(ref_out).max())
            print(f"{w.name} {path} b={b} j={j}: max|ref| {np.abs(ref_out).max():.3g} "
                  f"rel err {rel:.3g} lse err {lerr:.3g}")
            assert rel <= 1e-2, f"{w.name} b={b} j={j}: relative error {rel:.4g}"
    return out, lse, ws


def test_long_context(cuda_device):
    w = wl.long_context()
    pages = gpu_fill_cache(w, cuda_device)
    _check_sampled(w, pages, cuda_device, [0])


@pytest.mark.parametrize("kv_dtype", ["e4m3", "bf16"])
def test_concurrent(cuda_device, kv_dtype):
    w = wl.concurrent()
    pages = gpu_fill_cache(w, cuda_device, kv_dtype)
    _check_sampled(w, pages, cuda_device, [0, 17, 31], kv_dtype)


def test_prefix_shared(cuda_device):
    w = wl.prefix_shared()
    pages = gpu_fill_cache(w, cuda_device)
    _check_sampled(w, pages, cuda_device, [0, 1, 2, 3, 45])


def _speculative_cache(w, dev):
    pages = gpu_fill_cache(w, dev)
    # the step's new tokens go in through the same append path
    fresh = torch.from_numpy(w.fresh_token_latent().view(np.int16)).view(torch.bfloat16)
    fresh = fresh.to(dev)
    from paged_mla_decode_gb300 import binding
    binding.mla_kv_append(fresh[:, :512].contiguous(), fresh[:, 512:].contiguous(),
                          torch.from_numpy(w.fresh_token_slots()).to(dev), pages, w.kv_scale)
    return pages


def test_speculative(cuda_device):
    w = wl.speculative()
    _check_sampled(w, _speculative_cache(w, cuda_device), cuda_device, [0, 13, 31])


@pytest.mark.parametrize("name", ["long", "speculative"])
def test_f16_operands_full_size(cuda_device, name):
    # the ablation (e4m3 pages widened to f16 operands) at full length, 152-way split
    if name == "long":
        w = wl.long_context()
        pages, samples = gpu_fill_cache(w, cuda_device), [0]
    else:
        w = wl.speculative()
        pages, samples = _speculative_cache(w, cuda_device), [0, 31]
    _check_sampled(w, pages, cuda_device, samples, f16_operands=True)
