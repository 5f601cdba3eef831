"""mla_decode_grouped matches the float64 oracle (GPU).

The grouped decode computes exactly what mla_decode computes; only the cut of
the work differs (the forks of a group work each shared page at the same time).
So the oracle is the plain paged decode over each request's full block-table
row (oracle/attention.py); the tolerance is the stated one. Cases: several
group shapes and CTA counts (including counts that are not a multiple of the
group size, and fewer CTAs than forks), draft queries, no shared prefix, a
request shorter than its group's prefix, and the full prefix-shared workload.
"""

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import e4m3 as oe4m3
from paged_mla_decode_gb300 import binding
from paged_mla_decode_gb300 import workloads as wl

from .gpu_util import assert_close, bf16_tensor, gpu_fill_cache, oracle_decode, oracle_fill_cache

pytestmark = pytest.mark.gpu


def _grouped(w, pages, dev, prefix_pages, forks, num_ctas=0, seq_lens=None, block_table=None):
    q = bf16_tensor(w.q_bits, dev)
    table = torch.from_numpy(w.block_table if block_table is None else block_table).to(dev)
    lens = torch.from_numpy(w.seq_lens if seq_lens is None else seq_lens).to(dev)
    B, Q, H = q.shape[:3]
    out = torch.full((B, Q, H, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, Q, H), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.zeros(binding.mla_decode_grouped_workspace_size(B, Q, H, num_ctas),
                     dtype=torch.uint8, device=dev)
    pp = torch.from_numpy(np.asarray(prefix_pages, np.int32)).to(dev)
    binding.mla_decode_grouped(q, pages, table, lens, forks, pp, w.sm_scale, w.kv_scale, out, lse,
                               ws, num_ctas=num_ctas)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), binding.read_device_status(ws)


@pytest.mark.parametrize("groups,forks,prefix,num_ctas", [
    (3, 4, 640, 0), (3, 4, 640, 12), (3, 4, 640, 13), (2, 3, 1280, 7), (4, 2, 64, 0),
    (1, 8, 2048, 0), (2, 4, 640, 4), (5, 1, 320, 0), (3, 4, 1280, 400)])
def test_groups_match_oracle(cuda_device, groups, forks, prefix, num_ctas):
    w = wl.prefix_shared(seed=50 + groups + forks, groups=groups, forks=forks, prefix=prefix,
                         suffix_median=150.0, suffix_max=700)
    pages = gpu_fill_cache(w, cuda_device)
    ref_pages = oracle_fill_cache(w)
    assert np.array_equal(pages.cpu().numpy(), ref_pages)
    out, lse, status = _grouped(w, pages, cuda_device, w.extra["prefix_pages"], forks, num_ctas)
    assert status == 0
    ref_out, ref_lse = oracle_decode(w, ref_pages)
    assert_close(out, lse, ref_out, ref_lse, what=f"{groups}x{forks} prefix {prefix} G={num_ctas}")


@pytest.mark.parametrize("nq,prefix,suffix", [(2, 1024, 90.0), (4, 1024, 90.0), (4, 16384, 8.0)])
def test_groups_with_drafts(cuda_device, nq, prefix, suffix):
    """Drafts see the shared prefix and their own causal suffix; the last case has
    suffixes of a few tokens, so the four drafts' rows differ only in the last page."""
    w = wl.prefix_shared(seed=60 + nq, groups=2, forks=4, prefix=prefix, suffix_median=suffix,
                         suffix_max=400, num_queries=nq)
    pages = gpu_fill_cache(w, cuda_device)
    ref_pages = oracle_fill_cache(w)
    out, lse, status = _grouped(w, pages, cuda_device, w.extra["prefix_pages"], 4)
    assert status == 0
    ref_out, ref_lse = oracle_decode(w, ref_pages)
    assert_close(out, lse, ref_out, ref_lse, what=f"drafts Q={nq}")


def test_no_prefix_and_bad_rows(cuda_device):
    """prefix_pages = 0 is mla_decode; a request shorter than its prefix is a bad row."""
    dev = cuda_device
    w = wl.prefix_shared(seed=70, groups=3, forks=2, prefix=512, suffix_median=120.0,
                         suffix_max=600)
    pages = gpu_fill_cache(w, dev)
    ref_pages = oracle_fill_cache(w)
    ref_out, ref_lse = oracle_decode(w, ref_pages)
    out, lse, status = _grouped(w, pages, dev, [0, 0, 0], 2)
    assert status == 0
    assert_close(out, lse, ref_out, ref_lse, what="no shared prefix")
    # request 3 (group 1) cut to 100 tokens, shorter than its group's 8-page prefix
    lens = w.seq_lens.copy()
    lens[3] = 100
    out, lse, status = _grouped(w, pages, dev, w.extra["prefix_pages"], 2, seq_lens=lens)
    assert status & binding.MLA_DEVICE_ERR_BAD_LENGTH
    assert np.all(out[3] == 0) and np.all(np.isneginf(lse[3]))
    good = [b for b in range(w.batch) if b != 3]
    assert_close(out[good], lse[good], ref_out[good], ref_lse[good], what="other rows")


@pytest.mark.slow
def test_full_prefix_shared_workload(cuda_device):
    """The prefix-shared workload (16 groups x 4 forks, 120k-token prefix), sampled."""
    w = wl.prefix_shared()
    pages = gpu_fill_cache(w, cuda_device)
    out, lse, status = _grouped(w, pages, cuda_device, w.extra["prefix_pages"], 4)
    assert status == 0
    for b in [0, 1, 2, 3, 45]:
        bits = w.request_latent(b)
        codes = oe4m3.encode(oe4m3.bf16_bits_to_f64(bits), w.kv_scale)
        k = oatt.dequant(codes, oatt.KV_E4M3, w.kv_scale)
        ro, rl = oatt.attend(oe4m3.bf16_bits_to_f64(w.q_bits[b, 0]), k, w.sm_scale)
        _, _, lerr = assert_close(out[b, 0], lse[b, 0], ro, rl, what=f"prefix_shared b={b}")
        rel = float(np.abs(out[b, 0] - ro).max() / np.abs(ro).max())
        print(f"grouped prefix_shared b={b}: rel err {rel:.3g} lse err {lerr:.3g}")
        assert rel <= 1e-2
