"""mla_decode_static_scratch agrees with mla_decode (GPU).

The static-scratch entry point serves callers that cannot allocate device
memory while they decode: plug-ins inside an engine that keeps all device
memory in its own pool and offers them no allocator, and serving loops that may
not call cudaMalloc (it can synchronise the device) once they run. It keeps the
split-KV scratch in a fixed array inside libmla.so instead of a caller-provided
workspace.

Two calls in a row, on different problems, must each match what mla_decode
returns for the same inputs within the tolerance the parity tests use, so the
array's leftover contents from one call cannot leak into the next. A problem
larger than the array is refused with MLA_ERR_WORKSPACE. This file runs last in
a session and also passes on its own in a fresh process.
"""

import numpy as np
import pytest
import torch

from paged_mla_decode_gb300 import binding
from paged_mla_decode_gb300 import workloads as wl

from .gpu_util import (LSE_ABS_TOL, OUT_ABS_TOL, OUT_REL_TOL, bf16_tensor, gpu_fill_cache)

pytestmark = pytest.mark.gpu


def _inputs(w, dev):
    pages = gpu_fill_cache(w, dev)
    q = bf16_tensor(w.q_bits, dev)
    table = torch.from_numpy(w.block_table).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    return pages, q, table, lens


def _with_workspace(w, pages, q, table, lens, dev):
    B, Q, H = q.shape[:3]
    out = torch.empty((B, Q, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Q, H), dtype=torch.float32, device=dev)
    ws = torch.zeros(binding.mla_decode_workspace_size(B, Q, H), dtype=torch.uint8, device=dev)
    binding.mla_decode(q, pages, table, lens, w.sm_scale, w.kv_scale, out, lse, ws)
    return out, lse


def _static(w, pages, q, table, lens, dev):
    B, Q, H = q.shape[:3]
    out = torch.full((B, Q, H, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, Q, H), float("nan"), dtype=torch.float32, device=dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    binding.mla_decode_static_scratch(q, pages, table, lens, w.sm_scale, w.kv_scale, out, lse,
                                      device_status=status)
    return out, lse, status


def _assert_matches(got, ref):
    g_out, g_lse = got[0].float().cpu().numpy(), got[1].cpu().numpy()
    r_out, r_lse = ref[0].float().cpu().numpy(), ref[1].cpu().numpy()
    assert np.all(np.isfinite(g_out))
    err = np.abs(g_out - r_out).max()
    assert err <= OUT_REL_TOL * np.abs(r_out).max() + OUT_ABS_TOL, err
    assert np.abs(g_lse - r_lse).max() <= LSE_ABS_TOL


def test_two_calls_match_workspace_decode(cuda_device):
    dev = cuda_device
    wa = wl.make_lengths_workload("static-a", 50, [3000, 777, 64], num_heads=64, num_queries=2)
    wb = wl.make_lengths_workload("static-b", 51, [1500, 1, 200], num_heads=16, num_queries=1)
    a, b = _inputs(wa, dev), _inputs(wb, dev)
    ref_a = _with_workspace(wa, *a, dev)
    ref_b = _with_workspace(wb, *b, dev)
    got_a = _static(wa, *a, dev)      # first call
    got_b = _static(wb, *b, dev)      # second call, different shape, same scratch
    torch.cuda.synchronize()
    _assert_matches(got_a, ref_a)
    _assert_matches(got_b, ref_b)
    assert int(got_a[2].item()) == 0 and int(got_b[2].item()) == 0


def test_status_is_per_call_and_size_limit(cuda_device):
    dev = cuda_device
    w = wl.make_lengths_workload("static-c", 52, [300, 200], num_heads=16)
    pages, q, table, lens = _inputs(w, dev)
    bad = table.clone()
    bad[0, 1] = w.num_pages + 3                   # a page outside the cache
    _, _, st_bad = _static(w, pages, q, bad, lens, dev)
    got = _static(w, pages, q, table, lens, dev)  # the next call starts clean
    ref = _with_workspace(w, pages, q, table, lens, dev)
    torch.cuda.synchronize()
    assert int(st_bad.item()) & binding.MLA_DEVICE_ERR_BAD_PAGE
    assert int(got[2].item()) == 0
    _assert_matches(got, ref)
    # more rows than the array holds: refused on the host, nothing enqueued
    big = torch.empty((400, 4, 64, 576), dtype=torch.bfloat16, device=dev)
    with pytest.raises(binding.MlaError) as e:
        binding.mla_decode_static_scratch(
            big, pages, torch.zeros((400, 1), dtype=torch.int32, device=dev),
            torch.ones(400, dtype=torch.int32, device=dev), 0.1, 1.0,
            torch.empty((400, 4, 64, 512), dtype=torch.bfloat16, device=dev),
            torch.empty((400, 4, 64), dtype=torch.float32, device=dev))
    assert e.value.status == binding.MLA_ERR_WORKSPACE
