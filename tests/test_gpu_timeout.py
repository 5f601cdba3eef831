"""A pipeline wait of the FP8 decode kernel that runs out (GPU).

Every wait between the kernel's roles is bounded; when one runs out the CTA sets
MLA_DEVICE_ERR_TIMEOUT in the workspace status word, stops every role, waits for
the copies and MMAs it has already issued and frees its tensor memory, so the
call returns and the device stays usable. To make that path run, the build also
produces a test library (libmla_stall_test.so, not the product) whose QK issuer
waits, before its third page, on a barrier that nothing ever completes, with
waits between roles limited to 20 ms (the drain keeps 2 s). Nothing faults and
nothing waits without a bound.
"""

import numpy as np
import pytest
import torch

from paged_mla_decode_gb300 import binding
from paged_mla_decode_gb300 import build as mla_build
from paged_mla_decode_gb300 import workloads as wl

from .gpu_util import (assert_close, bf16_tensor, gpu_decode, gpu_fill_cache, oracle_decode,
                       oracle_fill_cache)

pytestmark = pytest.mark.gpu


def test_wait_timeout_sets_status_and_device_recovers(cuda_device):
    dev = cuda_device
    stall = binding.open_library(mla_build.STALL_LIB_PATH)
    w = wl.make_lengths_workload("stall", 61, [5000, 3000], num_heads=64)
    pages = gpu_fill_cache(w, dev)
    q = bf16_tensor(w.q_bits, dev)
    table = torch.from_numpy(w.block_table).to(dev)
    lens = torch.from_numpy(w.seq_lens).to(dev)
    out = torch.zeros((w.batch, 1, 64, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((w.batch, 1, 64), dtype=torch.float32, device=dev)
    ctas = 4   # every CTA holds more than two pages, so every CTA reaches the stall
    ws = torch.zeros(stall.mla_decode_workspace_size(w.batch, 1, 64, ctas), dtype=torch.uint8,
                     device=dev)
    st = stall.mla_decode(q.data_ptr(), pages.data_ptr(), pages.shape[0], 64,
                          binding.MLA_KV_E4M3, table.data_ptr(), table.shape[1],
                          lens.data_ptr(), w.batch, 1, 64, w.sm_scale, w.kv_scale, ctas,
                          ws.data_ptr(), ws.numel(), out.data_ptr(), lse.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    assert st == binding.MLA_OK
    torch.cuda.synchronize()   # the call ends: no wait is left running
    status = binding.read_device_status(ws)
    assert status & binding.MLA_DEVICE_ERR_TIMEOUT, f"status {status:#x}"
    # the device is usable afterwards: the product library's decode of the same
    # inputs matches the oracle and reports no error
    got_out, got_lse, ws2 = gpu_decode(w, pages, dev, num_ctas=ctas)
    assert binding.read_device_status(ws2) == 0
    ref_pages = oracle_fill_cache(w)
    assert np.array_equal(pages.cpu().numpy(), ref_pages)
    ref_out, ref_lse = oracle_decode(w, ref_pages)
    assert_close(got_out, got_lse, ref_out, ref_lse, what="after a timed-out call")
