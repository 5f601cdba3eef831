"""mla_decode_combine merges partials like the oracle's log-sum-exp merge (GPU)."""

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from paged_mla_decode_gb300 import binding

from .gpu_util import LSE_ABS_TOL, OUT_ABS_TOL, OUT_REL_TOL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("num_parts,rows", [(1, 3), (7, 64), (152, 5), (300, 2)])
def test_combine_matches_oracle_merge(cuda_device, num_parts, rows):
    rng = np.random.default_rng(num_parts * 1000 + rows)
    part_out = rng.standard_normal((num_parts, rows, 512)).astype(np.float32) * 0.1
    part_lse = (rng.standard_normal((num_parts, rows)) * 3).astype(np.float32)
    # empty parts (lse = -inf) and one all-empty row
    part_lse[rng.random((num_parts, rows)) < 0.2] = -np.inf
    part_lse[:, 0] = -np.inf
    out = torch.empty((rows, 512), dtype=torch.bfloat16, device=cuda_device)
    lse = torch.empty(rows, dtype=torch.float32, device=cuda_device)
    binding.mla_decode_combine(torch.from_numpy(part_out).to(cuda_device),
                               torch.from_numpy(part_lse).to(cuda_device), out, lse)
    torch.cuda.synchronize()
    ref_out, ref_lse = oatt.merge(part_out.astype(np.float64), part_lse.astype(np.float64))
    got_out, got_lse = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(got_out[0] == 0) and np.isneginf(got_lse[0])
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got_lse), fin)
    assert np.abs(got_lse[fin] - ref_lse[fin]).max() <= LSE_ABS_TOL
    err = np.abs(got_out - ref_out).max()
    assert err <= OUT_REL_TOL * np.abs(ref_out).max() + OUT_ABS_TOL


def test_combine_zero_parts(cuda_device):
    out = torch.full((4, 512), 7.0, dtype=torch.bfloat16, device=cuda_device)
    lse = torch.zeros(4, dtype=torch.float32, device=cuda_device)
    binding.mla_decode_combine(torch.zeros((0, 4, 512), device=cuda_device),
                               torch.zeros((0, 4), device=cuda_device), out, lse)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
