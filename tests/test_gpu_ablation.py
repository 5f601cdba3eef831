"""The FP8-operand ablation entry (mla_decode_f16_operands) against the oracle.

mla_decode reads an e4m3 cache's bytes as tensor-core operands; the ablation
widens them to f16 first. Both must meet the same tolerance against the oracle
("Smaller, faster, safer: running Kimi and GLM at scale", section "Quantizing the
KV cache": the FP8 cache is dequantised with one scale), and agree with each other.
"""
import numpy as np
import pytest

from paged_mla_decode_gb300 import workloads as wl

from .gpu_util import assert_close, gpu_decode, gpu_fill_cache, oracle_decode, oracle_fill_cache

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("heads,nq", [(64, 1), (32, 2), (16, 4)])
def test_f16_operand_path_matches_oracle(cuda_device, heads, nq):
    lengths = [nq, 63 + nq, 64 + nq, 700, 1500]
    w = wl.make_lengths_workload("ablation", 50 + heads + nq, lengths, num_heads=heads,
                                 num_queries=nq)
    pages = gpu_fill_cache(w, cuda_device)
    ref_out, ref_lse = oracle_decode(w, oracle_fill_cache(w))
    out16, lse16, _ = gpu_decode(w, pages, cuda_device, f16_operands=True)
    assert_close(out16, lse16, ref_out, ref_lse, what=f"f16 operands H={heads} Q={nq}")
    out8, lse8, _ = gpu_decode(w, pages, cuda_device)
    assert_close(out8, lse8, ref_out, ref_lse, what=f"fp8 operands H={heads} Q={nq}")
    # the two operand paths agree with each other at least as well as with the oracle
    scale = np.abs(ref_out).max()
    assert np.abs(out8 - out16).max() <= 2e-2 * scale + 2e-3
    assert np.abs(lse8 - lse16).max() <= 2e-3
