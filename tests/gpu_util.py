"""Helpers shared by the GPU parity tests.

Inputs come from the seeded workload generator; expected values come only from
the float64 oracle (``oracle/``), never from the CUDA path.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import attention as oatt
from oracle import e4m3 as oe4m3
from paged_mla_decode_gb300 import binding

OUT_REL_TOL = 1e-2   # max|err| <= 1e-2 * max|ref| + 1e-3 for out
OUT_ABS_TOL = 1e-3
LSE_ABS_TOL = 1e-3   # absolute, for lse


def bf16_tensor(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def gpu_fill_cache(w, dev, kv_dtype="e4m3", table_map=None, pages_total=None, chunk=1 << 16):
    """Fill a device page pool with every segment of ``w`` through mla_kv_append."""
    n = pages_total if pages_total is not None else w.num_pages
    dt = torch.uint8 if kv_dtype == "e4m3" else torch.bfloat16
    pages = torch.zeros((n, 64, 576), dtype=dt, device=dev)
    scale = w.kv_scale if kv_dtype == "e4m3" else 1.0
    for si in range(len(w.segments)):
        bits = w.segment_latent(si)
        slots = w.segment_slots(si, table_map)
        for a in range(0, bits.shape[0], chunk):
            x = bf16_tensor(bits[a:a + chunk], dev)
            binding.mla_kv_append(x[:, :512].contiguous(), x[:, 512:].contiguous(),
                                  torch.from_numpy(slots[a:a + chunk]).to(dev), pages, scale)
    return pages


def oracle_fill_cache(w, kv_dtype="e4m3"):
    """The same cache built by the oracle's codec (uint8 codes or bf16 bits)."""
    if kv_dtype == "e4m3":
        pages = np.zeros((w.num_pages, 64, 576), dtype=np.uint8)
    else:
        pages = np.zeros((w.num_pages, 64, 576), dtype=np.uint16)
    flat = pages.reshape(-1, 576)
    for si in range(len(w.segments)):
        bits = w.segment_latent(si)
        slots = w.segment_slots(si)
        if kv_dtype == "e4m3":
            flat[slots] = oe4m3.encode(oe4m3.bf16_bits_to_f64(bits), w.kv_scale)
        else:
            flat[slots] = bits
    return pages


def gpu_decode(w, pages, dev, num_ctas=0, q_bits=None, seq_lens=None, block_table=None,
               kv_scale=None, workspace=None, f16_operands=False):
    q = bf16_tensor(w.q_bits if q_bits is None else q_bits, dev)
    table = torch.from_numpy(w.block_table if block_table is None else block_table).to(dev)
    lens = torch.from_numpy(w.seq_lens if seq_lens is None else seq_lens).to(dev)
    B, Q, H = q.shape[:3]
    out = torch.full((B, Q, H, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, Q, H), float("nan"), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.zeros(binding.mla_decode_workspace_size(B, Q, H, num_ctas),
                                dtype=torch.uint8, device=dev)
    scale = w.kv_scale if kv_scale is None else kv_scale
    binding.mla_decode(q, pages, table, lens, w.sm_scale, scale, out, lse, workspace,
                       num_ctas=num_ctas, f16_operands=f16_operands)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), workspace


def assert_close(got_out, got_lse, ref_out, ref_lse, rows=None, what=""):
    """The stated tolerance: out within 1e-2*max|ref| + 1e-3, lse within 1e-3."""
    if rows is not None:
        idx = tuple(np.array(rows).T)
        got_out, ref_out = got_out[idx], ref_out[idx]
        got_lse, ref_lse = got_lse[idx], ref_lse[idx]
    assert np.all(np.isfinite(got_out)), f"{what}: non-finite output"
    err = np.abs(got_out - ref_out).max()
    tol = OUT_REL_TOL * np.abs(ref_out).max() + OUT_ABS_TOL
    lerr = np.abs(got_lse - ref_lse).max()
    assert err <= tol, f"{what}: out err {err:.4g} > tol {tol:.4g}"
    assert lerr <= LSE_ABS_TOL, f"{what}: lse err {lerr:.4g}"
    return err, tol, lerr


def oracle_decode(w, pages_ref, kv_dtype="e4m3", rows=None, q_bits=None, seq_lens=None,
                  block_table=None):
    return oatt.decode(w.q_bits if q_bits is None else q_bits, pages_ref,
                       w.block_table if block_table is None else block_table,
                       w.seq_lens if seq_lens is None else seq_lens, w.sm_scale,
                       w.kv_scale if kv_dtype == "e4m3" else 1.0,
                       kv_dtype=oatt.KV_E4M3 if kv_dtype == "e4m3" else oatt.KV_BF16, rows=rows)
