"""mla_kv_append is bit-exact against the oracle's e4m3 rounding (GPU).

Inputs cover every bfloat16 bit pattern, awkward float32 scales whose
quotients land near e4m3 rounding midpoints, signed zeros, saturation, NaN,
skipped slots (-1) and the bf16 copy variant.
"""

import numpy as np
import pytest
import torch

from oracle import e4m3 as oe4m3
from paged_mla_decode_gb300 import binding

from .gpu_util import bf16_tensor

pytestmark = pytest.mark.gpu


def _append(bits, slots, num_pages, scale, dev, dtype=torch.uint8):
    pages = torch.zeros((num_pages, 64, 576), dtype=dtype, device=dev)
    x = bf16_tensor(bits, dev)
    binding.mla_kv_append(x[:, :512].contiguous(), x[:, 512:].contiguous(),
                          torch.from_numpy(slots.astype(np.int32)).to(dev), pages, scale)
    torch.cuda.synchronize()
    return pages.cpu()


def _compare_codes(got, ref):
    got = got.astype(np.uint8)
    nan_g = (got & 0x7F) == 0x7F
    nan_r = (ref & 0x7F) == 0x7F
    assert np.array_equal(nan_g, nan_r)
    bad = np.nonzero((got != ref) & ~nan_r)
    assert bad[0].size == 0, (bad[0][:5], got[bad][:5], ref[bad][:5])


@pytest.mark.parametrize("scale", [1.0, float(np.float32(4.0 / 448.0)), float(np.float32(0.0123456)),
                                   float(np.float32(3.0e-5)), float(np.float32(7.77))])
def test_every_bf16_pattern(cuda_device, scale):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ntok = -(-bits.size // 576)
    padded = np.zeros(ntok * 576, np.uint16)
    padded[:bits.size] = bits
    tokens = padded.reshape(ntok, 576)
    rng = np.random.default_rng(1)
    npages = 4
    slots = rng.permutation(npages * 64)[:ntok]
    got = _append(tokens, slots, npages, scale, cuda_device).numpy().reshape(-1, 576)[slots]
    ref = oe4m3.encode(oe4m3.bf16_bits_to_f64(tokens), scale)
    _compare_codes(got, ref)


def test_near_midpoint_quotients(cuda_device):
    # x / s lands within float32 rounding of an e4m3 midpoint: for each midpoint m and a
    # random scale s, take the bf16 neighbours of m*s.
    rng = np.random.default_rng(2)
    mids = []
    vals = [oe4m3.code_value(c) for c in range(0x7E)]
    for a, b in zip(vals[:-1], vals[1:]):
        mids.append(0.5 * (a + b))
    mids = np.array(mids)
    xs, scales = [], []
    for s in rng.uniform(0.001, 3.0, size=40).astype(np.float32):
        target = mids * np.float64(s)
        t32 = target.astype(np.float32)
        b = (t32.view(np.uint32) >> 16).astype(np.int64)
        for d in (-1, 0, 1):
            xs.append(((b + d).astype(np.uint16)))
        scales.append(float(s))
    for s, chunk in zip(scales, np.array_split(np.concatenate(xs), len(scales))):
        ntok = -(-chunk.size // 576)
        tokens = np.zeros(ntok * 576, np.uint16)
        tokens[:chunk.size] = chunk
        tokens = tokens.reshape(ntok, 576)
        slots = np.arange(ntok)
        got = _append(tokens, slots, 1, s, cuda_device).numpy().reshape(-1, 576)[:ntok]
        ref = oe4m3.encode(oe4m3.bf16_bits_to_f64(tokens), s)
        _compare_codes(got, ref)


def test_skipped_and_out_of_range_slots(cuda_device):
    rng = np.random.default_rng(3)
    bits = (rng.standard_normal((5, 576)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    slots = np.array([3, -1, 64 * 2 - 1, 64 * 2, 5])   # 128 is outside a 2-page cache
    got = _append(bits, slots, 2, 0.01, cuda_device).numpy().reshape(-1, 576)
    ref = oe4m3.encode(oe4m3.bf16_bits_to_f64(bits), 0.01)
    assert np.array_equal(got[3], ref[0])
    assert np.array_equal(got[127], ref[2])
    assert np.array_equal(got[5], ref[4])
    written = {3, 127, 5}
    for s in range(128):
        if s not in written:
            assert not got[s].any()


def test_bf16_copy(cuda_device):
    rng = np.random.default_rng(4)
    bits = (rng.standard_normal((70, 576)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    slots = rng.permutation(128)[:70]
    got = _append(bits, slots, 2, 1.0, cuda_device, dtype=torch.bfloat16)
    got = got.view(torch.int16).numpy().view(np.uint16).reshape(-1, 576)[slots]
    assert np.array_equal(got, bits)


def test_invalid_arguments_raise(cuda_device):
    pages = torch.zeros((1, 64, 576), dtype=torch.uint8, device=cuda_device)
    x = torch.zeros((1, 576), dtype=torch.bfloat16, device=cuda_device)
    slots = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    with pytest.raises(binding.MlaError):
        binding.mla_kv_append(x[:, :512].contiguous(), x[:, 512:].contiguous(), slots, pages, 0.0)
    bpages = torch.zeros((1, 64, 576), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(binding.MlaError):
        binding.mla_kv_append(x[:, :512].contiguous(), x[:, 512:].contiguous(), slots, bpages, 2.0)


def test_float32_quotient_on_midpoint(cuda_device):
    # Scales chosen as s = float32(x / m) for an e4m3 midpoint m: the float32 quotient
    # x / s then rounds exactly onto m while the real quotient lies just beside it, so
    # only the exact-remainder correction gives the right code.
    rng = np.random.default_rng(5)
    vals = [oe4m3.code_value(c) for c in range(0x7E)]
    mids = [0.5 * (a + b) for a, b in zip(vals[:-1], vals[1:])]
    exercised = 0
    for trial in range(300):
        m = mids[rng.integers(len(mids))]
        xb = np.array([rng.standard_normal()], np.float32).view(np.uint32) >> 16
        xb = xb.astype(np.uint16)
        x = float(oe4m3.bf16_bits_to_f64(xb)[0])
        if x == 0.0:
            continue
        s = float(np.float32(abs(x) / m))
        if not np.isfinite(s) or s <= 0:
            continue
        q32 = np.float32(x) / np.float32(s)
        if abs(float(q32)) == m and abs(x) / s != m:
            exercised += 1
        token = np.zeros((1, 576), np.uint16)
        token[0, 0] = xb[0]
        token[0, 1:] = (rng.standard_normal(575).astype(np.float32).view(np.uint32) >> 16)
        got = _append(token, np.array([0]), 1, s, cuda_device).numpy().reshape(-1, 576)[:1]
        ref = oe4m3.encode(oe4m3.bf16_bits_to_f64(token), s)
        _compare_codes(got, ref)
    assert exercised >= 50
