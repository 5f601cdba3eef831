"""Thin ctypes binding of libmla.so (argument marshalling only).

Each function has the name of the C entry point it calls and takes PyTorch
tensors, from which it passes device pointers, sizes and the current CUDA
stream. All computation happens in the library's CUDA kernels; there is no
fallback: if ``libmla.so`` is missing the first call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CUDA = 4

MLA_KV_E4M3 = 0
MLA_KV_BF16 = 1

MLA_DEVICE_ERR_BAD_PAGE = 0x1
MLA_DEVICE_ERR_BAD_LENGTH = 0x2
MLA_DEVICE_ERR_TIMEOUT = 0x4

MLA_KV_CHECK_TAG_MISMATCH = 0x1
MLA_KV_CHECK_PAGE_RANGE = 0x2
MLA_KV_CHECK_BAD_LENGTH = 0x4

EXPORTED = ("mla_abi_version", "mla_status_string", "mla_kv_append",
            "mla_decode_workspace_size", "mla_decode", "mla_decode_f16_operands",
            "mla_decode_grouped_workspace_size", "mla_decode_grouped",
            "mla_decode_combine", "mla_kv_check", "mla_decode_static_scratch")

_lib = None


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmla.so once and declare the argument types of every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    _lib = open_library(path)
    return _lib


def open_library(path: str) -> ctypes.CDLL:
    """Open a build of the library at ``path`` (not cached) with its argument types."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run paged_mla_decode_gb300.build.build() "
                           "(or __graft_entry__.build()) first")
    lib = ctypes.CDLL(path)
    c = ctypes
    lib.mla_abi_version.restype = c.c_int
    lib.mla_abi_version.argtypes = []
    lib.mla_status_string.restype = c.c_char_p
    lib.mla_status_string.argtypes = [c.c_int]
    lib.mla_kv_append.restype = c.c_int
    lib.mla_kv_append.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64, c.c_void_p,
                                  c.c_int64, c.c_int, c.c_int, c.c_float, c.c_void_p]
    lib.mla_decode_workspace_size.restype = c.c_size_t
    lib.mla_decode_workspace_size.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int]
    lib.mla_decode.restype = c.c_int
    lib.mla_decode.argtypes = [c.c_void_p, c.c_void_p, c.c_int64, c.c_int, c.c_int, c.c_void_p,
                               c.c_int, c.c_void_p, c.c_int, c.c_int, c.c_int, c.c_float,
                               c.c_float, c.c_int, c.c_void_p, c.c_size_t, c.c_void_p,
                               c.c_void_p, c.c_void_p]
    lib.mla_decode_f16_operands.restype = c.c_int
    lib.mla_decode_f16_operands.argtypes = lib.mla_decode.argtypes
    lib.mla_decode_grouped_workspace_size.restype = c.c_size_t
    lib.mla_decode_grouped_workspace_size.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int]
    lib.mla_decode_grouped.restype = c.c_int
    lib.mla_decode_grouped.argtypes = [c.c_void_p, c.c_void_p, c.c_int64, c.c_int, c.c_int,
                                       c.c_void_p, c.c_int, c.c_void_p, c.c_int, c.c_int,
                                       c.c_int, c.c_int, c.c_void_p, c.c_float, c.c_float,
                                       c.c_int, c.c_void_p, c.c_size_t, c.c_void_p, c.c_void_p,
                                       c.c_void_p]
    lib.mla_decode_combine.restype = c.c_int
    lib.mla_decode_combine.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_int64, c.c_void_p,
                                       c.c_void_p, c.c_void_p]
    lib.mla_kv_check.restype = c.c_int
    lib.mla_kv_check.argtypes = [c.c_void_p, c.c_int64, c.c_void_p, c.c_void_p, c.c_int,
                                 c.c_void_p, c.c_int, c.c_int, c.c_void_p, c.c_void_p,
                                 c.c_void_p]
    lib.mla_decode_static_scratch.restype = c.c_int
    lib.mla_decode_static_scratch.argtypes = [
        c.c_void_p, c.c_void_p, c.c_int64, c.c_int, c.c_int, c.c_void_p, c.c_int, c.c_void_p,
        c.c_int, c.c_int, c.c_int, c.c_float, c.c_float, c.c_int, c.c_void_p, c.c_void_p,
        c.c_void_p, c.c_void_p]
    return lib


def status_string(status: int) -> str:
    return load_library().mla_status_string(int(status)).decode()


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check(status: int, where: str):
    if status != MLA_OK:
        raise MlaError(status, where)


def kv_dtype_code(kv_pages: torch.Tensor) -> int:
    if kv_pages.dtype == torch.uint8:
        return MLA_KV_E4M3
    if kv_pages.dtype == torch.bfloat16:
        return MLA_KV_BF16
    raise TypeError("kv_pages must be uint8 (e4m3 codes) or bfloat16")


def mla_kv_append(latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor,
                  kv_pages: torch.Tensor, kv_scale: float, stream=None) -> None:
    """Write tokens' 512 latent + 64 rope elements into their cache slots."""
    num_tokens = int(slot_mapping.numel())
    assert latent.dtype == torch.bfloat16 and rope.dtype == torch.bfloat16
    assert slot_mapping.dtype == torch.int32
    assert latent.is_contiguous() and rope.is_contiguous() and kv_pages.is_contiguous()
    assert latent.shape == (num_tokens, 512) and rope.shape == (num_tokens, 64)
    assert kv_pages.dim() == 3 and kv_pages.shape[2] == 576
    st = load_library().mla_kv_append(_ptr(latent), _ptr(rope), _ptr(slot_mapping), num_tokens,
                                      _ptr(kv_pages), int(kv_pages.shape[0]),
                                      int(kv_pages.shape[1]), kv_dtype_code(kv_pages),
                                      float(kv_scale), _stream(stream))
    _check(st, "mla_kv_append")


def mla_decode_workspace_size(batch: int, num_queries: int, num_heads: int,
                              num_ctas: int = 0) -> int:
    return int(load_library().mla_decode_workspace_size(batch, num_queries, num_heads, num_ctas))


def mla_decode(q: torch.Tensor, kv_pages: torch.Tensor, block_table: torch.Tensor,
               seq_lens: torch.Tensor, sm_scale: float, kv_scale: float, out: torch.Tensor,
               lse: torch.Tensor, workspace: torch.Tensor, num_ctas: int = 0,
               stream=None, f16_operands: bool = False) -> None:
    """Split-KV paged MLA decode (combine included) into ``out`` and ``lse``.

    ``f16_operands`` calls mla_decode_f16_operands (the e4m3 cache widened to f16
    operands) instead of mla_decode."""
    assert q.dtype == torch.bfloat16 and q.dim() == 4 and q.shape[3] == 576 and q.is_contiguous()
    batch, nq, heads, _ = q.shape
    assert block_table.dtype == torch.int32 and block_table.dim() == 2
    assert block_table.is_contiguous() and block_table.shape[0] == batch
    assert seq_lens.dtype == torch.int32 and seq_lens.numel() == batch
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == (batch, nq, heads, 512)
    assert lse.dtype == torch.float32 and tuple(lse.shape) == (batch, nq, heads)
    assert kv_pages.is_contiguous() and kv_pages.dim() == 3 and kv_pages.shape[2] == 576
    lib = load_library()
    fn = lib.mla_decode_f16_operands if f16_operands else lib.mla_decode
    st = fn(
        _ptr(q), _ptr(kv_pages), int(kv_pages.shape[0]), int(kv_pages.shape[1]),
        kv_dtype_code(kv_pages), _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
        batch, nq, heads, float(sm_scale), float(kv_scale), int(num_ctas), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _ptr(out), _ptr(lse),
        _stream(stream))
    _check(st, "mla_decode_f16_operands" if f16_operands else "mla_decode")


def mla_decode_grouped_workspace_size(batch: int, num_queries: int, num_heads: int,
                                      num_ctas: int = 0) -> int:
    return int(load_library().mla_decode_grouped_workspace_size(batch, num_queries, num_heads,
                                                                num_ctas))


def mla_decode_grouped(q: torch.Tensor, kv_pages: torch.Tensor, block_table: torch.Tensor,
                       seq_lens: torch.Tensor, forks: int, prefix_pages: torch.Tensor,
                       sm_scale: float, kv_scale: float, out: torch.Tensor, lse: torch.Tensor,
                       workspace: torch.Tensor, num_ctas: int = 0, stream=None) -> None:
    """mla_decode for groups of ``forks`` requests sharing ``prefix_pages[g]`` pages."""
    assert q.dtype == torch.bfloat16 and q.dim() == 4 and q.shape[3] == 576 and q.is_contiguous()
    batch, nq, heads, _ = q.shape
    assert block_table.dtype == torch.int32 and block_table.dim() == 2
    assert block_table.is_contiguous() and block_table.shape[0] == batch
    assert seq_lens.dtype == torch.int32 and seq_lens.numel() == batch
    assert prefix_pages.dtype == torch.int32 and prefix_pages.is_contiguous()
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == (batch, nq, heads, 512)
    assert lse.dtype == torch.float32 and tuple(lse.shape) == (batch, nq, heads)
    assert kv_pages.is_contiguous() and kv_pages.dim() == 3 and kv_pages.shape[2] == 576
    st = load_library().mla_decode_grouped(
        _ptr(q), _ptr(kv_pages), int(kv_pages.shape[0]), int(kv_pages.shape[1]),
        kv_dtype_code(kv_pages), _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
        batch, nq, heads, int(forks), _ptr(prefix_pages), float(sm_scale), float(kv_scale),
        int(num_ctas), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
        _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "mla_decode_grouped")


def mla_decode_combine(part_out: torch.Tensor, part_lse: torch.Tensor, out: torch.Tensor,
                       lse: torch.Tensor, stream=None) -> None:
    """Merge ``part_out [S, R, 512]`` / ``part_lse [S, R]`` into ``out [R, 512]`` / ``lse [R]``."""
    assert part_out.dtype == torch.float32 and part_lse.dtype == torch.float32
    num_parts, rows = int(part_lse.shape[0]), int(part_lse.shape[1])
    assert tuple(part_out.shape) == (num_parts, rows, 512) and part_out.is_contiguous()
    assert part_lse.is_contiguous()
    assert out.dtype == torch.bfloat16 and out.numel() == rows * 512 and out.is_contiguous()
    assert lse.dtype == torch.float32 and lse.numel() == rows
    st = load_library().mla_decode_combine(_ptr(part_out), _ptr(part_lse), num_parts, rows,
                                           _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "mla_decode_combine")


def mla_kv_check(page_tags: torch.Tensor, block_table: torch.Tensor,
                 expected_tags: torch.Tensor, seq_lens: torch.Tensor,
                 request_status: torch.Tensor, checked_seq_lens: torch.Tensor,
                 stream=None) -> None:
    """Compare each request's expected page tags with the pages' current tags.

    ``page_tags [num_pages]`` and ``expected_tags [batch, max_pages]`` hold 32-bit
    tags (int32 or uint32 tensors; compared as unsigned), ``block_table`` and
    ``seq_lens`` are the decode call's. Writes ``request_status [batch]``
    (MLA_KV_CHECK_* bits, int32) and ``checked_seq_lens [batch]`` (the lengths,
    -1 for every request that failed), to be passed to mla_decode as seq_lens.
    """
    tag_types = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
    assert page_tags.dtype in tag_types and page_tags.dim() == 1 and page_tags.is_contiguous()
    assert block_table.dtype == torch.int32 and block_table.dim() == 2
    assert block_table.is_contiguous()
    batch, max_pages = int(block_table.shape[0]), int(block_table.shape[1])
    assert expected_tags.dtype in tag_types and expected_tags.is_contiguous()
    assert tuple(expected_tags.shape) == (batch, max_pages)
    assert seq_lens.dtype == torch.int32 and seq_lens.numel() == batch
    assert request_status.dtype in tag_types and request_status.numel() == batch
    assert checked_seq_lens.dtype == torch.int32 and checked_seq_lens.numel() == batch
    st = load_library().mla_kv_check(_ptr(page_tags), int(page_tags.numel()), _ptr(block_table),
                                     _ptr(expected_tags), max_pages, _ptr(seq_lens), batch, 64,
                                     _ptr(request_status), _ptr(checked_seq_lens),
                                     _stream(stream))
    _check(st, "mla_kv_check")


def mla_decode_static_scratch(q: torch.Tensor, kv_pages: torch.Tensor,
                              block_table: torch.Tensor, seq_lens: torch.Tensor, sm_scale: float,
                              kv_scale: float, out: torch.Tensor, lse: torch.Tensor,
                              device_status: torch.Tensor | None = None, num_ctas: int = 0,
                              stream=None) -> None:
    """mla_decode without a workspace, for callers that cannot allocate device memory.

    The split-KV scratch is a fixed array inside libmla.so (MLA_STATIC_SCRATCH_BYTES),
    shared by every call on a device: calls must not overlap on the GPU. The first
    call on a device looks up the array's address and should precede any stream
    capture. ``device_status`` (int32, one element, optional) receives the call's
    MLA_DEVICE_ERR_* bits.
    """
    assert q.dtype == torch.bfloat16 and q.dim() == 4 and q.shape[3] == 576 and q.is_contiguous()
    batch, nq, heads, _ = q.shape
    assert block_table.dtype == torch.int32 and block_table.dim() == 2
    assert block_table.is_contiguous() and block_table.shape[0] == batch
    assert seq_lens.dtype == torch.int32 and seq_lens.numel() == batch
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == (batch, nq, heads, 512)
    assert lse.dtype == torch.float32 and tuple(lse.shape) == (batch, nq, heads)
    assert kv_pages.is_contiguous() and kv_pages.dim() == 3 and kv_pages.shape[2] == 576
    if device_status is not None:
        assert device_status.dtype == torch.int32 and device_status.numel() >= 1
    st = load_library().mla_decode_static_scratch(
        _ptr(q), _ptr(kv_pages), int(kv_pages.shape[0]), int(kv_pages.shape[1]),
        kv_dtype_code(kv_pages), _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
        batch, nq, heads, float(sm_scale), float(kv_scale), int(num_ctas), _ptr(out), _ptr(lse),
        _ptr(device_status), _stream(stream))
    _check(st, "mla_decode_static_scratch")


def read_device_status(workspace: torch.Tensor) -> int:
    """The sticky device status word at the head of a decode workspace (syncs)."""
    return int(workspace[:4].view(torch.int32).item()) & 0xFFFFFFFF
