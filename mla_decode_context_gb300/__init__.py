"""Thin Python binding of libdcp.so (the DCP MLA decode hot path on GB300).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Functions named like the C entry points take caller-allocated
torch tensors; ``decode_partial`` and ``lse_combine`` allocate their outputs
with torch and call the same entry points.  PyTorch provides device memory
and streams, nothing else.

The library is loaded on first use; if it has not been built the call raises
(there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build_lib import LIB as _LIB_PATH

LATENT_DIM = 512
ROPE_DIM = 64
KV_DIM = 576
MAX_SHARDS = 32

DEVERR_BAD_BLOCK = 1
DEVERR_SEQ_TOO_LONG = 2
DEVERR_BAD_ROWS = 4
DEVERR_TIMEOUT = 8

def compute_dtype() -> str:
    """Arithmetic type of the decode contraction: bf16 tensor-core MMAs with
    fp32 accumulation, or fp32 FMA when the CUDA-core kernel is forced
    (DCP_FORCE_SIMT=1) or the layout has no tensor-core tiling."""
    return "f32" if os.environ.get("DCP_FORCE_SIMT", "") == "1" else "bf16"

DTYPE_BF16 = 0
DTYPE_F32 = 1
KV_BF16 = 0
KV_FP8_E4M3 = 1

STATUS = {0: "DCP_OK", 1: "DCP_ERR_INVALID_ARG", 2: "DCP_ERR_UNSUPPORTED_DTYPE",
          3: "DCP_ERR_MISALIGNED", 4: "DCP_ERR_TABLE_TOO_NARROW",
          5: "DCP_ERR_WORKSPACE_TOO_SMALL", 6: "DCP_ERR_CUDA", 7: "DCP_ERR_TIMEOUT"}

# (name, restype, argtypes) of every symbol include/dcp.h declares
_P, _I32, _I64, _F, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
EXPORTS = [
    ("dcp_status_str", ctypes.c_char_p, [ctypes.c_int]),
    ("dcp_version", ctypes.c_int, []),
    ("dcp_shard_of", _I32, [_I64, _I32, _I32]),
    ("dcp_local_len", _I32, [_I32, _I32, _I32, _I32]),
    ("dcp_decode_workspace_size", _SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    ("dcp_decode_kernel_launches", _I32, [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _SZ]),
    ("dcp_mla_decode_partial", ctypes.c_int,
     [_P, _I64, _P, _I32, _I32, _P, _I32, _I64, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _F,
      _P, _P, _P, _SZ, _P, _P]),
    ("dcp_lse_combine", ctypes.c_int, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, ctypes.c_int, _P, _P]),
    ("dcp_mla_decode_partial_local", ctypes.c_int,
     [_P, _I64, _P, _I32, _I32, _P, _I32, _I64, _I64, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
      _I32, _F, _P, _P, _P, _SZ, _P, _P]),
    ("dcp_mla_decode_partial_v2", ctypes.c_int,
     [_P, _I64, _P, ctypes.c_int, _P, _I32, _I32, _P, _I32, _I64, _I32, _I64, _I32, _I32, _P, _P, _I32, _I32, _I32,
      _I32, _I32, _I32, _I32, _F, _P, ctypes.c_int, _P, _P, _SZ, _P, _P]),
    ("dcp_lse_combine_v2", ctypes.c_int, [_P, ctypes.c_int, _P, _P, _P, _I32, _I32, _I32, _I32, _P, ctypes.c_int, _P,
                                          _P]),
    ("dcp_decode_concat_cache", ctypes.c_int,
     [_P, _I64, _I64, _P, _I64, _I64, _P, _I64, _P, _I64, _P, _I32, _I32, _P, _I64, _P, _I64, _P, _P]),
    ("dcp_mla_decode_partial_noalloc", ctypes.c_int,
     [_P, _I64, _P, _I32, _I32, _P, _I32, _I64, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _F,
      _P, _P, _P, _P]),
]

_lib = None


class DCPError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__("%s returned %s" % (where, STATUS.get(status, status)))
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libdcp.so (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libdcp.so is not built (%s); run __graft_entry__.build()" % _LIB_PATH)
        l = ctypes.CDLL(_LIB_PATH)
        for name, res, args in EXPORTS:
            f = getattr(l, name)
            f.restype, f.argtypes = res, args
        _lib = l
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need_opt(t: Optional[torch.Tensor], name: str, dtype=None, allow_empty=False):
    """Optional device buffers (workspace, dev_error): the kernels write them,
    so a host tensor here would be a host address on the device."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor or None" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.numel() == 0 and not allow_empty:
        raise ValueError("%s must not be empty" % name)


try:  # NVTX ranges name the library calls on profiler timelines
    from torch.cuda import nvtx as _nvtx
except Exception:  # pragma: no cover
    _nvtx = None


class _Range:
    """NVTX range around one library call; a no-op where NVTX is missing
    (it never raises)."""

    def __init__(self, name: str):
        self.name = name
        self.pushed = False

    def __enter__(self):
        if _nvtx is not None:
            try:
                _nvtx.range_push(self.name)
                self.pushed = True
            except Exception:
                pass
        return self

    def __exit__(self, *exc):
        if self.pushed:
            try:
                _nvtx.range_pop()
            except Exception:
                pass
        return False


def _check(st: int, where: str):
    if st != 0:
        raise DCPError(st, where)


def _need(t: torch.Tensor, name: str, dtype, contiguous=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if contiguous and not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _decode_geometry(q, kv_cache, block_table, seq_lens, query_start_loc, O_part, lse_part, D: int,
                     local: bool = False):
    """Validate the decode arguments both decode entry points share and
    return (B, T, H).  Every size the kernels index by is checked here,
    because the C ABI receives bare pointers: a short block table or a
    flattened cache would otherwise be read past its end on the device.
    Shapes are checked before devices, so the checks run on any host."""
    kv_dt = torch.uint8 if isinstance(kv_cache, torch.Tensor) and kv_cache.dtype == torch.uint8 else torch.bfloat16
    o_dt = torch.bfloat16 if isinstance(O_part, torch.Tensor) and O_part.dtype == torch.bfloat16 else torch.float32
    args = (("q", q, torch.bfloat16, False), ("kv_cache", kv_cache, kv_dt, True),
            ("block_table", block_table, torch.int32, False), ("seq_lens", seq_lens, torch.int32, True),
            ("query_start_loc", query_start_loc, torch.int32, True), ("O_part", O_part, o_dt, True),
            ("lse_part", lse_part, torch.float32, True))
    for name, t, dtype, _ in args:
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a torch.Tensor" % name)
        if t.dtype != dtype:
            raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if q.dim() != 3 or q.shape[2] != KV_DIM or q.stride(2) != 1 or q.stride(1) != KV_DIM:
        raise ValueError("q must be [T, H, 576] with contiguous heads")
    if kv_cache.dim() != 3 or kv_cache.shape[2] != KV_DIM:
        raise ValueError("kv_cache must be [num_blocks, block_size, 576]")
    if local:
        if block_table.dim() != 3 or block_table.stride(2) != 1 or block_table.shape[0] != D:
            raise ValueError("block_table must be [D, B, W] with unit column stride")
    elif block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [B, W] with unit column stride")
    if seq_lens.dim() != 1 or query_start_loc.dim() != 1:
        raise ValueError("seq_lens and query_start_loc must be 1-D")
    T, H = q.shape[0], q.shape[1]
    B = seq_lens.shape[0]
    if query_start_loc.shape[0] != B + 1 or block_table.shape[-2] != B:
        raise ValueError("seq_lens [B], query_start_loc [B + 1] and block_table [.., B, W] disagree on B")
    if tuple(O_part.shape) != (D, T, H, LATENT_DIM) or tuple(lse_part.shape) != (D, T, H):
        raise ValueError("O_part must be [D, T, H, 512] and lse_part [D, T, H]")
    for name, t, dtype, contiguous in args:
        _need(t, name, dtype, contiguous=contiguous)
    return B, T, H


# ----------------------------------------------------------------------------
# entry points with the C names
# ----------------------------------------------------------------------------
def dcp_version() -> int:
    return lib().dcp_version()


def dcp_status_str(status: int) -> str:
    return lib().dcp_status_str(status).decode()


def dcp_shard_of(pos: int, D: int, interleave: int) -> int:
    return lib().dcp_shard_of(pos, D, interleave)


def dcp_local_len(L: int, d: int, D: int, interleave: int) -> int:
    return lib().dcp_local_len(L, d, D, interleave)


def dcp_decode_workspace_size(B: int, T: int, H: int, D: int, max_seq_len: int, max_q_len: int) -> int:
    n = lib().dcp_decode_workspace_size(B, T, H, D, max_seq_len, max_q_len)
    if n == ctypes.c_size_t(-1).value:
        raise DCPError(1, "dcp_decode_workspace_size")
    return n


def dcp_decode_kernel_launches(B: int, T: int, H: int, D: int, interleave: int, max_seq_len: int,
                               max_q_len: int, workspace_bytes: int) -> int:
    n = lib().dcp_decode_kernel_launches(B, T, H, D, interleave, max_seq_len, max_q_len, workspace_bytes)
    if n < 0:
        raise DCPError(1, "dcp_decode_kernel_launches")
    return n


def dcp_mla_decode_partial(q, kv_cache, block_table, seq_lens, query_start_loc, O_part, lse_part, *,
                           D: int, interleave: int, scale: float, max_seq_len: int, max_q_len: int,
                           workspace: Optional[torch.Tensor] = None, dev_error: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    """q bf16 [T, H, 576] (rows may be strided), kv_cache bf16 [NB, bs, 576],
    block_table int32 [B, W] (rows may be strided), seq_lens int32 [B],
    query_start_loc int32 [B + 1]; writes O_part fp32 [D, T, H, 512] and
    lse_part fp32 [D, T, H]."""
    B, T, H = _decode_geometry(q, kv_cache, block_table, seq_lens, query_start_loc, O_part, lse_part, D)
    _need_opt(workspace, "workspace", allow_empty=True)
    if workspace is not None and workspace.numel() == 0:
        workspace = None
    _need_opt(dev_error, "dev_error", torch.int32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _Range("dcp_mla_decode_partial"):
        st = lib().dcp_mla_decode_partial(
            _ptr(q), q.stride(0), _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1], _ptr(block_table),
            block_table.shape[1], block_table.stride(0), _ptr(seq_lens), _ptr(query_start_loc), B, T, H,
            max_seq_len, max_q_len, D, interleave, scale, _ptr(O_part), _ptr(lse_part), _ptr(workspace),
            ws_bytes, _ptr(dev_error), _stream(stream))
    _check(st, "dcp_mla_decode_partial")


def dcp_mla_decode_partial_local(q, kv_cache, block_table, seq_lens, query_start_loc, O_part, lse_part, *,
                                 D: int, interleave: int, scale: float, max_seq_len: int, max_q_len: int,
                                 shard_begin: int = 0, shard_count: Optional[int] = None,
                                 workspace: Optional[torch.Tensor] = None,
                                 dev_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """dcp_mla_decode_partial over per-shard tables for shards [shard_begin,
    shard_begin + shard_count) of D (default all): block_table int32
    [shard_count, B, W], shard d's j-th local token of request b in row
    block_table[d - shard_begin, b, j // bs] * bs + j % bs; O_part and
    lse_part have shard_count rows."""
    if shard_count is None:
        shard_count = D - shard_begin
    B, T, H = _decode_geometry(q, kv_cache, block_table, seq_lens, query_start_loc, O_part, lse_part,
                               shard_count, local=True)
    _need_opt(workspace, "workspace", allow_empty=True)
    if workspace is not None and workspace.numel() == 0:
        workspace = None
    _need_opt(dev_error, "dev_error", torch.int32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _Range("dcp_mla_decode_partial_local"):
        st = lib().dcp_mla_decode_partial_local(
            _ptr(q), q.stride(0), _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1], _ptr(block_table),
            block_table.shape[2], block_table.stride(1), block_table.stride(0), _ptr(seq_lens),
            _ptr(query_start_loc), B, T, H, max_seq_len, max_q_len, D, interleave, shard_begin, shard_count,
            scale, _ptr(O_part), _ptr(lse_part), _ptr(workspace), ws_bytes, _ptr(dev_error), _stream(stream))
    _check(st, "dcp_mla_decode_partial_local")


def dcp_mla_decode_partial_v2(q, kv_cache, block_table, seq_lens, query_start_loc, O_part, lse_part, *,
                              D: int, interleave: int, scale: float, max_seq_len: int, max_q_len: int,
                              kv_scale: Optional[torch.Tensor] = None, shard_begin: int = 0,
                              shard_count: Optional[int] = None, workspace: Optional[torch.Tensor] = None,
                              dev_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """The general decode: kv_cache bf16, or uint8 FP8 E4M3 codes with
    kv_scale fp32 [num_blocks, block_size]; block_table [B, W] or per-shard
    [shard_count, B, W]; O_part fp32 or bf16 [shard_count, T, H, 512]."""
    if shard_count is None:
        shard_count = D - shard_begin
    local = isinstance(block_table, torch.Tensor) and block_table.dim() == 3
    B, T, H = _decode_geometry(q, kv_cache, block_table, seq_lens, query_start_loc, O_part, lse_part,
                               shard_count, local=local)
    fp8 = kv_cache.dtype == torch.uint8
    if fp8:
        _need(kv_scale, "kv_scale", torch.float32)
        if tuple(kv_scale.shape) != tuple(kv_cache.shape[:2]):
            raise ValueError("kv_scale must be [num_blocks, block_size]")
    _need_opt(workspace, "workspace", allow_empty=True)
    if workspace is not None and workspace.numel() == 0:
        workspace = None
    _need_opt(dev_error, "dev_error", torch.int32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _Range("dcp_mla_decode_partial_v2"):
        st = lib().dcp_mla_decode_partial_v2(
            _ptr(q), q.stride(0), _ptr(kv_cache), KV_FP8_E4M3 if fp8 else KV_BF16, _ptr(kv_scale if fp8 else None),
            kv_cache.shape[0], kv_cache.shape[1], _ptr(block_table), block_table.shape[-1],
            block_table.stride(-2), 1 if local else 0, block_table.stride(0) if local else 0, shard_begin,
            shard_count, _ptr(seq_lens), _ptr(query_start_loc), B, T, H, max_seq_len, max_q_len, D, interleave,
            scale, _ptr(O_part), DTYPE_BF16 if O_part.dtype == torch.bfloat16 else DTYPE_F32, _ptr(lse_part),
            _ptr(workspace), ws_bytes, _ptr(dev_error), _stream(stream))
    _check(st, "dcp_mla_decode_partial_v2")


def dcp_mla_decode_partial_noalloc(q, kv_cache, block_table, seq_lens, query_start_loc, O_part, lse_part, *,
                                   D: int, interleave: int, scale: float, max_seq_len: int, max_q_len: int,
                                   dev_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """The decode for callers that cannot allocate device memory: same
    arguments and results as dcp_mla_decode_partial, but the split-KV scratch
    is a fixed 24 MiB array inside the library (shared by all calls, so calls
    that overlap on the GPU race; the first call on a device must precede
    any stream capture on it)."""
    B, T, H = _decode_geometry(q, kv_cache, block_table, seq_lens, query_start_loc, O_part, lse_part, D)
    _need_opt(dev_error, "dev_error", torch.int32)
    with _Range("dcp_mla_decode_partial_noalloc"):
        st = lib().dcp_mla_decode_partial_noalloc(
            _ptr(q), q.stride(0), _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1], _ptr(block_table),
            block_table.shape[1], block_table.stride(0), _ptr(seq_lens), _ptr(query_start_loc), B, T, H,
            max_seq_len, max_q_len, D, interleave, scale, _ptr(O_part), _ptr(lse_part), _ptr(dev_error),
            _stream(stream))
    _check(st, "dcp_mla_decode_partial_noalloc")


def dcp_lse_combine(O_part, lse_part, seq_lens, query_start_loc, out, out_lse, *, stream=None) -> None:
    """O_part fp32 [D, T, H, 512], lse_part fp32 [D, T, H] -> out [T, H, 512]
    (bf16 or fp32, by out.dtype) and out_lse fp32 [T, H].  Shapes are checked
    (on any host) before devices: the kernel reads D*T*H*512 floats of O_part
    and indexes query_start_loc up to B."""
    part_dt = torch.bfloat16 if isinstance(O_part, torch.Tensor) and O_part.dtype == torch.bfloat16 else torch.float32
    args = (("O_part", O_part, part_dt), ("lse_part", lse_part, torch.float32),
            ("seq_lens", seq_lens, torch.int32), ("query_start_loc", query_start_loc, torch.int32),
            ("out_lse", out_lse, torch.float32))
    for name, t, dtype in args:
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a torch.Tensor" % name)
        if t.dtype != dtype:
            raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not isinstance(out, torch.Tensor):
        raise TypeError("out must be a torch.Tensor")
    if out.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif out.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    if lse_part.dim() != 3:
        raise ValueError("lse_part must be [D, T, H]")
    D, T, H = lse_part.shape
    if tuple(O_part.shape) != (D, T, H, LATENT_DIM):
        raise ValueError("O_part must be [D, T, H, 512] with lse_part [D, T, H]")
    if tuple(out.shape) != (T, H, LATENT_DIM) or tuple(out_lse.shape) != (T, H):
        raise ValueError("out must be [T, H, 512] and out_lse [T, H]")
    if seq_lens.dim() != 1 or query_start_loc.dim() != 1:
        raise ValueError("seq_lens and query_start_loc must be 1-D")
    B = seq_lens.shape[0]
    if query_start_loc.shape[0] != B + 1:
        raise ValueError("query_start_loc must have B + 1 = %d entries" % (B + 1))
    for name, t, dtype in args:
        _need(t, name, dtype, contiguous=name != "out_lse")
    _need(out, "out", out.dtype)
    if not (out_lse.is_contiguous() or out_lse.data_ptr() == lse_part.data_ptr()):
        raise ValueError("out_lse must be contiguous")
    if part_dt == torch.float32:
        with _Range("dcp_lse_combine"):
            st = lib().dcp_lse_combine(_ptr(O_part), _ptr(lse_part), _ptr(seq_lens), _ptr(query_start_loc), B, T,
                                       H, D, _ptr(out), dt, _ptr(out_lse), _stream(stream))
        _check(st, "dcp_lse_combine")
    else:
        with _Range("dcp_lse_combine_v2"):
            st = lib().dcp_lse_combine_v2(_ptr(O_part), DTYPE_BF16, _ptr(lse_part), _ptr(seq_lens),
                                          _ptr(query_start_loc), B, T, H, D, _ptr(out), dt, _ptr(out_lse),
                                          _stream(stream))
        _check(st, "dcp_lse_combine_v2")


def dcp_decode_concat_cache(ql_nope, q_pe, kv_c, k_pe, slot_mapping, q_out, kv_cache, *,
                            dev_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """ql_nope bf16 [T, H, 512], q_pe bf16 [T, H, 64] (any token/head strides,
    unit element stride), kv_c bf16 [T, 512], k_pe bf16 [T, 64] (row strides
    allowed), slot_mapping int64 [T]; writes q_out bf16 [T, H, 576] and the
    rows of kv_cache bf16 [num_blocks, block_size, 576] at the non-negative
    slots."""
    for name, t, dt, dims, last in (("ql_nope", ql_nope, torch.bfloat16, 3, LATENT_DIM),
                                    ("q_pe", q_pe, torch.bfloat16, 3, ROPE_DIM),
                                    ("kv_c", kv_c, torch.bfloat16, 2, LATENT_DIM),
                                    ("k_pe", k_pe, torch.bfloat16, 2, ROPE_DIM),
                                    ("q_out", q_out, torch.bfloat16, 3, KV_DIM)):
        if not isinstance(t, torch.Tensor) or t.dtype != dt:
            raise TypeError("%s must be a %s tensor" % (name, dt))
        if t.dim() != dims or t.shape[-1] != last or t.stride(-1) != 1:
            raise ValueError("%s must have %d dims, last of size %d with unit stride" % (name, dims, last))
    T, H = ql_nope.shape[0], ql_nope.shape[1]
    if tuple(q_pe.shape[:2]) != (T, H) or kv_c.shape[0] != T or k_pe.shape[0] != T:
        raise ValueError("ql_nope, q_pe, kv_c and k_pe disagree on T or H")
    if tuple(q_out.shape[:2]) != (T, H) or q_out.stride(1) != KV_DIM:
        raise ValueError("q_out must be [T, H, 576] with dense heads")
    if not isinstance(slot_mapping, torch.Tensor) or slot_mapping.dtype != torch.int64 or \
            tuple(slot_mapping.shape) != (T,):
        raise ValueError("slot_mapping must be an int64 [T] tensor")
    if not isinstance(kv_cache, torch.Tensor) or kv_cache.dtype != torch.bfloat16 or kv_cache.dim() != 3 or \
            kv_cache.shape[2] != KV_DIM:
        raise ValueError("kv_cache must be bf16 [num_blocks, block_size, 576]")
    for name, t in (("ql_nope", ql_nope), ("q_pe", q_pe), ("kv_c", kv_c), ("k_pe", k_pe), ("q_out", q_out)):
        _need(t, name, torch.bfloat16, contiguous=False)
    _need(slot_mapping, "slot_mapping", torch.int64)
    _need(kv_cache, "kv_cache", torch.bfloat16)
    _need_opt(dev_error, "dev_error", torch.int32)
    with _Range("dcp_decode_concat_cache"):
        st = lib().dcp_decode_concat_cache(
            _ptr(ql_nope), ql_nope.stride(0), ql_nope.stride(1), _ptr(q_pe), q_pe.stride(0), q_pe.stride(1),
            _ptr(kv_c), kv_c.stride(0), _ptr(k_pe), k_pe.stride(0), _ptr(slot_mapping), T, H, _ptr(q_out),
            q_out.stride(0), _ptr(kv_cache), kv_cache.shape[0] * kv_cache.shape[1], _ptr(dev_error),
            _stream(stream))
    _check(st, "dcp_decode_concat_cache")


# ----------------------------------------------------------------------------
# allocating conveniences
# ----------------------------------------------------------------------------
def decode_workspace(B: int, T: int, H: int, D: int, max_seq_len: int, max_q_len: int,
                     device=None) -> Optional[torch.Tensor]:
    n = dcp_decode_workspace_size(B, T, H, D, max_seq_len, max_q_len)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def decode_partial(q, kv_cache, block_table, seq_lens, query_start_loc, D: int, interleave: int,
                   scale: float, max_seq_len: Optional[int] = None, max_q_len: Optional[int] = None,
                   dev_error: Optional[torch.Tensor] = None, stream=None, kv_scale: Optional[torch.Tensor] = None,
                   out_dtype=torch.float32):
    """Allocating form: returns (O_part fp32 [D, T, H, 512], lse_part fp32 [D, T, H]).
    A 3-D block_table [D, B, W] selects the per-shard layout
    (dcp_mla_decode_partial_local).

    ``max_seq_len``/``max_q_len`` default to the bounds implied by the table
    width and the row count (no device->host copy)."""
    T, H = q.shape[0], q.shape[1]
    B = seq_lens.shape[0]
    local = block_table.dim() == 3
    if max_seq_len is None:
        max_seq_len = block_table.shape[-1] * kv_cache.shape[1] * (D if local else 1)
    if max_q_len is None:
        max_q_len = max(1, T)
    O = torch.empty((D, T, H, LATENT_DIM), dtype=out_dtype, device=q.device)
    lse = torch.empty((D, T, H), dtype=torch.float32, device=q.device)
    ws = decode_workspace(B, T, H, D, max_seq_len, max_q_len, q.device)
    if kv_cache.dtype == torch.uint8 or out_dtype != torch.float32:
        dcp_mla_decode_partial_v2(q, kv_cache, block_table, seq_lens, query_start_loc, O, lse, D=D,
                                  interleave=interleave, scale=scale, max_seq_len=max_seq_len, max_q_len=max_q_len,
                                  kv_scale=kv_scale, workspace=ws, dev_error=dev_error, stream=stream)
        return O, lse
    entry = dcp_mla_decode_partial_local if local else dcp_mla_decode_partial
    entry(q, kv_cache, block_table, seq_lens, query_start_loc, O, lse, D=D, interleave=interleave, scale=scale,
          max_seq_len=max_seq_len, max_q_len=max_q_len, workspace=ws, dev_error=dev_error, stream=stream)
    return O, lse


def lse_combine(O_part, lse_part, seq_lens, query_start_loc, out_dtype=torch.bfloat16, stream=None):
    """Allocating form: returns (out [T, H, 512] of out_dtype, out_lse fp32 [T, H])."""
    D, T, H = lse_part.shape
    out = torch.empty((T, H, LATENT_DIM), dtype=out_dtype, device=O_part.device)
    out_lse = torch.empty((T, H), dtype=torch.float32, device=O_part.device)
    dcp_lse_combine(O_part, lse_part, seq_lens, query_start_loc, out, out_lse, stream=stream)
    return out, out_lse


def decode_concat_cache(ql_nope, q_pe, kv_c, k_pe, slot_mapping, kv_cache, dev_error=None, stream=None):
    """Allocating form: returns the decode query q bf16 [T, H, 576]; writes
    the step's latent rows into kv_cache in place."""
    T, H = ql_nope.shape[0], ql_nope.shape[1]
    q = torch.empty((T, H, KV_DIM), dtype=torch.bfloat16, device=ql_nope.device)
    dcp_decode_concat_cache(ql_nope, q_pe, kv_c, k_pe, slot_mapping, q, kv_cache, dev_error=dev_error,
                            stream=stream)
    return q
