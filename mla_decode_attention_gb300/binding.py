"""ctypes binding of ``libmla_decode.so`` (declared in include/mla_decode.h).

Argument marshalling only: every function takes torch tensors (device memory
for the device entry points), checks dtypes and contiguity, and passes raw
pointers and sizes to the C function of the same name.  A non-zero status
raises ``MlaError``.  There is no fallback: if the library is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmla_decode.so")

MLA_KV_BF16 = 0
MLA_KV_FP8_656 = 1
MLA_KV_FP8_528 = 2
MLA_DEVERR_BAD_PAGE = 1
MLA_DEVERR_BAD_INDEX = 2
MLA_DEVERR_TIMEOUT = 4
MLA_DEVERR_METADATA = 8

META_HEADER_WORDS = 16
META_PART_WORDS = 8
META_SEQ_WORDS = 8

_c_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_f = ctypes.c_float
_sz = ctypes.c_size_t

_SIGS = {
    "mla_status_string": (ctypes.c_char_p, [_i]),
    "mla_last_error": (ctypes.c_char_p, []),
    "mla_num_sm_parts": (_i, [_i, _i, ctypes.POINTER(_i)]),
    "mla_metadata_size": (_i, [_i, _i, _i, ctypes.POINTER(_sz)]),
    "mla_get_metadata": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "mla_get_metadata_host": (_i, [_vp, _i, _i, _i, _i, _i, _vp]),
    "mla_workspace_size": (_i, [_i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "mla_decode": (_i, [_vp, _vp, _i, _i64, _vp, _i64, _vp, _i, _i, _i, _f, _i, _vp, _i, _vp,
                        _vp, _vp, _vp, _vp]),
    "mla_decode_splitkv": (_i, [_vp, _vp, _i, _i64, _vp, _i64, _vp, _i, _i, _i, _f, _i, _vp, _i,
                                _vp, _vp, _vp, _vp, _vp]),
    "mla_decode_noalloc": (_i, [_vp, _vp, _i, _i64, _vp, _i64, _vp, _i, _i, _i, _f, _i, _vp, _vp,
                                _vp, _vp]),
    "mla_sparse_decode": (_i, [_vp, _vp, _i64, _vp, _i, _i, _i, _i, _f, _vp, _vp, _i, _vp, _vp,
                               _vp, _vp, _vp]),
    "mla_sparse_decode_splitkv": (_i, [_vp, _vp, _i64, _vp, _i, _i, _i, _i, _f, _vp, _vp, _i, _vp,
                                       _vp, _vp, _vp, _vp]),
    "mla_sparse_prefill": (_i, [_vp, _vp, _i64, _vp, _i, _i, _i, _f, _vp, _vp, _i, _vp, _vp, _vp,
                                _vp, _vp]),
    "mla_combine": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "mla_check_wait_timeout": (_i, [_vp, _vp]),
}

_lib = None


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = lib().mla_last_error().decode() if status in (-2, -5) else ""
        super().__init__(f"{fn} failed with status {status}: {status_string(status)}"
                         + (f" [{detail}]" if detail else ""))


def lib() -> ctypes.CDLL:
    """Loads the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().mla_status_string(status).decode()


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MlaError(fn, status)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ---------------------------------------------------------------- sizes

def mla_num_sm_parts(device: int, h_q: int) -> int:
    n = _i()
    _check("mla_num_sm_parts", lib().mla_num_sm_parts(device, h_q, ctypes.byref(n)))
    return n.value


def mla_metadata_size(batch: int, s_q: int, num_sm_parts: int) -> int:
    n = _sz()
    _check("mla_metadata_size", lib().mla_metadata_size(batch, s_q, num_sm_parts, ctypes.byref(n)))
    return n.value


def mla_workspace_size(batch: int, s_q: int, h_q: int, num_sm_parts: int) -> int:
    n = _sz()
    _check("mla_workspace_size",
           lib().mla_workspace_size(batch, s_q, h_q, num_sm_parts, ctypes.byref(n)))
    return n.value


# ---------------------------------------------------------------- schedule

def mla_get_metadata(cache_seqlens: Optional[torch.Tensor], batch: int, s_q: int, causal: bool,
                     topk: int, num_sm_parts: int, metadata: torch.Tensor, stream=None) -> None:
    if cache_seqlens is not None:
        _dev(cache_seqlens, torch.int32, "cache_seqlens")
    _dev(metadata, torch.int32, "metadata")
    _check("mla_get_metadata",
           lib().mla_get_metadata(_ptr(cache_seqlens), batch, s_q, int(bool(causal)), topk,
                                  num_sm_parts, _ptr(metadata), _stream(stream)))


def mla_get_metadata_host(cache_seqlens, batch: int, s_q: int, causal: bool, topk: int,
                          num_sm_parts: int) -> np.ndarray:
    """Host mirror of the schedule: returns the metadata words (int32)."""
    words = mla_metadata_size(batch, s_q, num_sm_parts) // 4
    out = np.zeros(words, dtype=np.int32)
    sl = None
    if cache_seqlens is not None:
        sl = np.ascontiguousarray(np.asarray(cache_seqlens, dtype=np.int32))
    _check("mla_get_metadata_host",
           lib().mla_get_metadata_host(None if sl is None else sl.ctypes.data, batch, s_q,
                                       int(bool(causal)), topk, num_sm_parts, out.ctypes.data))
    return out


# ---------------------------------------------------------------- decode

# query width and bytes per cached token of each cache format
_FORMATS = {MLA_KV_BF16: (576, None), MLA_KV_FP8_656: (576, 656), MLA_KV_FP8_528: (512, 528)}


def _check_format(q, kv_cache, kv_format):
    if kv_format not in _FORMATS:
        raise ValueError(f"unknown kv_format {kv_format}")
    d_qk, token_bytes = _FORMATS[kv_format]
    _dev(kv_cache, torch.bfloat16 if kv_format == MLA_KV_BF16 else torch.uint8, "kv_cache")
    if q.shape[-1] != d_qk or (token_bytes is not None and kv_cache.shape[-1] != token_bytes):
        raise ValueError(f"kv_format {kv_format} needs q [..., {d_qk}] and "
                         f"kv_cache [..., {token_bytes or 576}]")


def _decode_call(name, q, kv_cache, kv_format, block_table, cache_seqlens, softmax_scale,
                 causal, metadata, num_sm_parts, workspace, out, lse, err, stream):
    _dev(q, torch.bfloat16, "q")
    _check_format(q, kv_cache, kv_format)
    _dev(cache_seqlens, torch.int32, "cache_seqlens")
    _dev(metadata, torch.int32, "metadata")
    _dev(out, torch.bfloat16, "out")
    _dev(lse, torch.float32, "lse")
    if not block_table.is_cuda or block_table.dtype != torch.int32 or block_table.stride(1) != 1:
        raise ValueError("block_table must be a CUDA int32 tensor with unit column stride")
    if err is not None:
        _dev(err, torch.int32, "err")
    b, s_q, h, d = q.shape
    _check(name, getattr(lib(), name)(
        _ptr(q), _ptr(kv_cache), kv_format, kv_cache.shape[0], _ptr(block_table),
        block_table.stride(0), _ptr(cache_seqlens), b, s_q, h, float(softmax_scale),
        int(bool(causal)), _ptr(metadata), num_sm_parts, _ptr(workspace), _ptr(out), _ptr(lse),
        _ptr(err), _stream(stream)))


def mla_decode(q: torch.Tensor, kv_cache: torch.Tensor, kv_format: int,
               block_table: torch.Tensor, cache_seqlens: torch.Tensor, softmax_scale: float,
               causal: bool, metadata: torch.Tensor, num_sm_parts: int,
               workspace: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
               err: Optional[torch.Tensor] = None, stream=None) -> None:
    """q [b, s_q, h, 576] bf16; kv_cache [pages, 64, 576] bf16 (MLA_KV_BF16),
    [pages, 64, 656] uint8 (MLA_KV_FP8_656) or, with q [b, s_q, h, 512],
    [pages, 64, 528] uint8 (MLA_KV_FP8_528, V4.1); block_table [b, max_pages]
    int32; cache_seqlens [b] int32; out [b, s_q, h, 512] bf16; lse [b, h, s_q]
    fp32."""
    _decode_call("mla_decode", q, kv_cache, kv_format, block_table, cache_seqlens,
                 softmax_scale, causal, metadata, num_sm_parts, workspace, out, lse, err, stream)


def mla_decode_splitkv(q, kv_cache, kv_format, block_table, cache_seqlens, softmax_scale,
                       causal, metadata, num_sm_parts, workspace, out, lse, err=None,
                       stream=None) -> None:
    """The split kernel of mla_decode alone (partials need mla_combine)."""
    _decode_call("mla_decode_splitkv", q, kv_cache, kv_format, block_table, cache_seqlens,
                 softmax_scale, causal, metadata, num_sm_parts, workspace, out, lse, err, stream)


def mla_decode_noalloc(q: torch.Tensor, kv_cache: torch.Tensor, kv_format: int,
                       block_table: torch.Tensor, cache_seqlens: torch.Tensor,
                       softmax_scale: float, causal: bool, out: torch.Tensor, lse: torch.Tensor,
                       err: Optional[torch.Tensor] = None, stream=None) -> None:
    """mla_decode with the schedule and split workspace in the library's fixed
    device scratch array: the caller passes only inputs and outputs.  Calls
    sharing that array must not overlap on the GPU."""
    _dev(q, torch.bfloat16, "q")
    _check_format(q, kv_cache, kv_format)
    _dev(cache_seqlens, torch.int32, "cache_seqlens")
    _dev(out, torch.bfloat16, "out")
    _dev(lse, torch.float32, "lse")
    if not block_table.is_cuda or block_table.dtype != torch.int32 or block_table.stride(1) != 1:
        raise ValueError("block_table must be a CUDA int32 tensor with unit column stride")
    if err is not None:
        _dev(err, torch.int32, "err")
    b, s_q, h, d = q.shape
    _check("mla_decode_noalloc", lib().mla_decode_noalloc(
        _ptr(q), _ptr(kv_cache), kv_format, kv_cache.shape[0], _ptr(block_table),
        block_table.stride(0), _ptr(cache_seqlens), b, s_q, h, float(softmax_scale),
        int(bool(causal)), _ptr(out), _ptr(lse), _ptr(err), _stream(stream)))


def _sparse_call(name, q: torch.Tensor, kv: torch.Tensor, indices: torch.Tensor,
                 softmax_scale: float, metadata: torch.Tensor, num_sm_parts: int,
                 workspace: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
                 err: Optional[torch.Tensor] = None, stream=None,
                 attn_sink: Optional[torch.Tensor] = None) -> None:
    _dev(q, torch.bfloat16, "q")
    if attn_sink is not None:
        _dev(attn_sink, torch.float32, "attn_sink")
        if attn_sink.numel() != q.shape[2]:
            raise ValueError("attn_sink must hold one value per query head")
    _dev(kv, torch.bfloat16, "kv")
    _dev(indices, torch.int32, "indices")
    _dev(metadata, torch.int32, "metadata")
    _dev(out, torch.bfloat16, "out")
    _dev(lse, torch.float32, "lse")
    if err is not None:
        _dev(err, torch.int32, "err")
    b, s_q, h, d = q.shape
    topk = indices.shape[-1]
    _check(name,
           getattr(lib(), name)(_ptr(q), _ptr(kv), kv.shape[0], _ptr(indices), topk, b, s_q,
                                h, float(softmax_scale), _ptr(attn_sink), _ptr(metadata), num_sm_parts,
                                _ptr(workspace), _ptr(out), _ptr(lse), _ptr(err),
                                _stream(stream)))


def mla_sparse_decode(q, kv, indices, softmax_scale, metadata, num_sm_parts, workspace, out, lse,
                      err=None, stream=None, attn_sink=None) -> None:
    """q [b, s_q, h, 576] bf16; kv [s_kv, 576] bf16; indices [b, s_q, topk] int32;
    attn_sink optional [h] float32.  A per-token topk_length goes to
    mla_get_metadata in place of cache_seqlens."""
    _sparse_call("mla_sparse_decode", q, kv, indices, softmax_scale, metadata, num_sm_parts,
                 workspace, out, lse, err, stream, attn_sink)


def mla_sparse_prefill(q, kv, indices, softmax_scale, metadata, num_sm_parts, workspace, out, lse,
                       err=None, stream=None, attn_sink=None) -> None:
    """DSA sparse prefill: q [s_q, h, 576] bf16; kv [s_kv, 576] or [s_kv, 1, 576]
    bf16; indices [s_q, topk] or [s_q, 1, topk] int32; out [s_q, h, 512] bf16;
    lse [s_q, h] float32.  metadata from mla_get_metadata(topk_length, s_q, 1,
    False, topk, ...) (each query token a request of one token)."""
    _dev(q, torch.bfloat16, "q")
    if attn_sink is not None:
        _dev(attn_sink, torch.float32, "attn_sink")
        if attn_sink.numel() != q.shape[1]:
            raise ValueError("attn_sink must hold one value per query head")
    _dev(kv, torch.bfloat16, "kv")
    _dev(indices, torch.int32, "indices")
    _dev(metadata, torch.int32, "metadata")
    _dev(out, torch.bfloat16, "out")
    _dev(lse, torch.float32, "lse")
    if err is not None:
        _dev(err, torch.int32, "err")
    if q.dim() != 3 or kv.shape[-1] != q.shape[-1] or (kv.dim() == 3 and kv.shape[1] != 1):
        raise ValueError("q must be [s_q, h, 576] and kv [s_kv, 576] or [s_kv, 1, 576]")
    s_q, h, _ = q.shape
    topk = indices.shape[-1]
    if indices.numel() != s_q * topk:
        raise ValueError("indices must be [s_q, topk] or [s_q, 1, topk]")
    _check("mla_sparse_prefill",
           lib().mla_sparse_prefill(_ptr(q), _ptr(kv), kv.shape[0], _ptr(indices), topk, s_q, h,
                                    float(softmax_scale), _ptr(attn_sink), _ptr(metadata), num_sm_parts,
                                    _ptr(workspace), _ptr(out), _ptr(lse), _ptr(err), _stream(stream)))


def mla_sparse_decode_splitkv(q, kv, indices, softmax_scale, metadata, num_sm_parts, workspace,
                              out, lse, err=None, stream=None, attn_sink=None) -> None:
    """The split kernel of mla_sparse_decode alone (partials need mla_combine)."""
    _sparse_call("mla_sparse_decode_splitkv", q, kv, indices, softmax_scale, metadata,
                 num_sm_parts, workspace, out, lse, err, stream, attn_sink)


def mla_combine(metadata: torch.Tensor, batch: int, s_q: int, h_q: int, num_sm_parts: int,
                workspace: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
                stream=None, attn_sink: Optional[torch.Tensor] = None) -> None:
    if attn_sink is not None:
        _dev(attn_sink, torch.float32, "attn_sink")
    _check("mla_combine",
           lib().mla_combine(_ptr(metadata), batch, s_q, h_q, num_sm_parts, _ptr(workspace),
                             _ptr(attn_sink), _ptr(out), _ptr(lse), _stream(stream)))


def mla_check_wait_timeout(err: torch.Tensor, stream=None) -> None:
    """Runs the library's bounded wait on a barrier nothing completes; the
    kernel ORs MLA_DEVERR_TIMEOUT into err (uint32 device word) after ~2 s."""
    _dev(err, torch.int32, "err")
    _check("mla_check_wait_timeout", lib().mla_check_wait_timeout(_ptr(err), _stream(stream)))


# ---------------------------------------------------------------- convenience

class DecodeBuffers:
    """Device buffers for one decode shape: metadata, workspace, out, lse, err.

    Allocation happens here (through torch), never inside the library.
    """

    def __init__(self, batch: int, s_q: int, h_q: int, device="cuda", num_sm_parts=None):
        dev = torch.device(device)
        idx = dev.index if dev.index is not None else torch.cuda.current_device()
        self.num_sm_parts = num_sm_parts or mla_num_sm_parts(idx, h_q)
        self.batch, self.s_q, self.h_q = batch, s_q, h_q
        mbytes = mla_metadata_size(batch, s_q, self.num_sm_parts)
        wbytes = mla_workspace_size(batch, s_q, h_q, self.num_sm_parts)
        self.metadata = torch.zeros(mbytes // 4, dtype=torch.int32, device=dev)
        self.workspace = torch.empty(wbytes // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty(batch, s_q, h_q, 512, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(batch, h_q, s_q, dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
