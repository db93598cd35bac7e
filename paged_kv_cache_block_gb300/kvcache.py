"""Python binding of libpagedkv.so (the C ABI in include/pagedkv.h).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.  PyTorch
supplies device memory and the current stream.  Importing this module loads the library and
raises if it has not been built (``python -m paged_kv_cache_block_gb300.build``); there is no
fallback implementation.

Same names as the C ABI:
    compute_slot_mapping(...)        kv_compute_slot_mapping
    reshape_and_cache(...)           kv_reshape_and_cache
    paged_attention_workspace_size() kv_paged_attention_workspace_size
    paged_attention_decode(...)      kv_paged_attention_decode
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

KV_F16, KV_BF16, KV_FP8_E4M3 = 0, 1, 2
KV_DERR_BAD_BLOCK, KV_DERR_BAD_SLOT, KV_DERR_PAST_TABLE, KV_DERR_TIMEOUT, KV_DERR_BAD_LEN = 1, 2, 4, 8, 16
SIZE_MAX = (1 << 64) - 1

LIB_PATH = _build.LIB


class KVError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{_STATUS.get(status, status)}: {detail}")
        self.status = status


_STATUS = {0: "KV_OK", 1: "KV_ERR_INVALID_ARG", 2: "KV_ERR_UNSUPPORTED", 3: "KV_ERR_CUDA",
           4: "KV_ERR_WORKSPACE"}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -m paged_kv_cache_block_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.kv_compute_slot_mapping.argtypes = [P, i64, i32, i32, P, P, i32, i32, i32, P, P, P]
    lib.kv_compute_slot_mapping.restype = i32
    lib.kv_reshape_and_cache.argtypes = [P, P, i32, i64, i64, i32, i32, i32, P, P, P, i32, i32, i32,
                                         f32, f32, P, P]
    lib.kv_reshape_and_cache.restype = i32
    lib.kv_paged_attention_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32]
    lib.kv_paged_attention_workspace_size.restype = sz
    lib.kv_paged_attention_decode.argtypes = [P, i32, i32, i32, i32, P, P, i32, i32, i32, i32, i32, P,
                                              i64, i32, P, i32, f32, i32, f32, f32, i32, P, sz, P, P,
                                              P, P]
    lib.kv_paged_attention_decode.restype = i32
    lib.kv_decode_step.argtypes = [P, i64, i32, P, P, P, P, P, i64, i64, P, i32, i32, i32, i32, P, P,
                                   i32, i32, i32, i32, i32, P, i32, f32, i32, f32, f32, i32, P, sz, P,
                                   P, P, P]
    lib.kv_decode_step.restype = i32
    lib.kv_paged_attention_decode_noalloc.argtypes = [P, i32, i32, i32, i32, P, P, i32, i32, i32, i32,
                                                      i32, P, i64, i32, P, i32, f32, i32, f32, f32,
                                                      i32, P, P, P, P]
    lib.kv_paged_attention_decode_noalloc.restype = i32
    lib.kv_status_string.argtypes = [i32]
    lib.kv_status_string.restype = ctypes.c_char_p
    lib.kv_last_error.argtypes = []
    lib.kv_last_error.restype = ctypes.c_char_p
    return lib


lib = _load()


def _check(status: int) -> None:
    if status != 0:
        raise KVError(status, lib.kv_last_error().decode())


def dtype_code(t: torch.dtype) -> int:
    if t == torch.float16:
        return KV_F16
    if t == torch.bfloat16:
        return KV_BF16
    if t in (torch.uint8, torch.float8_e4m3fn):
        return KV_FP8_E4M3
    raise TypeError(f"unsupported dtype {t}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def compute_slot_mapping(block_table: torch.Tensor, query_start_loc: torch.Tensor,
                         positions: torch.Tensor, block_size: int, num_blocks: int,
                         slot_mapping: Optional[torch.Tensor] = None,
                         d_err: Optional[torch.Tensor] = None, max_blocks_per_seq: Optional[int] = None,
                         stream=None) -> torch.Tensor:
    assert block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.stride(1) == 1
    assert query_start_loc.dtype == torch.int32 and positions.dtype == torch.int32
    T = positions.shape[0]
    if slot_mapping is None:
        slot_mapping = torch.empty(T, dtype=torch.int64, device=positions.device)
    _check(lib.kv_compute_slot_mapping(
        _ptr(block_table), block_table.stride(0), block_table.shape[0],
        block_table.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq,
        _ptr(query_start_loc), _ptr(positions), T, block_size, num_blocks, _ptr(slot_mapping),
        _ptr(d_err), _stream(stream)))
    return slot_mapping


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: float = 1.0,
                      v_scale: float = 1.0, d_err: Optional[torch.Tensor] = None, stream=None) -> None:
    """key/value [T, Hkv, D] (row stride = stride(0)); caches [NB, bs, Hkv, D]."""
    T, H, D = key.shape
    assert key.stride(2) == 1 and key.stride(1) == D and value.stride(2) == 1 and value.stride(1) == D
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    _check(lib.kv_reshape_and_cache(
        _ptr(key), _ptr(value), dtype_code(key.dtype), key.stride(0), value.stride(0), T, H, D,
        _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), dtype_code(k_cache.dtype), NB, bs,
        float(k_scale), float(v_scale), _ptr(d_err), _stream(stream)))


def paged_attention_workspace_size(num_seqs: int, q_len: int, num_q_heads: int, num_kv_heads: int,
                                   head_dim: int, block_size: int, cache_dtype: int,
                                   max_seq_len: int, window: int = 0, num_workers: int = 0) -> int:
    n = lib.kv_paged_attention_workspace_size(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim,
                                              block_size, cache_dtype, max_seq_len, window,
                                              num_workers)
    if n == SIZE_MAX:
        raise KVError(2, lib.kv_last_error().decode() or "invalid or unsupported sizes")
    return int(n)


def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                           q_len: int, scale: float, window: int = 0, k_scale: float = 1.0,
                           v_scale: float = 1.0, num_workers: int = 0,
                           workspace: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None, lse_out: Optional[torch.Tensor] = None,
                           d_err: Optional[torch.Tensor] = None, max_blocks_per_seq: Optional[int] = None,
                           stream=None) -> torch.Tensor:
    """q [B*q_len, Hq, D]; caches [NB, bs, Hkv, D]; block_table int32 [B, W]; seq_lens int32 [B]."""
    TQ, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    B = seq_lens.shape[0]
    assert TQ == B * q_len and q.is_contiguous() and block_table.stride(1) == 1
    cdt = dtype_code(k_cache.dtype)
    if out is None:
        out = torch.empty_like(q)
    need = paged_attention_workspace_size(B, q_len, Hq, Hkv, D, bs, cdt, max_seq_len, window,
                                          num_workers)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.kv_paged_attention_decode(
        _ptr(q), dtype_code(q.dtype), B, q_len, Hq, _ptr(k_cache), _ptr(v_cache), cdt, Hkv, D, bs, NB,
        _ptr(block_table), block_table.stride(0),
        block_table.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq,
        _ptr(seq_lens), max_seq_len, float(scale), window, float(k_scale), float(v_scale),
        num_workers, _ptr(workspace), ws_bytes, _ptr(out), _ptr(lse_out), _ptr(d_err),
        _stream(stream)))
    return out


def decode_step(block_table: torch.Tensor, query_start_loc: torch.Tensor, positions: torch.Tensor,
                key: torch.Tensor, value: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                v_cache: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, q_len: int,
                scale: float, window: int = 0, k_scale: float = 1.0, v_scale: float = 1.0,
                num_workers: int = 0, workspace: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, lse_out: Optional[torch.Tensor] = None,
                slot_mapping: Optional[torch.Tensor] = None, d_err: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """kv_decode_step: slot mapping, cache write and attention of one decode step, one launch."""
    TQ, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    B = seq_lens.shape[0]
    assert TQ == B * q_len and q.is_contiguous() and block_table.stride(1) == 1
    assert key.stride(2) == 1 and key.stride(1) == D and value.stride(2) == 1 and value.stride(1) == D
    cdt = dtype_code(k_cache.dtype)
    if out is None:
        out = torch.empty_like(q)
    need = paged_attention_workspace_size(B, q_len, Hq, Hkv, D, bs, cdt, max_seq_len, window,
                                          num_workers)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.kv_decode_step(
        _ptr(block_table), block_table.stride(0), block_table.shape[1], _ptr(query_start_loc),
        _ptr(positions), _ptr(slot_mapping), _ptr(key), _ptr(value), key.stride(0), value.stride(0),
        _ptr(q), dtype_code(q.dtype), B, q_len, Hq, _ptr(k_cache), _ptr(v_cache), cdt, Hkv, D, bs, NB,
        _ptr(seq_lens), max_seq_len, float(scale), window, float(k_scale), float(v_scale),
        num_workers, _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _ptr(lse_out), _ptr(d_err), _stream(stream)))
    return out


def paged_attention_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                   block_table: torch.Tensor, seq_lens: torch.Tensor,
                                   max_seq_len: int, q_len: int, scale: float, window: int = 0,
                                   k_scale: float = 1.0, v_scale: float = 1.0, num_workers: int = 0,
                                   out: Optional[torch.Tensor] = None,
                                   lse_out: Optional[torch.Tensor] = None,
                                   d_err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """kv_paged_attention_decode_noalloc: the same attention with the library's static scratch,
    for callers that cannot allocate device memory (pass ``out`` to allocate nothing here)."""
    TQ, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    B = seq_lens.shape[0]
    assert TQ == B * q_len and q.is_contiguous() and block_table.stride(1) == 1
    if out is None:
        out = torch.empty_like(q)
    _check(lib.kv_paged_attention_decode_noalloc(
        _ptr(q), dtype_code(q.dtype), B, q_len, Hq, _ptr(k_cache), _ptr(v_cache),
        dtype_code(k_cache.dtype), Hkv, D, bs, NB, _ptr(block_table), block_table.stride(0),
        block_table.shape[1], _ptr(seq_lens), max_seq_len, float(scale), window, float(k_scale),
        float(v_scale), num_workers, _ptr(out), _ptr(lse_out), _ptr(d_err), _stream(stream)))
    return out
