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
    decode_step(...)                 kv_decode_step
    paged_attention_prefill(...)     kv_paged_attention_prefill
    BlockManager                     kv_bm_* (host block manager, one object per handle)
    apply_block_updates(...)         kv_apply_block_updates
    reshape_and_cache_int4(...)      kv_reshape_and_cache_int4       (include/pagedkv_int4.h)
    paged_attention_decode_int4(...) kv_paged_attention_decode_int4
    decode_step_int4(...)            kv_decode_step_int4
    selftest_bounded_wait(...)       kv_selftest_bounded_wait         (include/pagedkv_selftest.h)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

KV_F16, KV_BF16, KV_FP8_E4M3, KV_INT4 = 0, 1, 2, 3
KV_DERR_BAD_BLOCK, KV_DERR_BAD_SLOT, KV_DERR_PAST_TABLE, KV_DERR_TIMEOUT, KV_DERR_BAD_LEN = 1, 2, 4, 8, 16
KV_DERR_BAD_UPDATE = 32
KV_OK, KV_ERR_INVALID_ARG, KV_ERR_UNSUPPORTED, KV_ERR_CUDA, KV_ERR_WORKSPACE, KV_ERR_OUT_OF_BLOCKS = range(6)
KV_MAX_ZERO_CACHES = 128
SIZE_MAX = (1 << 64) - 1

LIB_PATH = _build.LIB


class KVError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{_STATUS.get(status, status)}: {detail}")
        self.status = status


_STATUS = {0: "KV_OK", 1: "KV_ERR_INVALID_ARG", 2: "KV_ERR_UNSUPPORTED", 3: "KV_ERR_CUDA",
           4: "KV_ERR_WORKSPACE", 5: "KV_ERR_OUT_OF_BLOCKS"}


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
    lib.kv_paged_attention_plan_info.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, P]
    lib.kv_paged_attention_plan_info.restype = i32
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
    pi32 = ctypes.POINTER(i32)
    lib.kv_bm_create.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(P)]
    lib.kv_bm_create.restype = i32
    lib.kv_bm_destroy.argtypes = [P]
    lib.kv_bm_destroy.restype = None
    lib.kv_bm_allocate.argtypes = [P, i32, i32]
    lib.kv_bm_allocate.restype = i32
    lib.kv_bm_allocate_batch.argtypes = [P, P, P, i32, P]
    lib.kv_bm_allocate_batch.restype = i32
    lib.kv_bm_free.argtypes = [P, i32]
    lib.kv_bm_free.restype = i32
    lib.kv_bm_share_prefix.argtypes = [P, i32, i32, i32]
    lib.kv_bm_share_prefix.restype = i32
    lib.kv_bm_num_free_blocks.argtypes = [P]
    lib.kv_bm_num_free_blocks.restype = i32
    lib.kv_bm_ref_count.argtypes = [P, i32]
    lib.kv_bm_ref_count.restype = i32
    lib.kv_bm_row.argtypes = [P, i32, pi32, pi32, P, i32]
    lib.kv_bm_row.restype = i32
    lib.kv_bm_pending.argtypes = [P, pi32, pi32]
    lib.kv_bm_pending.restype = i32
    lib.kv_bm_flush.argtypes = [P, P, i32, pi32, P, i32, pi32]
    lib.kv_bm_flush.restype = i32
    lib.kv_paged_attention_prefill.argtypes = [P, i32, P, i32, i32, i32, i32, P, P, i32, i32, i32, i32,
                                               i32, P, i64, i32, P, i32, f32, i32, P, P, P, P]
    lib.kv_paged_attention_prefill.restype = i32
    lib.kv_apply_block_updates.argtypes = [P, i32, P, i64, i32, i32, P, i32, P, i32, i64, i32, P, P]
    lib.kv_apply_block_updates.restype = i32
    lib.kv_reshape_and_cache_int4.argtypes = [P, P, i32, i64, i64, i32, i32, i32, P, P, P, i32, i32, P, P,
                                              i32, P, P]
    lib.kv_reshape_and_cache_int4.restype = i32
    lib.kv_paged_attention_decode_int4.argtypes = [P, i32, i32, i32, i32, P, P, i32, i32, i32, i32, P, i64,
                                                   i32, P, i32, f32, i32, P, P, i32, i32, P, sz, P, P, P, P]
    lib.kv_paged_attention_decode_int4.restype = i32
    lib.kv_decode_step_int4.argtypes = [P, i64, i32, P, P, P, P, P, i64, i64, P, i32, i32, i32, i32, P, P,
                                        i32, i32, i32, i32, P, i32, f32, i32, P, P, i32, i32, P, sz, P, P,
                                        P, P]
    lib.kv_decode_step_int4.restype = i32
    lib.kv_selftest_bounded_wait.argtypes = [i32, P, P, P]
    lib.kv_selftest_bounded_wait.restype = i32
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


PLAN_FIELDS = ("stages", "stage_bytes", "heads_per_cta", "ctas", "threads", "rows_per_warp", "items",
               "workspace_bytes")


def paged_attention_plan_info(num_seqs: int, q_len: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                              block_size: int, cache_dtype: int, max_seq_len: int, window: int = 0,
                              num_workers: int = 0) -> dict:
    """The decode launch geometry for these sizes (kv_paged_attention_plan_info)."""
    info = (ctypes.c_int64 * 8)()
    _check(lib.kv_paged_attention_plan_info(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                            cache_dtype, max_seq_len, window, num_workers, info))
    return dict(zip(PLAN_FIELDS, list(info)))


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


def _int4_group(head_dim: int, k_scales: torch.Tensor, v_scales: torch.Tensor) -> int:
    assert k_scales.dtype == torch.float32 and v_scales.dtype == torch.float32
    assert k_scales.is_contiguous() and v_scales.is_contiguous() and k_scales.shape == v_scales.shape
    return head_dim // k_scales.shape[-1]


def reshape_and_cache_int4(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor,
                           k_cache: torch.Tensor, v_cache: torch.Tensor, k_scales: torch.Tensor,
                           v_scales: torch.Tensor, d_err: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    """key/value [T, Hkv, D] fp16/bf16; caches uint8 [NB, bs, Hkv, D/2]; scales float32
    [Hkv, D/group_size] (the group size follows from their shape)."""
    T, H, D = key.shape
    assert key.stride(2) == 1 and key.stride(1) == D and value.stride(2) == 1 and value.stride(1) == D
    assert k_cache.dtype == torch.uint8 and k_cache.shape[-1] * 2 == D
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    _check(lib.kv_reshape_and_cache_int4(
        _ptr(key), _ptr(value), dtype_code(key.dtype), key.stride(0), value.stride(0), T, H, D,
        _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), NB, bs, _ptr(k_scales), _ptr(v_scales),
        _int4_group(D, k_scales, v_scales), _ptr(d_err), _stream(stream)))


def paged_attention_decode_int4(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                                q_len: int, scale: float, k_scales: torch.Tensor, v_scales: torch.Tensor,
                                window: int = 0, num_workers: int = 0,
                                workspace: Optional[torch.Tensor] = None,
                                out: Optional[torch.Tensor] = None, lse_out: Optional[torch.Tensor] = None,
                                d_err: Optional[torch.Tensor] = None,
                                max_blocks_per_seq: Optional[int] = None, stream=None) -> torch.Tensor:
    """q [B*q_len, Hq, D]; caches uint8 [NB, bs, Hkv, D/2]; scales float32 [Hkv, D/group_size]."""
    TQ, Hq, D = q.shape
    NB, bs, Hkv, half = k_cache.shape
    B = seq_lens.shape[0]
    assert TQ == B * q_len and q.is_contiguous() and block_table.stride(1) == 1
    assert k_cache.dtype == torch.uint8 and half * 2 == D
    if out is None:
        out = torch.empty_like(q)
    need = paged_attention_workspace_size(B, q_len, Hq, Hkv, D, bs, KV_INT4, max_seq_len, window,
                                          num_workers)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.kv_paged_attention_decode_int4(
        _ptr(q), dtype_code(q.dtype), B, q_len, Hq, _ptr(k_cache), _ptr(v_cache), Hkv, D, bs, NB,
        _ptr(block_table), block_table.stride(0),
        block_table.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq,
        _ptr(seq_lens), max_seq_len, float(scale), window, _ptr(k_scales), _ptr(v_scales),
        _int4_group(D, k_scales, v_scales), num_workers, _ptr(workspace), ws_bytes, _ptr(out),
        _ptr(lse_out), _ptr(d_err), _stream(stream)))
    return out


def selftest_bounded_wait(limit_us: int, d_err: torch.Tensor, d_waited_us: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    """kv_selftest_bounded_wait: a kernel whose wait runs out after limit_us (sets
    KV_DERR_TIMEOUT in d_err, the waited microseconds in d_waited_us)."""
    assert d_err.dtype == torch.int32
    _check(lib.kv_selftest_bounded_wait(int(limit_us), _ptr(d_err), _ptr(d_waited_us), _stream(stream)))


def decode_step_int4(block_table: torch.Tensor, query_start_loc: torch.Tensor, positions: torch.Tensor,
                     key: torch.Tensor, value: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                     v_cache: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, q_len: int,
                     scale: float, k_scales: torch.Tensor, v_scales: torch.Tensor, window: int = 0,
                     num_workers: int = 0, workspace: Optional[torch.Tensor] = None,
                     out: Optional[torch.Tensor] = None, lse_out: Optional[torch.Tensor] = None,
                     slot_mapping: Optional[torch.Tensor] = None, d_err: Optional[torch.Tensor] = None,
                     stream=None) -> torch.Tensor:
    """kv_decode_step_int4: slot mapping, INT4 cache write and attention of one decode step."""
    TQ, Hq, D = q.shape
    NB, bs, Hkv, half = k_cache.shape
    B = seq_lens.shape[0]
    assert TQ == B * q_len and q.is_contiguous() and block_table.stride(1) == 1
    assert key.stride(2) == 1 and key.stride(1) == D and value.stride(2) == 1 and value.stride(1) == D
    assert k_cache.dtype == torch.uint8 and half * 2 == D
    if out is None:
        out = torch.empty_like(q)
    need = paged_attention_workspace_size(B, q_len, Hq, Hkv, D, bs, KV_INT4, max_seq_len, window,
                                          num_workers)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.kv_decode_step_int4(
        _ptr(block_table), block_table.stride(0), block_table.shape[1], _ptr(query_start_loc),
        _ptr(positions), _ptr(slot_mapping), _ptr(key), _ptr(value), key.stride(0), value.stride(0),
        _ptr(q), dtype_code(q.dtype), B, q_len, Hq, _ptr(k_cache), _ptr(v_cache), Hkv, D, bs, NB,
        _ptr(seq_lens), max_seq_len, float(scale), window, _ptr(k_scales), _ptr(v_scales),
        _int4_group(D, k_scales, v_scales), num_workers, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse_out), _ptr(d_err),
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


def paged_attention_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_table: torch.Tensor, seq_lens: torch.Tensor,
                            query_start_loc: torch.Tensor, max_seq_len: int, max_query_len: int,
                            scale: float, window: int = 0, out: Optional[torch.Tensor] = None,
                            lse_out: Optional[torch.Tensor] = None, d_err: Optional[torch.Tensor] = None,
                            max_blocks_per_seq: Optional[int] = None, stream=None) -> torch.Tensor:
    """kv_paged_attention_prefill: q [T, Hq, D] (rows of sequence b are query_start_loc[b] ..
    query_start_loc[b+1]-1, its last positions); caches [NB, bs, Hkv, D]; block_table int32
    [B, W]; seq_lens int32 [B] (including the new rows)."""
    T, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    B = seq_lens.shape[0]
    assert q.is_contiguous() and block_table.stride(1) == 1 and query_start_loc.numel() == B + 1
    if out is None:
        out = torch.empty_like(q)
    _check(lib.kv_paged_attention_prefill(
        _ptr(q), dtype_code(q.dtype), _ptr(query_start_loc), B, T, max_query_len, Hq, _ptr(k_cache),
        _ptr(v_cache), dtype_code(k_cache.dtype), Hkv, D, bs, NB, _ptr(block_table), block_table.stride(0),
        block_table.shape[1] if max_blocks_per_seq is None else max_blocks_per_seq, _ptr(seq_lens),
        max_seq_len, float(scale), window, _ptr(out), _ptr(lse_out), _ptr(d_err), _stream(stream)))
    return out


class BlockManager:
    """Host block manager (kv_bm_*): free pool, reference counts, block-table rows, prefix
    sharing, window release and staged table writes.  allocate / free / share_prefix return the
    C status (0 = OK, KV_ERR_OUT_OF_BLOCKS when the pool is short, KV_ERR_INVALID_ARG for a
    request the manager refuses) instead of raising, since a refusal is an ordinary scheduling
    outcome (kv_last_error() says why); the constructor, row and flush raise KVError."""

    def __init__(self, num_blocks: int, block_size: int, num_rows: int, max_blocks_per_row: int,
                 window: int = 0, zero_fill: bool = True):
        h = ctypes.c_void_p()
        _check(lib.kv_bm_create(num_blocks, block_size, num_rows, max_blocks_per_row, window,
                                int(bool(zero_fill)), ctypes.byref(h)))
        self._h = h
        self.num_blocks, self.block_size = num_blocks, block_size
        self.num_rows, self.max_blocks_per_row, self.window = num_rows, max_blocks_per_row, window

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            lib.kv_bm_destroy(h)
            self._h = None

    def allocate(self, row: int, num_new_tokens: int) -> int:
        return lib.kv_bm_allocate(self._h, row, num_new_tokens)

    def allocate_batch(self, rows, num_new_tokens):
        """kv_bm_allocate_batch over int32 host arrays; returns the per-row statuses."""
        import numpy as np
        r = np.ascontiguousarray(rows, dtype=np.int32)
        n = np.ascontiguousarray(num_new_tokens, dtype=np.int32)
        assert r.shape == n.shape
        st = np.empty(r.shape, dtype=np.int32)
        lib.kv_bm_allocate_batch(self._h, r.ctypes.data, n.ctypes.data, r.size, st.ctypes.data)
        return st

    def free(self, row: int) -> int:
        return lib.kv_bm_free(self._h, row)

    def share_prefix(self, dst_row: int, src_row: int, num_blocks: int) -> int:
        return lib.kv_bm_share_prefix(self._h, dst_row, src_row, num_blocks)

    def num_free_blocks(self) -> int:
        return lib.kv_bm_num_free_blocks(self._h)

    def ref_count(self, block: int) -> int:
        return lib.kv_bm_ref_count(self._h, block)

    def row(self, row: int):
        """(tokens, [physical id per logical block, -1 = released])."""
        import numpy as np
        t, n = ctypes.c_int32(), ctypes.c_int32()
        _check(lib.kv_bm_row(self._h, row, ctypes.byref(t), ctypes.byref(n), None, 0))
        out = np.empty(n.value, dtype=np.int32)
        _check(lib.kv_bm_row(self._h, row, ctypes.byref(t), ctypes.byref(n), out.ctypes.data, out.size))
        return t.value, out.tolist()

    def pending(self):
        u, z = ctypes.c_int32(), ctypes.c_int32()
        _check(lib.kv_bm_pending(self._h, ctypes.byref(u), ctypes.byref(z)))
        return u.value, z.value

    def flush(self, updates=None, zero_ids=None):
        """kv_bm_flush into host int32 arrays (numpy, or pinned torch tensors for an asynchronous
        copy; allocated here when None).  Returns (updates [n, 3], zero_ids [m]) views."""
        import numpy as np
        nu, nz = self.pending()
        if updates is None:
            updates = np.empty((max(nu, 1), 3), dtype=np.int32)
        if zero_ids is None:
            zero_ids = np.empty(max(nz, 1), dtype=np.int32)
        up_ptr = updates.data_ptr() if isinstance(updates, torch.Tensor) else updates.ctypes.data
        z_ptr = zero_ids.data_ptr() if isinstance(zero_ids, torch.Tensor) else zero_ids.ctypes.data
        cap_u = updates.numel() // 3 if isinstance(updates, torch.Tensor) else updates.size // 3
        cap_z = zero_ids.numel() if isinstance(zero_ids, torch.Tensor) else zero_ids.size
        a, b = ctypes.c_int32(), ctypes.c_int32()
        _check(lib.kv_bm_flush(self._h, up_ptr, cap_u, ctypes.byref(a), z_ptr, cap_z, ctypes.byref(b)))
        return updates.reshape(-1)[:3 * a.value].reshape(-1, 3), zero_ids.reshape(-1)[:b.value]


def apply_block_updates(updates: torch.Tensor, block_table: torch.Tensor, zero_ids: torch.Tensor,
                        caches, num_blocks: int, d_err: Optional[torch.Tensor] = None,
                        max_blocks_per_row: Optional[int] = None, stream=None) -> None:
    """kv_apply_block_updates: device int32 updates [n, 3] into block_table [rows, stride];
    zero every cache's block of each id in zero_ids (device int32 [m]).  caches: device tensors
    whose first axis is the block id (e.g. [NB, bs, Hkv, D] K and V of each layer)."""
    assert updates.dtype == torch.int32 and zero_ids.dtype == torch.int32
    assert block_table.dtype == torch.int32 and block_table.stride(1) == 1
    n_up = updates.numel() // 3
    n_zero = zero_ids.numel()
    ptrs = (ctypes.c_void_p * max(len(caches), 1))(*[c.data_ptr() for c in caches])
    block_bytes = 0
    if caches:
        c0 = caches[0]
        block_bytes = c0[0].numel() * c0.element_size()
        for c in caches:
            assert c.is_contiguous() and c.shape[0] == num_blocks
            assert c[0].numel() * c.element_size() == block_bytes
    _check(lib.kv_apply_block_updates(
        _ptr(updates) if n_up else None, n_up, _ptr(block_table), block_table.stride(0),
        block_table.shape[0], block_table.shape[1] if max_blocks_per_row is None else max_blocks_per_row,
        _ptr(zero_ids) if n_zero else None, n_zero, ptrs, len(caches), block_bytes, num_blocks,
        _ptr(d_err), _stream(stream)))
