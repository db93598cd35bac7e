"""CPU oracle for the paged KV cache decode path (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this package.
It wraps ``kv_oracle.c`` (plain C, fp64 accumulation, pthreads over (sequence, kv head)),
which is compiled here with gcc.  It shares no code with the CUDA library, and the library
never imports it.

Pins: every function here is checked against facts that do not come from the oracle itself
(worked examples printed on the pages, closed forms, library routines on special cases,
brute force on tiny inputs); see tests/test_oracle_pins.py.  The fp8 attention tolerance
(relative 2e-2 over each output tensor) is a reading of the specification, not a number the
pages give: that tolerance is "parity unpinned" by the pages.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkv_oracle.so")

# oracle-side dtype codes (its own numbering)
_DT = {"f16": 0, "bf16": 1, "e4m3": 2, "int4": 3}

_lib: Optional[ctypes.CDLL] = None


def build(force: bool = False) -> str:
    """Compile kv_oracle.c into libkv_oracle.so beside it (gcc, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
                               "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Temporarily route every oracle call through another build of kv_oracle.c (the tests
    use this to check that planted mistakes in the oracle make its pins fail)."""
    global _lib
    saved = _lib
    _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def compile_variant(source: str, out_path: str) -> str:
    """Compile C source text (a variant of kv_oracle.c) with the oracle's own flags."""
    src_path = out_path + ".c"
    with open(src_path, "w") as f:
        f.write(source)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
                           "-shared", "-fPIC", "-pthread", src_path, "-o", out_path, "-lm"])
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    lib.orc_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_f16_to_double.restype = f64
    lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_double.restype = f64
    lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_to_double.restype = f64
    lib.orc_e4m3_from_float.argtypes = [f32]
    lib.orc_e4m3_from_float.restype = ctypes.c_uint8
    lib.orc_slot_mapping.argtypes = [P, i64, i32, i32, P, P, i32, i32, i32, P]
    lib.orc_slot_mapping.restype = i32
    lib.orc_reshape_and_cache.argtypes = [P, P, i32, i64, i64, i32, i32, i32, P, P, P, i32,
                                          i32, i32, f32, f32]
    lib.orc_reshape_and_cache.restype = i32
    lib.orc_paged_attention.argtypes = [P, i32, i32, i32, i32, P, P, i32, i32, i32, i32, i32,
                                        P, i64, i32, P, f64, i32, f64, f64, P, i32, P, P, i32]
    lib.orc_paged_attention.restype = i32
    lib.orc_paged_attention_varlen.argtypes = [P, i32, i32, P, i32, P, P, i32, i32, i32, i32, i32,
                                               P, i64, i32, P, f64, i32, f64, f64, P, i32, P, P,
                                               i32]
    lib.orc_paged_attention_varlen.restype = i32
    lib.orc_int4_from_float.argtypes = [f32]
    lib.orc_int4_from_float.restype = ctypes.c_uint8
    lib.orc_int4_to_double.argtypes = [ctypes.c_uint8]
    lib.orc_int4_to_double.restype = f64
    lib.orc_reshape_and_cache_int4.argtypes = [P, P, i32, i64, i64, i32, i32, i32, P, P, P, i32, i32,
                                               P, P, i32]
    lib.orc_reshape_and_cache_int4.restype = i32
    lib.orc_paged_attention_int4.argtypes = [P, i32, i32, i32, i32, P, P, i32, i32, i32, i32, P, i64,
                                             i32, P, f64, i32, P, P, i32, P, i32, P, P, i32]
    lib.orc_paged_attention_int4.restype = i32
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ---------------------------------------------------------------- number formats

def f16_to_double(bits: int) -> float:
    return _load().orc_f16_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits))


def e4m3_to_double(code: int) -> float:
    return _load().orc_e4m3_to_double(int(code))


def e4m3_from_float(x: float) -> int:
    return int(_load().orc_e4m3_from_float(float(np.float32(x))))


# ---------------------------------------------------------------- the path

def slot_mapping(block_table, query_start_loc, positions, block_size: int, num_blocks: int):
    """Returns (slot_mapping int64 [T], error bits)."""
    bt = _c(block_table, np.int32)
    qsl = _c(query_start_loc, np.int32)
    pos = _c(positions, np.int32)
    out = np.empty(pos.shape[0], np.int64)
    err = _load().orc_slot_mapping(_ptr(bt), bt.shape[1], bt.shape[0], bt.shape[1], _ptr(qsl),
                                   _ptr(pos), pos.shape[0], block_size, num_blocks, _ptr(out))
    return out, int(err)


def reshape_and_cache(key_bits, value_bits, src_dtype: str, slots, k_cache, v_cache,
                      cache_dtype: str, block_size: int, k_scale: float = 1.0,
                      v_scale: float = 1.0) -> int:
    """Writes key/value rows [T, Hkv, D] (uint16 bits) into k_cache/v_cache in place.

    Caches are numpy arrays [NB, bs, Hkv, D] of uint16 (16-bit dtypes) or uint8 (e4m3).
    Returns the error bits."""
    k = _c(key_bits, np.uint16)
    v = _c(value_bits, np.uint16)
    s = _c(slots, np.int64)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    T, H, D = k.shape
    NB = k_cache.shape[0]
    err = _load().orc_reshape_and_cache(_ptr(k), _ptr(v), _DT[src_dtype], H * D, H * D, T, H, D,
                                        _ptr(s), _ptr(k_cache), _ptr(v_cache), _DT[cache_dtype],
                                        NB, block_size, float(k_scale), float(v_scale))
    if err < 0:
        raise ValueError("oracle: unsupported dtype pair")
    return int(err)


def paged_attention(q_bits, q_dtype: str, k_cache, v_cache, cache_dtype: str, block_table,
                    seq_lens, q_len: int, scale: float, window: int = 0, k_scale: float = 1.0,
                    v_scale: float = 1.0, seqs: Optional[Sequence[int]] = None,
                    threads: Optional[int] = None):
    """Textbook softmax attention over each sequence's materialised K/V.

    q_bits: uint16 [B*q_len, Hq, D]; caches [NB, bs, Hkv, D].  Returns (out float64
    [B*q_len, Hq, D], lse float64 [B*q_len, Hq]); rows of sequences not in ``seqs`` are NaN."""
    q = _c(q_bits, np.uint16)
    bt = _c(block_table, np.int32)
    L = _c(seq_lens, np.int32)
    T, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    assert D2 == D and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    B = L.shape[0]
    sel = _c(np.arange(B) if seqs is None else seqs, np.int32)
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    err = _load().orc_paged_attention(
        _ptr(q), _DT[q_dtype], B, q_len, Hq, _ptr(k_cache), _ptr(v_cache), _DT[cache_dtype], Hkv,
        D, bs, NB, _ptr(bt), bt.shape[1], bt.shape[1], _ptr(L), float(scale), int(window),
        float(k_scale), float(v_scale), _ptr(sel), sel.shape[0], _ptr(out), _ptr(lse),
        int(threads or default_threads()))
    if err:
        raise ValueError(f"oracle: invalid input (error bits {err})")
    return out, lse


def paged_attention_varlen(q_bits, q_dtype: str, k_cache, v_cache, cache_dtype: str, block_table,
                           seq_lens, query_start_loc, scale: float, window: int = 0,
                           k_scale: float = 1.0, v_scale: float = 1.0,
                           seqs: Optional[Sequence[int]] = None, threads: Optional[int] = None):
    """paged_attention with n_b = query_start_loc[b+1] - query_start_loc[b] query rows for
    sequence b (a prefill chunk), at positions L_b - n_b .. L_b - 1.  q_bits: uint16
    [query_start_loc[-1], Hq, D].  Rows of sequences not in ``seqs`` are NaN."""
    q = _c(q_bits, np.uint16)
    bt = _c(block_table, np.int32)
    L = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    T, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    B = L.shape[0]
    assert D2 == D and qsl.shape[0] == B + 1 and qsl[-1] == T
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    sel = _c(np.arange(B) if seqs is None else seqs, np.int32)
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    err = _load().orc_paged_attention_varlen(
        _ptr(q), _DT[q_dtype], B, _ptr(qsl), Hq, _ptr(k_cache), _ptr(v_cache), _DT[cache_dtype],
        Hkv, D, bs, NB, _ptr(bt), bt.shape[1], bt.shape[1], _ptr(L), float(scale), int(window),
        float(k_scale), float(v_scale), _ptr(sel), sel.shape[0], _ptr(out), _ptr(lse),
        int(threads or default_threads()))
    if err:
        raise ValueError(f"oracle: invalid input (error bits {err})")
    return out, lse


def int4_from_float(x: float) -> int:
    """The 4-bit code (two's complement nibble) of x, already divided by its scale."""
    return int(_load().orc_int4_from_float(float(np.float32(x))))


def int4_to_double(nibble: int) -> float:
    return _load().orc_int4_to_double(int(nibble))


def reshape_and_cache_int4(key_bits, value_bits, src_dtype: str, slots, k_cache, v_cache,
                           block_size: int, k_scales, v_scales, group_size: int) -> int:
    """INT4 cache write: caches uint8 [NB, bs, Hkv, D/2] (even dim in the low nibble), scales
    float32 [Hkv, D/group_size].  Returns the error bits."""
    k = _c(key_bits, np.uint16)
    v = _c(value_bits, np.uint16)
    sl = _c(slots, np.int64)
    ks = _c(k_scales, np.float32)
    vs = _c(v_scales, np.float32)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous and k_cache.dtype == np.uint8
    T, H, D = k.shape
    NB = k_cache.shape[0]
    err = _load().orc_reshape_and_cache_int4(_ptr(k), _ptr(v), _DT[src_dtype], H * D, H * D, T, H, D,
                                             _ptr(sl), _ptr(k_cache), _ptr(v_cache), NB, block_size,
                                             _ptr(ks), _ptr(vs), int(group_size))
    if err < 0:
        raise ValueError("oracle: invalid INT4 group size")
    return int(err)


def paged_attention_int4(q_bits, q_dtype: str, k_cache, v_cache, block_table, seq_lens, q_len: int,
                         scale: float, window: int, k_scales, v_scales, group_size: int,
                         seqs: Optional[Sequence[int]] = None, threads: Optional[int] = None):
    """paged_attention over INT4 caches (uint8 [NB, bs, Hkv, D/2]) with (head, dim group) scales."""
    q = _c(q_bits, np.uint16)
    bt = _c(block_table, np.int32)
    L = _c(seq_lens, np.int32)
    ks = _c(k_scales, np.float32)
    vs = _c(v_scales, np.float32)
    T, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    assert D2 * 2 == D and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    B = L.shape[0]
    sel = _c(np.arange(B) if seqs is None else seqs, np.int32)
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    err = _load().orc_paged_attention_int4(
        _ptr(q), _DT[q_dtype], B, q_len, Hq, _ptr(k_cache), _ptr(v_cache), Hkv, D, bs, NB, _ptr(bt),
        bt.shape[1], bt.shape[1], _ptr(L), float(scale), int(window), _ptr(ks), _ptr(vs),
        int(group_size), _ptr(sel), sel.shape[0], _ptr(out), _ptr(lse), int(threads or default_threads()))
    if err:
        raise ValueError(f"oracle: invalid input (error bits {err})")
    return out, lse


def cache_zeros(num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                cache_dtype: str) -> np.ndarray:
    if cache_dtype == "int4":
        return np.zeros((num_blocks, block_size, num_kv_heads, head_dim // 2), np.uint8)
    dt = np.uint8 if cache_dtype == "e4m3" else np.uint16
    return np.zeros((num_blocks, block_size, num_kv_heads, head_dim), dt)
