"""Runs one decode step of a workload on both sides: the CUDA library (through the C ABI binding)
and the CPU oracle, from the same seeded inputs.  Used by the parity tests and the smoke check.

Neither side sees the other's results: the CUDA side fills its cache with its own cache-write
kernel over every slot of the pool, the oracle with its own (16-bit caches are a bit copy, so
the oracle's cache is the pool bits themselves), then each runs slot mapping, the cache write of
the new tokens and attention.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

import oracle
from paged_kv_cache_block_gb300 import workloads as W

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.uint8, "int4": torch.uint8}
# stated tolerances of the specification (max abs for 16-bit, relative to max|oracle| for fp8)
TOL = {"f16": 1e-3, "bf16": 8e-3}
FP8_REL_TOL = 2e-2
# INT4 caches: the codes are exact on both sides; the kernel rounds q * k_scale and the softmax
# weights to fp16 (relative 2^-11 each), so 1e-2 of max|oracle| leaves room for the 16-bit output
INT4_REL_TOL = 1e-2
LSE_TOL = 2e-3


def to_dev(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(TORCH_DT[dtype])


@dataclass
class GpuStep:
    slots: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    out: torch.Tensor
    lse: torch.Tensor
    err: int


def gpu_fill_cache(wl: W.Workload, layer: W.LayerInputs, device="cuda"):
    from paged_kv_cache_block_gb300 import kvcache as kv
    s = wl.spec
    NB, bs, H, D = wl.num_blocks, s.block_size, s.num_kv_heads, s.head_dim
    cdt = TORCH_DT[s.cache_dtype]
    int4 = s.cache_dtype == "int4"
    k_cache = torch.zeros((NB, bs, H, D // 2 if int4 else D), dtype=cdt, device=device)
    v_cache = torch.zeros_like(k_cache)
    pk = to_dev(layer.pool_k, s.dtype, device)
    pv = to_dev(layer.pool_v, s.dtype, device)
    ident = torch.arange(NB * bs, dtype=torch.int64, device=device)
    if int4:
        ks, vs = int4_scales(layer, device)
        kv.reshape_and_cache_int4(pk, pv, ident, k_cache, v_cache, ks, vs)
    else:
        kv.reshape_and_cache(pk, pv, ident, k_cache, v_cache, layer.k_scale, layer.v_scale)
    del pk, pv
    return k_cache, v_cache


def int4_scales(layer: W.LayerInputs, device="cuda"):
    return (torch.from_numpy(layer.k_gscales).to(device), torch.from_numpy(layer.v_gscales).to(device))


def gpu_step(wl: W.Workload, layer: W.LayerInputs, k_cache, v_cache, num_workers: int = 0,
             device="cuda", block_table: Optional[np.ndarray] = None) -> GpuStep:
    from paged_kv_cache_block_gb300 import kvcache as kv
    s = wl.spec
    bt_np = wl.block_table if block_table is None else block_table
    bt = torch.from_numpy(bt_np).to(device)
    qsl = torch.from_numpy(wl.query_start_loc).to(device)
    pos = torch.from_numpy(wl.positions).to(device)
    L = torch.from_numpy(wl.seq_lens).to(device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    slots = kv.compute_slot_mapping(bt, qsl, pos, s.block_size, wl.num_blocks, d_err=err)
    nk = to_dev(layer.new_k, s.dtype, device)
    nv = to_dev(layer.new_v, s.dtype, device)
    q = to_dev(layer.q, s.dtype, device)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=device)
    if s.cache_dtype == "int4":
        ks, vs = int4_scales(layer, device)
        kv.reshape_and_cache_int4(nk, nv, slots, k_cache, v_cache, ks, vs, d_err=err)
        out = kv.paged_attention_decode_int4(q, k_cache, v_cache, bt, L, wl.max_seq_len, s.q_len,
                                             s.softmax_scale, ks, vs, layer.window,
                                             num_workers=num_workers, lse_out=lse, d_err=err)
    else:
        kv.reshape_and_cache(nk, nv, slots, k_cache, v_cache, layer.k_scale, layer.v_scale, d_err=err)
        out = kv.paged_attention_decode(q, k_cache, v_cache, bt, L, wl.max_seq_len, s.q_len,
                                        s.softmax_scale, layer.window, layer.k_scale, layer.v_scale,
                                        num_workers=num_workers, lse_out=lse, d_err=err)
    torch.cuda.synchronize()
    return GpuStep(slots, k_cache, v_cache, out, lse, int(err.item()))


@dataclass
class OracleStep:
    slots: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    out: np.ndarray
    lse: np.ndarray


def oracle_step(wl: W.Workload, layer: W.LayerInputs, seqs: Optional[Sequence[int]] = None,
                block_table: Optional[np.ndarray] = None) -> OracleStep:
    s = wl.spec
    NB, bs, H, D = wl.num_blocks, s.block_size, s.num_kv_heads, s.head_dim
    bt = wl.block_table if block_table is None else block_table
    if s.cache_dtype == "int4":
        return _oracle_step_int4(wl, layer, bt, seqs)
    if s.cache_dtype == s.dtype:
        kc = layer.pool_k.reshape(NB, bs, H, D).copy()
        vc = layer.pool_v.reshape(NB, bs, H, D).copy()
    else:
        kc = oracle.cache_zeros(NB, bs, H, D, s.cache_dtype)
        vc = oracle.cache_zeros(NB, bs, H, D, s.cache_dtype)
        ident = np.arange(NB * bs, dtype=np.int64)
        assert oracle.reshape_and_cache(layer.pool_k, layer.pool_v, s.dtype, ident, kc, vc,
                                        s.cache_dtype, bs, layer.k_scale, layer.v_scale) == 0
    slots, err = oracle.slot_mapping(bt, wl.query_start_loc, wl.positions, bs, NB)
    assert err == 0
    assert oracle.reshape_and_cache(layer.new_k, layer.new_v, s.dtype, slots, kc, vc,
                                    s.cache_dtype, bs, layer.k_scale, layer.v_scale) == 0
    out, lse = oracle.paged_attention(layer.q, s.dtype, kc, vc, s.cache_dtype, bt, wl.seq_lens,
                                      s.q_len, s.softmax_scale, layer.window, layer.k_scale,
                                      layer.v_scale, seqs=seqs)
    return OracleStep(slots, kc, vc, out, lse)


def _oracle_step_int4(wl: W.Workload, layer: W.LayerInputs, bt: np.ndarray,
                      seqs: Optional[Sequence[int]]) -> OracleStep:
    s = wl.spec
    NB, bs, H, D = wl.num_blocks, s.block_size, s.num_kv_heads, s.head_dim
    kc = oracle.cache_zeros(NB, bs, H, D, "int4")
    vc = oracle.cache_zeros(NB, bs, H, D, "int4")
    ks, vs, G = layer.k_gscales, layer.v_gscales, s.group_size
    ident = np.arange(NB * bs, dtype=np.int64)
    assert oracle.reshape_and_cache_int4(layer.pool_k, layer.pool_v, s.dtype, ident, kc, vc, bs, ks, vs, G) == 0
    slots, err = oracle.slot_mapping(bt, wl.query_start_loc, wl.positions, bs, NB)
    assert err == 0
    assert oracle.reshape_and_cache_int4(layer.new_k, layer.new_v, s.dtype, slots, kc, vc, bs, ks, vs, G) == 0
    out, lse = oracle.paged_attention_int4(layer.q, s.dtype, kc, vc, bt, wl.seq_lens, s.q_len,
                                           s.softmax_scale, layer.window, ks, vs, G, seqs=seqs)
    return OracleStep(slots, kc, vc, out, lse)


def rows_of(wl: W.Workload, seqs: Sequence[int]) -> np.ndarray:
    ql = wl.spec.q_len
    return np.concatenate([np.arange(b * ql, (b + 1) * ql) for b in seqs])


def check_attention(wl: W.Workload, g: GpuStep, o: OracleStep, rows: Optional[np.ndarray] = None):
    """Element-wise comparison at the specification's tolerance; returns the error figure."""
    s = wl.spec
    out = g.out.float().cpu().numpy().astype(np.float64)
    lse = g.lse.cpu().numpy().astype(np.float64)
    ref_out, ref_lse = o.out, o.lse
    if rows is not None:
        out, lse, ref_out, ref_lse = out[rows], lse[rows], ref_out[rows], ref_lse[rows]
    assert np.isfinite(out).all(), "non-finite attention output"
    assert np.isfinite(ref_out).all()
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=LSE_TOL)
    if s.cache_dtype in ("e4m3", "int4"):
        tol = FP8_REL_TOL if s.cache_dtype == "e4m3" else INT4_REL_TOL
        rel = np.abs(out - ref_out).max() / np.abs(ref_out).max()
        assert rel <= tol, f"{s.cache_dtype} relative error {rel:.3e} > {tol}"
        return rel
    return check_close16(out, ref_out, s.dtype)


def check_close16(out: np.ndarray, ref_out: np.ndarray, dtype: str) -> float:
    """16-bit outputs against the oracle, element by element; returns the max abs error.

    The stated max-abs tolerance bounds the kernel's own error; the output format adds its
    rounding on top (half an ulp of the result: 7.8e-3 for bf16 at |x| in [2,4), so an exactly
    rounded bf16 output alone can exceed 8e-3)."""
    diff = np.abs(out - ref_out)
    allowed = TOL[dtype] + 0.5 * out_ulp(ref_out, dtype)
    worst = np.unravel_index(np.argmax(diff - allowed), diff.shape)
    assert (diff <= allowed).all(), (
        f"error {diff[worst]:.3e} > {TOL[dtype]} + half-ulp at {worst} (oracle {ref_out[worst]:.5f}); "
        f"max abs error {diff.max():.3e}")
    return float(diff.max())


def out_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the 16-bit output format at |x| (normal range)."""
    mant = 7 if dtype == "bf16" else 10
    _, e = np.frexp(np.abs(x))
    return np.ldexp(1.0, np.maximum(e - 1, -14) - mant)


def cache_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_whole_cache(g: GpuStep, o: OracleStep) -> None:
    """Every slot of both caches bit for bit (written, untouched and never-read blocks alike),
    compared a slice of blocks at a time so host memory stays bounded."""
    NB = g.k_cache.shape[0]
    step = max(1, (256 << 20) // max(1, g.k_cache[0].numel() * g.k_cache.element_size()))
    for dev, ref in ((g.k_cache, o.k_cache), (g.v_cache, o.v_cache)):
        ref = ref.reshape((NB,) + tuple(dev.shape[1:]))
        for b0 in range(0, NB, step):
            got = cache_bits(dev[b0:b0 + step])
            want = ref[b0:b0 + step]
            if not np.array_equal(got, want):
                bad = np.argwhere(got != want)[0]
                raise AssertionError(f"cache differs from the oracle at block {b0 + bad[0]}, index {tuple(bad[1:])}")


def gpu_step_fused(wl: W.Workload, layer: W.LayerInputs, k_cache, v_cache, num_workers: int = 0,
                   device="cuda") -> GpuStep:
    """The same decode step through kv_decode_step (one launch)."""
    from paged_kv_cache_block_gb300 import kvcache as kv
    s = wl.spec
    bt = torch.from_numpy(wl.block_table).to(device)
    qsl = torch.from_numpy(wl.query_start_loc).to(device)
    pos = torch.from_numpy(wl.positions).to(device)
    L = torch.from_numpy(wl.seq_lens).to(device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    nk = to_dev(layer.new_k, s.dtype, device)
    nv = to_dev(layer.new_v, s.dtype, device)
    q = to_dev(layer.q, s.dtype, device)
    lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=device)
    slots = torch.empty(q.shape[0], dtype=torch.int64, device=device)
    if s.cache_dtype == "int4":
        ks, vs = int4_scales(layer, device)
        out = kv.decode_step_int4(bt, qsl, pos, nk, nv, q, k_cache, v_cache, L, wl.max_seq_len, s.q_len,
                                  s.softmax_scale, ks, vs, layer.window, num_workers=num_workers,
                                  lse_out=lse, slot_mapping=slots, d_err=err)
    else:
        out = kv.decode_step(bt, qsl, pos, nk, nv, q, k_cache, v_cache, L, wl.max_seq_len, s.q_len,
                             s.softmax_scale, layer.window, layer.k_scale, layer.v_scale,
                             num_workers=num_workers, lse_out=lse, slot_mapping=slots, d_err=err)
    torch.cuda.synchronize()
    return GpuStep(slots, k_cache, v_cache, out, lse, int(err.item()))
