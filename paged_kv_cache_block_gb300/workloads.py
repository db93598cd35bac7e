"""Seeded synthetic decode batches for the paged KV cache path.

This module is the only code that the CUDA path and the CPU oracle both consume.  It draws
random numbers and lays out block tables the way a block allocator would hand them out; it
computes nothing that the method computes (no slot mapping, no cache write, no attention).
Everything it returns is plain numpy: integer metadata and the raw bit patterns of fp16/bf16
tensors (as uint16), so that each side decodes and uses them on its own.

Workload shapes follow the decode batches named in the specification of this library:

* ``tiny``          4 sequences of lengths {5, 4, 9, 13}, block size 4, 32 physical blocks,
                    4 q heads / 2 kv heads, head_dim 64, fp16, softmax scale 1/8.
* ``opt125m``       12/12 heads, head_dim 64, block size 16, 64 sequences of U{128..2048},
                    16384-block pool, fp16.
* ``llama3_8b``     32/8 heads, head_dim 128, block size 16, 256 sequences of U{512..8192},
                    pool sized to fit, bf16.
* ``llama70b_fp8``  64/8 heads, head_dim 128, block size 16, 32 sequences of 4096 tokens,
                    8192-block pool, e4m3 cache with per-tensor scales, bf16 q/out.
* ``mistral_hybrid`` 32/8 heads, head_dim 128, block size 16, 128 sequences with log-normal
                    lengths (median 2048, sigma 1.0, floor 64, cap 32768), 4 speculative
                    query tokens, 25% of sequences sharing a 1024-token prefix of common
                    physical blocks, two layers: full attention and a 4096-token window.
* ``llama3_8b_int4`` the llama3_8b batch (seed 1008) over INT4 caches with group size 32.

Recipe (identical for every workload):
  * seeds are ``1000 + index`` (index 1..5 in the order above);
  * every random array has its own numpy PCG64 stream, keyed by (seed, stream id, chunk), so
    results do not depend on the thread count or on which arrays are drawn;
  * values are float32 N(0, 1) rounded to the stated dtype with round-to-nearest-even;
  * the physical pool is a seeded permutation of 0..NB-1; sequences take consecutive chunks
    of it in batch order, prefix-sharing sequences first point at the common prefix blocks;
  * ``seq_lens`` include this step's new tokens, which sit at positions L-q_len .. L-1;
  * the existing cache is described by ``pool_k``/``pool_v`` (one source row per physical
    slot, in the q dtype); a consumer writes it into its cache with its own cache-write
    routine over every slot, so fp8 caches are quantised by the code under test;
  * fp8 scales are amax/448 over the float32 values of that layer's K (resp. V) population
    (pool plus new tokens), the usual per-tensor calibration;
  * INT4 group scales are synthetic (no calibration data exists here): float32 U(0.25, 0.5) per
    (kv head, group of dims), one stream for K and one for V, so that codes of N(0, 1) values
    span the whole [-8, 7] range with a few percent saturating.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

# stream ids: one per random array, so arrays can be drawn independently of each other
_S_LENGTHS, _S_PERM, _S_SHARE = 1, 2, 3
_S_POOL_K, _S_POOL_V, _S_NEW_K, _S_NEW_V, _S_Q = 10, 11, 12, 13, 14
_S_K_GSCALE, _S_V_GSCALE = 15, 16
_CHUNK = 1 << 22

E4M3_MAX = 448.0  # largest finite e4m3 magnitude (OCP 8-bit floating point, E4M3)


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str                      # q / new K,V / out: "f16" | "bf16"
    cache_dtype: str                # "f16" | "bf16" | "e4m3" | "int4"
    lengths: Tuple                  # ("fixed", (..)) | ("uniform", lo, hi) | ("lognormal", median, sigma, floor, cap)
    q_len: int = 1
    num_blocks: Optional[int] = None        # None: sized to fit the batch
    windows: Tuple[int, ...] = (0,)         # one entry per layer; 0 = full attention
    scale: Optional[float] = None           # None: 1/sqrt(head_dim)
    shared_prefix_frac: float = 0.0
    shared_prefix_tokens: int = 0
    table_pad: int = 1                      # extra -1 columns in the block table
    seed: int = 0
    group_size: int = 0                     # INT4 caches: dims per scale group

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_dim)

    def replace(self, **kw) -> "WorkloadSpec":
        return dataclasses.replace(self, **kw)


TINY = WorkloadSpec("tiny", 4, 4, 2, 64, 4, "f16", "f16", ("fixed", (5, 4, 9, 13)),
                    num_blocks=32, scale=1.0 / 8.0, seed=1001)
OPT125M = WorkloadSpec("opt125m", 64, 12, 12, 64, 16, "f16", "f16", ("uniform", 128, 2048),
                       num_blocks=16384, seed=1002)
LLAMA3_8B = WorkloadSpec("llama3_8b", 256, 32, 8, 128, 16, "bf16", "bf16", ("uniform", 512, 8192),
                         seed=1003)
LLAMA70B_FP8 = WorkloadSpec("llama70b_fp8", 32, 64, 8, 128, 16, "bf16", "e4m3", ("fixed", (4096,) * 32),
                            num_blocks=8192, seed=1004)
MISTRAL_HYBRID = WorkloadSpec("mistral_hybrid", 128, 32, 8, 128, 16, "bf16", "bf16",
                              ("lognormal", 2048, 1.0, 64, 32768), q_len=4, windows=(0, 4096),
                              shared_prefix_frac=0.25, shared_prefix_tokens=1024, seed=1005)

LLAMA3_8B_INT4 = LLAMA3_8B.replace(name="llama3_8b_int4", cache_dtype="int4", group_size=32, seed=1008)

CONFIGS = {1: TINY, 2: OPT125M, 3: LLAMA3_8B, 4: LLAMA70B_FP8, 5: MISTRAL_HYBRID}
BY_NAME = {s.name: s for s in (*CONFIGS.values(), LLAMA3_8B_INT4)}


@dataclass
class LayerInputs:
    window: int
    q: np.ndarray          # uint16 bits [T, Hq, D]
    new_k: np.ndarray      # uint16 bits [T, Hkv, D]
    new_v: np.ndarray      # uint16 bits [T, Hkv, D]
    pool_k: np.ndarray     # uint16 bits [NB*bs, Hkv, D]: existing cache, one row per slot
    pool_v: np.ndarray
    k_scale: float = 1.0   # fp8 caches only
    v_scale: float = 1.0
    k_gscales: Optional[np.ndarray] = None  # INT4 caches only: float32 [Hkv, D / group_size]
    v_gscales: Optional[np.ndarray] = None


@dataclass
class Workload:
    spec: WorkloadSpec
    seq_lens: np.ndarray          # int32 [B], including this step's tokens
    block_table: np.ndarray       # int32 [B, max_blocks_per_seq], -1 padded
    query_start_loc: np.ndarray   # int32 [B+1]
    positions: np.ndarray         # int32 [T]
    num_blocks: int
    shared: np.ndarray            # bool [B]: sequence starts with the common prefix
    layers: List[LayerInputs] = field(default_factory=list)

    @property
    def num_tokens(self) -> int:
        return int(self.positions.shape[0])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.seq_lens.size else 0


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def _round_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> uint16 bit patterns of fp16 / bf16, round to nearest even."""
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32)
        return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)
    raise ValueError(dtype)


def normal_bits(seed: int, stream: int, shape: Sequence[int], dtype: str,
                want_amax: bool = False):
    """N(0,1) float32 rounded to ``dtype`` bits; chunked so that threads can fill it."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    amax = np.zeros(max(nchunks, 1), np.float32)

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        buf = np.empty(hi - lo, np.float32)
        _rng(seed, stream, c).standard_normal(out=buf, dtype=np.float32)
        bits = _round_f32(buf, dtype)
        out[lo:hi] = bits
        if want_amax:
            amax[c] = np.abs(_bits_to_f32(bits, dtype)).max(initial=0.0)

    workers = min(nchunks, os.cpu_count() or 1)
    if workers <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    out = out.reshape(shape)
    return (out, float(amax.max())) if want_amax else out


def _bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _lengths(spec: WorkloadSpec) -> np.ndarray:
    kind = spec.lengths[0]
    rng = _rng(spec.seed, _S_LENGTHS)
    if kind == "fixed":
        L = np.asarray(spec.lengths[1], np.int64)
        assert L.shape[0] == spec.num_seqs, "fixed lengths must list every sequence"
    elif kind == "uniform":
        _, lo, hi = spec.lengths
        L = rng.integers(lo, hi, size=spec.num_seqs, endpoint=True)
    elif kind == "lognormal":
        _, median, sigma, floor, cap = spec.lengths
        z = rng.standard_normal(spec.num_seqs)
        L = np.rint(np.exp(math.log(median) + sigma * z)).astype(np.int64)
        L = np.clip(L, floor, cap)
    else:
        raise ValueError(kind)
    return L


def make_workload(spec: WorkloadSpec, with_values: bool = True) -> Workload:
    B, bs, ql = spec.num_seqs, spec.block_size, spec.q_len
    L = _lengths(spec)

    shared = np.zeros(B, bool)
    prefix_blocks = 0
    if spec.shared_prefix_frac > 0:
        assert spec.shared_prefix_tokens % bs == 0, "shared prefix must be whole blocks"
        prefix_blocks = spec.shared_prefix_tokens // bs
        n_share = int(round(spec.shared_prefix_frac * B))
        pick = _rng(spec.seed, _S_SHARE).choice(B, size=n_share, replace=False)
        shared[pick] = True
        # sharing sequences extend past the prefix by at least one whole block plus this
        # step's tokens, so new tokens never land in a shared block
        L = np.where(shared, np.maximum(L, spec.shared_prefix_tokens + bs + ql), L)
    L = np.maximum(L, ql)

    need = -(-L // bs)                                   # blocks per sequence
    own = need - np.where(shared, prefix_blocks, 0)      # blocks a sequence owns alone
    used = int(own.sum()) + (prefix_blocks if shared.any() else 0)
    NB = spec.num_blocks if spec.num_blocks is not None else used
    if used > NB:
        raise ValueError(f"{spec.name}: batch needs {used} blocks, pool has {NB}")

    perm = _rng(spec.seed, _S_PERM).permutation(NB).astype(np.int32)
    width = int(need.max()) + spec.table_pad
    table = np.full((B, width), -1, np.int32)
    cursor = prefix_blocks if shared.any() else 0
    for b in range(B):
        row = []
        if shared[b]:
            row.extend(perm[:prefix_blocks])
        row.extend(perm[cursor:cursor + own[b]])
        cursor += int(own[b])
        table[b, :need[b]] = row

    qsl = (np.arange(B + 1, dtype=np.int64) * ql).astype(np.int32)
    positions = (L[:, None] - ql + np.arange(ql)[None, :]).reshape(-1).astype(np.int32)
    wl = Workload(spec, L.astype(np.int32), table, qsl, positions, NB, shared)
    if with_values:
        for li, w in enumerate(spec.windows):
            wl.layers.append(_layer_values(spec, li, w, NB, B * ql))
    return wl


def _layer_values(spec: WorkloadSpec, li: int, window: int, NB: int, T: int) -> LayerInputs:
    H, Hq, D, bs = spec.num_kv_heads, spec.num_q_heads, spec.head_dim, spec.block_size
    base = 100 * li
    fp8 = spec.cache_dtype == "e4m3"
    pk = normal_bits(spec.seed, base + _S_POOL_K, (NB * bs, H, D), spec.dtype, want_amax=fp8)
    pv = normal_bits(spec.seed, base + _S_POOL_V, (NB * bs, H, D), spec.dtype, want_amax=fp8)
    nk = normal_bits(spec.seed, base + _S_NEW_K, (T, H, D), spec.dtype, want_amax=fp8)
    nv = normal_bits(spec.seed, base + _S_NEW_V, (T, H, D), spec.dtype, want_amax=fp8)
    q = normal_bits(spec.seed, base + _S_Q, (T, Hq, D), spec.dtype)
    if spec.cache_dtype == "int4":
        G = spec.group_size
        assert G > 0 and D % G == 0, "INT4 workloads need a group size dividing head_dim"
        ks = _rng(spec.seed, base + _S_K_GSCALE).uniform(0.25, 0.5, (H, D // G)).astype(np.float32)
        vs = _rng(spec.seed, base + _S_V_GSCALE).uniform(0.25, 0.5, (H, D // G)).astype(np.float32)
        return LayerInputs(window, q, nk, nv, pk, pv, k_gscales=ks, v_gscales=vs)
    if fp8:
        (pk, ak), (pv, av), (nk, bk), (nv, bv) = pk, pv, nk, nv
        k_scale = float(np.float32(max(ak, bk)) / np.float32(E4M3_MAX))
        v_scale = float(np.float32(max(av, bv)) / np.float32(E4M3_MAX))
        return LayerInputs(window, q, nk, nv, pk, pv, k_scale, v_scale)
    return LayerInputs(window, q, nk, nv, pk, pv)


# ---------------------------------------------------------------- chunked prefill


@dataclass(frozen=True)
class PrefillSpec:
    """A chunked-prefill batch: each sequence has a cached context and a chunk of new tokens
    (their K/V already written), all attending through the block table."""
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    chunk: Tuple                    # ("fixed", n) | ("uniform", lo, hi): new tokens per sequence
    context: Tuple                  # ("fixed", c) | ("uniform", lo, hi): cached tokens before them
    window: int = 0
    seed: int = 0

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


@dataclass
class PrefillWorkload:
    spec: PrefillSpec
    seq_lens: np.ndarray            # int32 [B]: context + chunk
    chunks: np.ndarray              # int32 [B]
    query_start_loc: np.ndarray     # int32 [B+1]
    block_table: np.ndarray         # int32 [B, width], -1 padded
    num_blocks: int
    q: np.ndarray                   # uint16 bits [T, Hq, D]
    pool_k: np.ndarray              # uint16 bits [NB*bs, Hkv, D]
    pool_v: np.ndarray

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    def visible_keys(self) -> np.ndarray:
        """Per query token, the keys it attends (p + 1, or the window)."""
        out = []
        for L, n in zip(self.seq_lens.astype(np.int64), self.chunks.astype(np.int64)):
            p = L - n + np.arange(n)
            out.append(np.minimum(p + 1, self.spec.window) if self.spec.window > 0 else p + 1)
        return np.concatenate(out) if out else np.zeros(0, np.int64)


def _draw(kind: Tuple, rng: np.random.Generator, n: int) -> np.ndarray:
    if kind[0] == "fixed":
        return np.full(n, kind[1], np.int64)
    return rng.integers(kind[1], kind[2], size=n, endpoint=True)


def make_prefill(spec: PrefillSpec) -> PrefillWorkload:
    B, bs = spec.num_seqs, spec.block_size
    rng = _rng(spec.seed, _S_LENGTHS)
    chunks = _draw(spec.chunk, rng, B)
    ctx = _draw(spec.context, rng, B)
    L = ctx + chunks
    need = -(-L // bs)
    NB = int(need.sum())
    perm = _rng(spec.seed, _S_PERM).permutation(NB).astype(np.int32)
    table = np.full((B, int(need.max()) + 1), -1, np.int32)
    o = 0
    for b in range(B):
        table[b, :need[b]] = perm[o:o + need[b]]
        o += int(need[b])
    qsl = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(qsl[-1])
    H, Hq, D = spec.num_kv_heads, spec.num_q_heads, spec.head_dim
    q = normal_bits(spec.seed, _S_Q, (T, Hq, D), spec.dtype)
    pk = normal_bits(spec.seed, _S_POOL_K, (NB * bs, H, D), spec.dtype)
    pv = normal_bits(spec.seed, _S_POOL_V, (NB * bs, H, D), spec.dtype)
    return PrefillWorkload(spec, L.astype(np.int32), chunks.astype(np.int32), qsl, table, NB, q, pk, pv)


# 16 sequences, a 1024-token chunk each after a cached context of U{0..7168} tokens (chunked
# prefill at Llama-3-8B's attention shape), and 8 whole 2048-token prompts (causal only)
PREFILL_LLAMA3_8B = PrefillSpec("prefill_llama3_8b", 16, 32, 8, 128, 16, "bf16", ("fixed", 1024),
                                ("uniform", 0, 7168), seed=1006)
PREFILL_PROMPT_LLAMA3_8B = PrefillSpec("prefill_prompt_llama3_8b", 8, 32, 8, 128, 16, "bf16",
                                       ("fixed", 2048), ("fixed", 0), seed=1007)
PREFILL_BY_NAME = {s.name: s for s in (PREFILL_LLAMA3_8B, PREFILL_PROMPT_LLAMA3_8B)}


def bits_to_float(bits: np.ndarray, dtype: str) -> np.ndarray:
    """uint16 bits of fp16/bf16 -> float32 (exact)."""
    return _bits_to_f32(np.ascontiguousarray(bits), dtype)


def elem_bytes(dtype: str) -> float:
    return {"e4m3": 1, "int4": 0.5}.get(dtype, 2)
