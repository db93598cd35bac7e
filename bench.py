"""Benchmark of one decode step of the paged KV cache path on GB300.

A step is the whole hot path for one batch: slot mapping, the cache write of the step's new K/V
rows and paged decode attention (with its log-sum-exp merge), for every attention layer of the
workload.  Default workload: the Llama-3-8B-shaped GQA decode layer (256 sequences of U{512..8192}
tokens, 32/8 heads, head_dim 128, block size 16, bf16).  Inputs are resident in HBM when the timed
region starts; the KV cache (4.6 GB) is larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own batch of the same shape
(sequences are independent: weak scaling, no collective on the data path); the time is the max
over ranks.  ``--impl reference`` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_block_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV-read GB/s and % of HBM peak; decode tokens/s"
UNIT = "GB/s"
# layers of the model each decode workload is shaped after (context for the per-layer tokens/s)
MODEL_LAYERS = {"tiny": 1, "opt125m": 12, "llama3_8b": 32, "llama70b_fp8": 80, "mistral_hybrid": 32}
PREFILL_METRIC = "chunked-prefill paged attention TFLOP/s (visible query-key pairs) and % of bf16 tensor peak"
ADMISSION_METRIC = "block-table update + zero fill of new blocks, GB/s and % of HBM peak"


# ---------------------------------------------------------------- byte accounting

def attended_keys(wl: W.Workload, window: int) -> np.ndarray:
    """Per sequence, the keys any of its queries attends: [first key of the first query, L)."""
    L = wl.seq_lens.astype(np.int64)
    ql = wl.spec.q_len
    lo = np.maximum(0, L - ql - window + 1) if window > 0 else np.zeros_like(L)
    return lo, L


def algorithmic_bytes(wl: W.Workload) -> dict:
    """Bytes the path must move at least once, per step.

    attention: each distinct physical cache slot that some query attends, read once for K and
               once for V (a prefix shared by several sequences counts once), plus q, out and
               the block-table entries of the attended blocks (4 B each);
    cache write: new K/V rows read and written; slot mapping: positions, table entries, slots."""
    s = wl.spec
    bs = s.block_size
    eb_c = W.elem_bytes(s.cache_dtype)
    row = int(2 * s.num_kv_heads * s.head_dim * eb_c)
    # INT4 group scales of K and V, read once per layer
    scales = 2 * s.num_kv_heads * (s.head_dim // s.group_size) * 4 if s.cache_dtype == "int4" else 0
    T = wl.num_tokens
    q_out = 2 * T * s.num_q_heads * s.head_dim * 2
    per_layer = []
    for layer in wl.layers:
        lo, hi = attended_keys(wl, layer.window)
        seen = np.zeros(wl.num_blocks * bs, dtype=bool)
        n_blocks = 0
        for b in range(len(hi)):
            keys = np.arange(lo[b], hi[b])
            seen[wl.block_table[b, keys // bs].astype(np.int64) * bs + keys % bs] = True
            n_blocks += int((hi[b] + bs - 1) // bs - lo[b] // bs)
        n_unique = int(seen.sum())
        attn = n_unique * row + q_out + 4 * n_blocks + scales
        write = T * row + T * s.num_kv_heads * s.head_dim * 2 * 2 + scales
        per_layer.append({"attention": attn, "cache_write": write,
                          "logical_kv": int((hi - lo).sum()) * row})
    slot_map = T * (4 + 8 + 4) + 4 * (wl.num_tokens // s.q_len + 1)
    return {"layers": per_layer, "slot_mapping": slot_map,
            "step": slot_map + sum(l["attention"] + l["cache_write"] for l in per_layer)}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """SM clock and clock-event reasons sampled every 10 ms from NVML (read only) in a thread,
    over exactly the timed region; nvidia-smi at 200 ms if NVML cannot be loaded."""

    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id: str):
        import threading
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self._stop = threading.Event()
        self._thread = None
        self._smi = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for " + pci_bus_id)
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._nv, self._h = nv, h
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        except OSError:
            self._smi = subprocess.Popen(
                ["nvidia-smi", f"--id={pci_bus_id}", "--query-gpu=clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self._nv.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if self._nv.nvmlDeviceGetCurrentClocksEventReasons(self._h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            self._stop.wait(0.01)

    def stop(self) -> dict:
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            src = "nvml 10 ms"
        elif self._smi is not None:
            self._smi.terminate()
            out, _ = self._smi.communicate(timeout=5)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.strip().splitlines():
                f = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except (ValueError, IndexError):
                    continue
                for n, v in zip(names, f[2:6]):
                    if v.lower() == "active":
                        self.reasons.add(n)
            src = "nvidia-smi 200 ms"
        else:
            src = "unavailable"
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples), "source": src,
                "reasons": sorted(self.reasons)}


# ---------------------------------------------------------------- peaks and profile data

def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def kernel_source_hash(workload: str = "") -> str:
    h = hashlib.sha256()
    kernel = "paged_decode_int4.cu" if W.BY_NAME.get(workload) is not None and \
        W.BY_NAME[workload].cache_dtype == "int4" else "paged_decode_kernel.cuh"
    for f in (kernel, "decode_common.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_block_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary, or None
    when that summary was taken on a different kernel source."""
    p = os.path.join(ROOT, "profiles", f"paged_decode_{workload}.md")
    if not os.path.exists(p):
        return None
    src, traffic = None, None
    for line in open(p):
        if line.startswith("kernel_source_sha256_16:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_full_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if src == kernel_source_hash(workload) else None


# ---------------------------------------------------------------- CPU oracle timing

def oracle_sample_rate(wl: W.Workload, budget_s: float, threads: int):
    """Time the oracle (attention of every layer over a growing subset of sequences, with the
    slot mapping and cache write of their new tokens) until ~budget_s has been spent."""
    import oracle
    s = wl.spec
    NB, bs, H, D = wl.num_blocks, s.block_size, s.num_kv_heads, s.head_dim
    caches = []
    int4 = s.cache_dtype == "int4"
    G = s.group_size
    for layer in wl.layers:
        if s.cache_dtype == s.dtype:
            caches.append((layer.pool_k.reshape(NB, bs, H, D), layer.pool_v.reshape(NB, bs, H, D)))
        else:
            caches.append(None)   # quantised per sample below
    order = np.random.default_rng(0).permutation(len(wl.seq_lens))
    done_bytes, spent, n_seqs, i = 0.0, 0.0, 0, 0
    chunk = 1
    while i < len(order) and spent < budget_s:
        sel = np.sort(order[i:i + chunk])
        i += chunk
        sub = _sub_workload(wl, sel)
        t0 = time.perf_counter()
        slots, _ = oracle.slot_mapping(sub.block_table, sub.query_start_loc, sub.positions, bs, NB)
        for li, layer in enumerate(sub.layers):
            if caches[li] is not None:
                kc, vc = caches[li]
            else:
                # E4M3 / INT4: the oracle quantises the slots this sample reads
                kc = oracle.cache_zeros(NB, bs, H, D, s.cache_dtype)
                vc = oracle.cache_zeros(NB, bs, H, D, s.cache_dtype)
                need = np.unique(np.concatenate([
                    np.arange(sub.block_table[b, j] * bs, sub.block_table[b, j] * bs + bs)
                    for b in range(len(sel)) for j in range(-(-int(sub.seq_lens[b]) // bs))]))
                if int4:
                    oracle.reshape_and_cache_int4(layer.pool_k[need], layer.pool_v[need], s.dtype, need, kc,
                                                  vc, bs, layer.k_gscales, layer.v_gscales, G)
                else:
                    oracle.reshape_and_cache(layer.pool_k[need], layer.pool_v[need], s.dtype, need, kc, vc,
                                             s.cache_dtype, bs, layer.k_scale, layer.v_scale)
            if int4:
                oracle.reshape_and_cache_int4(layer.new_k, layer.new_v, s.dtype, slots, kc, vc, bs,
                                              layer.k_gscales, layer.v_gscales, G)
                oracle.paged_attention_int4(layer.q, s.dtype, kc, vc, sub.block_table, sub.seq_lens,
                                            s.q_len, s.softmax_scale, layer.window, layer.k_gscales,
                                            layer.v_gscales, G, threads=threads)
                continue
            oracle.reshape_and_cache(layer.new_k, layer.new_v, s.dtype, slots, kc, vc,
                                     s.cache_dtype, bs, layer.k_scale, layer.v_scale)
            oracle.paged_attention(layer.q, s.dtype, kc, vc, s.cache_dtype, sub.block_table,
                                   sub.seq_lens, s.q_len, s.softmax_scale, layer.window,
                                   layer.k_scale, layer.v_scale, threads=threads)
        spent += time.perf_counter() - t0
        done_bytes += algorithmic_bytes(sub)["step"]
        n_seqs += len(sel)
        chunk *= 2
    return done_bytes / spent / 1e9, n_seqs, spent


def _sub_workload(wl: W.Workload, sel: np.ndarray) -> W.Workload:
    ql = wl.spec.q_len
    rows = np.concatenate([np.arange(b * ql, (b + 1) * ql) for b in sel])
    layers = [W.LayerInputs(l.window, l.q[rows], l.new_k[rows], l.new_v[rows], l.pool_k, l.pool_v,
                            l.k_scale, l.v_scale, l.k_gscales, l.v_gscales) for l in wl.layers]
    spec = wl.spec.replace(num_seqs=len(sel))
    return W.Workload(spec, wl.seq_lens[sel], wl.block_table[sel],
                      (np.arange(len(sel) + 1) * ql).astype(np.int32), wl.positions[rows],
                      wl.num_blocks, wl.shared[sel], layers)


# ---------------------------------------------------------------- ranks (one process per GPU)

def ranks_init(world: int, backend: str = "nccl") -> None:
    """One process per GPU under torchrun: the process group (rendezvous from the environment)."""
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        if not dist.is_initialized():
            dist.init_process_group(backend)


def ranks_barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def ranks_max(values, world: int, device="cpu"):
    """The largest of each value over the ranks: the slowest rank's time is the job's time."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def ranks_done(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- timing

def cuda_timed(fn, n: int, stream) -> float:
    """ms for n calls of fn, from CUDA events on the launching stream, synchronised on both sides."""
    import torch
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def timed_windows(fn, n: int, stream, world: int, repeats: int, min_ms: float = 200.0):
    """Windows of exactly n calls each, every window bracketed by a barrier over the ranks and a
    device synchronisation, and its time the max over ranks.  At least `repeats` windows, more
    when needed so that the windows together last about `min_ms` (enough NVML clock samples).
    Returns the per-window times in ms."""
    first = cuda_timed(fn, n, stream)
    count = max(repeats, min(1000, int(np.ceil(min_ms / max(first, 1e-3)))))
    out = []
    for _ in range(count):
        ranks_barrier(world)
        ms = cuda_timed(fn, n, stream)
        out.append(ranks_max([ms], world, _rank_device())[0])
    return out


def _rank_device():
    import torch
    return torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))


def window_summary(ms_windows, n: int) -> dict:
    """Median and min of the per-step time over the timed windows."""
    return {"count": len(ms_windows), "steps_each": n,
            "ms_per_step_median": round(statistics.median(ms_windows) / n, 5),
            "ms_per_step_min": round(min(ms_windows) / n, 5)}


# ---------------------------------------------------------------- the GPU arm

def to_dev(bits: np.ndarray, dtype: str, device):
    """16-bit element bits (uint16) as a device tensor of that dtype."""
    import torch
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(tdt)


def fill_cache(wl: W.Workload, layer: W.LayerInputs, device):
    """The layer's cache written by the library's own cache-write kernel over every slot."""
    import torch
    from paged_kv_cache_block_gb300 import kvcache as kv
    s = wl.spec
    int4 = s.cache_dtype == "int4"
    cdt = torch.uint8 if s.cache_dtype in ("e4m3", "int4") else \
        {"f16": torch.float16, "bf16": torch.bfloat16}[s.cache_dtype]
    k_cache = torch.zeros((wl.num_blocks, s.block_size, s.num_kv_heads, s.head_dim // 2 if int4 else s.head_dim),
                          dtype=cdt, device=device)
    v_cache = torch.zeros_like(k_cache)
    ident = torch.arange(wl.num_blocks * s.block_size, dtype=torch.int64, device=device)
    pk, pv = to_dev(layer.pool_k, s.dtype, device), to_dev(layer.pool_v, s.dtype, device)
    if int4:
        ks, vs = int4_scales(layer, device)
        kv.reshape_and_cache_int4(pk, pv, ident, k_cache, v_cache, ks, vs)
    else:
        kv.reshape_and_cache(pk, pv, ident, k_cache, v_cache, layer.k_scale, layer.v_scale)
    return k_cache, v_cache


def int4_scales(layer: W.LayerInputs, device):
    import torch
    return torch.from_numpy(layer.k_gscales).to(device), torch.from_numpy(layer.v_gscales).to(device)


def pack_layout(sizes, align: int = 256):
    """Offsets of buffers of the given byte sizes packed one after another, each starting on an
    `align`-byte boundary, and the total size (at least 1)."""
    offs, off = [], 0
    for n in sizes:
        off = (off + align - 1) // align * align
        offs.append(off)
        off += n
    return offs, max(off, 1)


def copy_pieces(n: int, align: int = 256, piece_min: int = 16 << 20, max_pieces: int = 4):
    """[lo, hi) byte ranges that cover [0, n) in order: one range, or up to `max_pieces` of at
    least `piece_min` bytes each with every inner cut on an `align`-byte boundary."""
    k = max(1, min(max_pieces, n // piece_min))
    cut = [(n * i // k) // align * align for i in range(k)] + [n]
    return list(zip(cut[:-1], cut[1:]))


class HostPipe:
    """End-to-end steps from host memory, as a serving loop runs them: a step's inputs sit in one
    pinned host buffer and go to the device in one copy, its outputs come back in one copy (split
    into up to four pieces on their own copy streams when they are large, so that several copy
    engines share them).  Two device sets (inputs and outputs) alternate; uploads and downloads
    run on their own streams, so step i + 1's upload and step i - 1's download overlap step i's
    kernels.  Every copy of every timed step lies inside the timed region.

    inputs: {name: (numpy array, torch dtype)}; outputs: {name: (torch dtype, shape)}."""

    ALIGN = 256

    def __init__(self, device, inputs: dict, outputs: dict):
        import torch
        self.torch = torch

        def layout(sizes):
            return pack_layout(sizes, self.ALIGN)

        arrs = {k: np.ascontiguousarray(a) for k, (a, _) in inputs.items()}
        offs, size = layout([a.nbytes for a in arrs.values()])
        self.h_in = torch.empty(size, dtype=torch.uint8).pin_memory()
        hv = self.h_in.numpy()
        self.in_meta = []
        for (k, a), o in zip(arrs.items(), offs):
            hv[o:o + a.nbytes] = a.reshape(-1).view(np.uint8)
            self.in_meta.append((k, o, a.nbytes, inputs[k][1], a.shape))
        onb = {k: int(np.prod(shape)) * torch.empty((), dtype=dt).element_size() for k, (dt, shape) in outputs.items()}
        ooffs, osize = layout(list(onb.values()))
        self.out_meta = [(k, o, onb[k], outputs[k][0], outputs[k][1]) for k, o in zip(outputs, ooffs)]
        self.h_out = [torch.empty(osize, dtype=torch.uint8).pin_memory() for _ in range(2)]
        self.d_in = [torch.empty(size, dtype=torch.uint8, device=device) for _ in range(2)]
        self.d_out = [torch.zeros(osize, dtype=torch.uint8, device=device) for _ in range(2)]
        for d in self.d_in:
            d.copy_(self.h_in)
        self.h2d_bytes, self.d2h_bytes = size, osize

        self.up_pieces, self.down_pieces = copy_pieces(size, self.ALIGN), copy_pieces(osize, self.ALIGN)
        self.up = [torch.cuda.Stream(device) for _ in self.up_pieces]
        self.down = [torch.cuda.Stream(device) for _ in self.down_pieces]

    def views(self, k: int) -> dict:
        v = {}
        for name, o, nb, dt, shape in self.in_meta:
            v[name] = self.d_in[k][o:o + nb].view(dt).view(shape)
        for name, o, nb, dt, shape in self.out_meta:
            v[name] = self.d_out[k][o:o + nb].view(dt).view(shape)
        return v

    def run(self, n: int, step, stream) -> float:
        """n steps; step(views) enqueues one step's work on the current stream.  Returns ms."""
        torch = self.torch
        sets = [self.views(k) for k in range(2)]
        up_done = [[torch.cuda.Event() for _ in self.up] for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        down_done = [[torch.cuda.Event() for _ in self.down] for _ in range(2)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for st in self.up + self.down:
            st.wait_event(e0)
        for i in range(n):
            k = i & 1
            for st, (lo, hi), ev in zip(self.up, self.up_pieces, up_done[k]):
                with torch.cuda.stream(st):
                    if i >= 2:
                        st.wait_event(comp_done[k])  # step i - 2 has finished reading set k
                    self.d_in[k][lo:hi].copy_(self.h_in[lo:hi], non_blocking=True)
                    ev.record(st)
            for ev in up_done[k]:
                stream.wait_event(ev)
            if i >= 2:
                for ev in down_done[k]:
                    stream.wait_event(ev)  # step i - 2's outputs have left set k
            with torch.cuda.stream(stream):
                step(sets[k])
            comp_done[k].record(stream)
            for st, (lo, hi), ev in zip(self.down, self.down_pieces, down_done[k]):
                with torch.cuda.stream(st):
                    st.wait_event(comp_done[k])
                    self.h_out[k][lo:hi].copy_(self.d_out[k][lo:hi], non_blocking=True)
                    ev.record(st)
        for k in range(min(n, 2)):
            for ev in down_done[k]:
                stream.wait_event(ev)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def output(self, k: int, name: str):
        for nm, o, nb, dt, shape in self.out_meta:
            if nm == name:
                return self.h_out[k][o:o + nb].view(dt).view(shape)
        raise KeyError(name)


def run_gpu(args, name: str, rank: int, world: int):
    import torch
    from paged_kv_cache_block_gb300 import kvcache as kv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    spec = W.BY_NAME[name]
    if args.num_seqs:
        spec = spec.replace(num_seqs=args.num_seqs, num_blocks=None) if spec.lengths[0] != "fixed" else \
            spec.replace(num_seqs=args.num_seqs, num_blocks=None,
                         lengths=("fixed", spec.lengths[1][:args.num_seqs]))
    wl = W.make_workload(spec)
    s = wl.spec
    stream = torch.cuda.current_stream()
    int4 = s.cache_dtype == "int4"

    # resident inputs
    bt = torch.from_numpy(wl.block_table).to(dev)
    qsl = torch.from_numpy(wl.query_start_loc).to(dev)
    pos = torch.from_numpy(wl.positions).to(dev)
    L = torch.from_numpy(wl.seq_lens).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    layers = []
    for layer in wl.layers:
        kc, vc = fill_cache(wl, layer, dev)
        q = to_dev(layer.q, s.dtype, dev)
        nk = to_dev(layer.new_k, s.dtype, dev)
        nv = to_dev(layer.new_v, s.dtype, dev)
        out = torch.empty_like(q)
        need = kv.paged_attention_workspace_size(s.num_seqs, s.q_len, s.num_q_heads, s.num_kv_heads,
                                                 s.head_dim, s.block_size,
                                                 kv.KV_INT4 if int4 else kv.dtype_code(kc.dtype),
                                                 wl.max_seq_len, layer.window, args.workers)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        ks, vs = int4_scales(layer, dev) if int4 else (None, None)
        layers.append(dict(layer=layer, kc=kc, vc=vc, q=q, nk=nk, nv=nv, out=out, ws=ws, ks=ks, vs=vs))
    slots = torch.empty(wl.num_tokens, dtype=torch.int64, device=dev)
    torch.cuda.synchronize()

    # a step's per-call tensors: the resident ones here, a HostPipe set in the end-to-end leg
    resident = dict(bt=bt, qsl=qsl, pos=pos, L=L)
    for i, d in enumerate(layers):
        for k in ("q", "nk", "nv", "out"):
            resident[f"{k}{i}"] = d[k]

    def step(t=resident):
        if args.mode == "fused":
            for i, d in enumerate(layers):
                fused(d, t, i)
            return
        kv.compute_slot_mapping(t["bt"], t["qsl"], t["pos"], s.block_size, wl.num_blocks, slot_mapping=slots,
                                d_err=err)
        for i, d in enumerate(layers):
            l = d["layer"]
            if int4:
                kv.reshape_and_cache_int4(t[f"nk{i}"], t[f"nv{i}"], slots, d["kc"], d["vc"], d["ks"], d["vs"],
                                          d_err=err)
            else:
                kv.reshape_and_cache(t[f"nk{i}"], t[f"nv{i}"], slots, d["kc"], d["vc"], l.k_scale, l.v_scale,
                                     d_err=err)
            attention(d, t, i)

    def fused(d, t, i):
        l = d["layer"]
        if int4:
            kv.decode_step_int4(t["bt"], t["qsl"], t["pos"], t[f"nk{i}"], t[f"nv{i}"], t[f"q{i}"], d["kc"], d["vc"],
                                t["L"], wl.max_seq_len, s.q_len, s.softmax_scale, d["ks"], d["vs"], l.window,
                                num_workers=args.workers, workspace=d["ws"], out=t[f"out{i}"], d_err=err)
            return
        kv.decode_step(t["bt"], t["qsl"], t["pos"], t[f"nk{i}"], t[f"nv{i}"], t[f"q{i}"], d["kc"], d["vc"], t["L"],
                       wl.max_seq_len, s.q_len, s.softmax_scale, l.window, l.k_scale, l.v_scale,
                       num_workers=args.workers, workspace=d["ws"], out=t[f"out{i}"], d_err=err)

    def attention(d, t, i):
        l = d["layer"]
        if int4:
            kv.paged_attention_decode_int4(t[f"q{i}"], d["kc"], d["vc"], t["bt"], t["L"], wl.max_seq_len, s.q_len,
                                           s.softmax_scale, d["ks"], d["vs"], l.window, num_workers=args.workers,
                                           workspace=d["ws"], out=t[f"out{i}"], d_err=err)
            return
        kv.paged_attention_decode(t[f"q{i}"], d["kc"], d["vc"], t["bt"], t["L"], wl.max_seq_len, s.q_len,
                                  s.softmax_scale, l.window, l.k_scale, l.v_scale, num_workers=args.workers,
                                  workspace=d["ws"], out=t[f"out{i}"], d_err=err)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if err.item() != 0:
        raise RuntimeError(f"device error bits {err.item()} during warm-up")

    # the K timed steps are one CUDA graph, replayed once per timed window (as a serving loop
    # replays a whole decode iteration, every layer, as one graph); the attention calls alone are
    # captured the same way, to time the dominant kernel without the rest of the step
    g_step, g_attn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        for _ in range(args.steps):
            step()
    with torch.cuda.graph(g_attn):
        for _ in range(args.steps):
            for i, d in enumerate(layers):
                if args.mode == "fused":
                    fused(d, resident, i)
                else:
                    attention(d, resident, i)
    for _ in range(max(1, args.warmup // args.steps)):
        g_step.replay()
        g_attn.replay()
    torch.cuda.synchronize()

    def timed(fn, n):
        return cuda_timed(fn, n, stream)

    ranks_barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(pci_of(dev))
    win_step = timed_windows(g_step.replay, 1, stream, world, args.repeats)
    clk = clocks.stop()
    ranks_barrier(world)
    win_attn = timed_windows(g_attn.replay, 1, stream, world, args.repeats)
    ms_eager = timed(step, args.steps)

    # the write path alone (slot mapping + cache write of the first layer), as a graph replay
    def write_path():
        kv.compute_slot_mapping(bt, qsl, pos, s.block_size, wl.num_blocks, slot_mapping=slots, d_err=err)
        d, l = layers[0], layers[0]["layer"]
        if int4:
            kv.reshape_and_cache_int4(d["nk"], d["nv"], slots, d["kc"], d["vc"], d["ks"], d["vs"], d_err=err)
        else:
            kv.reshape_and_cache(d["nk"], d["nv"], slots, d["kc"], d["vc"], l.k_scale, l.v_scale, d_err=err)
    g_write = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_write):
        write_path()
    for _ in range(args.warmup):
        g_write.replay()
    torch.cuda.synchronize()
    us_write = timed(g_write.replay, args.steps) / args.steps * 1e3

    # end to end through the public API: every step's inputs from pinned host memory, its outputs
    # back to the host (HostPipe: one copy each way, double-buffered on copy streams)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[s.dtype]
    h_inputs = dict(bt=(wl.block_table, torch.int32), qsl=(wl.query_start_loc, torch.int32),
                    pos=(wl.positions, torch.int32), L=(wl.seq_lens, torch.int32))
    h_outputs = {}
    for i, d in enumerate(layers):
        l = d["layer"]
        h_inputs[f"q{i}"] = (l.q, tdt)
        h_inputs[f"nk{i}"] = (l.new_k, tdt)
        h_inputs[f"nv{i}"] = (l.new_v, tdt)
        h_outputs[f"out{i}"] = (tdt, tuple(d["out"].shape))
    pipe = HostPipe(dev, h_inputs, h_outputs)
    pipe.run(max(1, args.warmup), step, stream)
    ms_e2e = pipe.run(args.steps, step, stream)
    h2d, d2h = pipe.h2d_bytes, pipe.d2h_bytes
    if err.item() != 0:
        raise RuntimeError(f"device error bits {err.item()}")
    # the outputs that came back are the resident step's outputs, bit for bit
    for i, d in enumerate(layers):
        got = pipe.output((args.steps - 1) & 1, f"out{i}")
        if not torch.equal(got.view(torch.int16), d["out"].cpu().view(torch.int16)):
            raise RuntimeError("end-to-end outputs differ from the resident step's")

    ms_e2e, ms_eager = ranks_max([ms_e2e, ms_eager], world, dev)
    return dict(wl=wl, win_step=win_step, win_attn=win_attn, ms_e2e=ms_e2e, ms_eager=ms_eager, h2d=h2d,
                d2h=d2h, clk=clk, layers=layers, us_write=us_write)


def pci_of(dev) -> str:
    import torch
    props = torch.cuda.get_device_properties(dev)
    return f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"


# ---------------------------------------------------------------- block manager: admission

ADMISSION = dict(layers=32, num_blocks=8192, block_size=16, num_kv_heads=8, head_dim=128,
                 rows=256, max_blocks=1024, new_requests=16, prompt=2048)


def admission_bytes(n_updates: int, n_zero: int, n_caches: int, block_bytes: int) -> int:
    """Bytes kv_apply_block_updates must move: each update read (12 B) and its entry written
    (4 B), each zero-fill id read (4 B), every listed block of every cache written once."""
    return 16 * n_updates + 4 * n_zero + n_zero * n_caches * block_bytes


def oracle_admission_rate(budget_s: float):
    """The oracle's block manager + apply_updates (Python + numpy) on the admission workload's
    geometry, one request of 2048 tokens at a time, until ~budget_s has been spent."""
    from oracle import block_manager as bmo
    a = ADMISSION
    blk_elems = a["block_size"] * a["num_kv_heads"] * a["head_dim"]
    # a slice of the pool is enough for the sample (one request's 128 blocks and some spare):
    # ids are taken first in, first out, so every admission zeroes other blocks
    nb = 160
    caches = [np.ones((nb, blk_elems), np.uint16) for _ in range(2 * a["layers"])]
    table = np.full((a["rows"], a["max_blocks"]), -1, np.int32)
    bm = bmo.BlockManager(nb, a["block_size"], a["rows"], a["max_blocks"])
    done, spent, n = 0, 0.0, 0
    while spent < budget_s:
        t0 = time.perf_counter()
        r = n % a["rows"]
        assert bm.allocate(r, a["prompt"]) == bmo.OK
        ups, zero = bm.flush()
        bmo.apply_updates(table, caches, ups, zero, nb)
        bm.free(r)
        spent += time.perf_counter() - t0
        done += admission_bytes(len(ups), len(zero), len(caches), blk_elems * 2)
        n += 1
    return done / spent / 1e9, n, spent


def run_block_admission(args, rank: int, world: int, cpu_budget: float) -> dict:
    """Admission of new requests through the block manager: host allocation + flush, the copy of
    the staged writes, and kv_apply_block_updates (table writes + zero fill of every new block
    in every layer's K and V cache)."""
    import torch
    from paged_kv_cache_block_gb300 import kvcache as kv

    a = dict(ADMISSION, layers=args.layers or ADMISSION["layers"])
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    NB, n_caches = a["num_blocks"], 2 * a["layers"]
    pool = torch.ones((n_caches, NB, a["block_size"], a["num_kv_heads"], a["head_dim"]),
                      dtype=torch.bfloat16, device=dev)
    caches = [pool[i] for i in range(n_caches)]
    block_bytes = caches[0][0].numel() * 2
    table = torch.full((a["rows"], a["max_blocks"]), -1, dtype=torch.int32, device=dev)
    n_new = a["new_requests"] * a["prompt"] // a["block_size"]
    d_upd = torch.empty(n_new * 3, dtype=torch.int32, device=dev)
    d_zero = torch.empty(n_new, dtype=torch.int32, device=dev)
    h_upd = [torch.empty(n_new * 3, dtype=torch.int32).pin_memory() for _ in range(2)]
    h_zero = [torch.empty(n_new, dtype=torch.int32).pin_memory() for _ in range(2)]
    done_ev = [torch.cuda.Event(), torch.cuda.Event()]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    bm = kv.BlockManager(NB, a["block_size"], a["rows"], a["max_blocks"])
    host_s = []
    state = {"i": 0}

    def admit_step():
        i = state["i"] % 2
        state["i"] += 1
        done_ev[i].synchronize()          # the copy that last read this pinned buffer is done
        t0 = time.perf_counter()
        rows = [(state["i"] * a["new_requests"] + j) % a["rows"] for j in range(a["new_requests"])]
        st = bm.allocate_batch(rows, [a["prompt"]] * len(rows))
        assert (st == 0).all()
        u, z = bm.flush(h_upd[i], h_zero[i])
        for r in rows:              # the requests end at once: their blocks go back to the pool
            bm.free(r)
        host_s.append(time.perf_counter() - t0)
        nu, nz = u.shape[0], z.shape[0]
        d_upd[:3 * nu].copy_(h_upd[i][:3 * nu], non_blocking=True)
        d_zero[:nz].copy_(h_zero[i][:nz], non_blocking=True)
        done_ev[i].record(stream)
        kv.apply_block_updates(d_upd[:3 * nu].view(-1, 3), table, d_zero[:nz], caches, NB, d_err=err)
        return nu, nz

    for _ in range(args.warmup):
        nu, nz = admit_step()
    torch.cuda.synchronize()
    assert err.item() == 0 and nu == n_new and nz == n_new

    def timed(fn, n):
        return cuda_timed(fn, n, stream)

    # device value: the kernel on resident staged writes (the last flush), replayed as a CUDA
    # graph so that the Python call overhead stays out of the kernel's time
    launch = lambda: kv.apply_block_updates(d_upd.view(-1, 3), table, d_zero, caches, NB, d_err=err)  # noqa: E731
    launch()
    graph = torch.cuda.CUDAGraph()  # the K timed launches as one graph
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            launch()
    kernel = graph.replay
    kernel()
    torch.cuda.synchronize()
    ranks_barrier(world)
    clocks = ClockSampler(pci_of(dev))
    win = timed_windows(kernel, 1, stream, world, args.repeats)
    clk = clocks.stop()
    ms_kernel = statistics.median(win)
    ranks_barrier(world)
    host_s.clear()
    ms_e2e = timed(admit_step, args.steps)
    assert err.item() == 0
    ms_e2e, = ranks_max([ms_e2e], world, dev)

    # host manager cost of a decode-shaped step: 256 rows, one token each, then the flush
    dbm = kv.BlockManager(70000, a["block_size"], a["rows"], a["max_blocks"])
    rng = np.random.default_rng(0)
    lens = rng.integers(512, 8193, a["rows"])
    dbm.allocate_batch(np.arange(a["rows"]), lens)
    dbm.flush()
    hu = np.empty((a["rows"] * 2, 3), np.int32)
    hz = np.empty(a["rows"] * 2, np.int32)
    t0 = time.perf_counter()
    for _ in range(200):
        dbm.allocate_batch(np.arange(a["rows"]), np.ones(a["rows"], np.int32))
        dbm.flush(hu, hz)
    decode_us = (time.perf_counter() - t0) / 200 * 1e6

    bytes_step = admission_bytes(n_new, n_new, n_caches, block_bytes)
    peaks = measured_peaks()
    value = world * bytes_step * args.steps / (ms_kernel / 1e3) / 1e9
    result = {
        "metric": ADMISSION_METRIC,
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_kernel / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bytes)",
        "data": "synthetic (block manager trace: 16 requests of 2048 tokens admitted per step)",
        "config": admission_config(a["layers"]),
        "windows": window_summary(win, args.steps),
        "step_bytes": bytes_step,
        "roofline": {"kernel": "apply_block_updates_kernel (table writes + bulk-store zero fill)",
                     "bound": "hbm", "achieved": round(value / world, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(value / world / peaks["hbm_gbs"], 4),
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)",
                     "bytes_per_launch": bytes_step, "traffic": None},
        "e2e": {"value": round(world * bytes_step * args.steps / (ms_e2e / 1e3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(ms_e2e / args.steps, 4),
                "host_manager_us_per_step": round(1e6 * statistics.median(host_s), 1),
                "h2d_bytes_per_step": 16 * n_new, "d2h_bytes_per_step": 0},
        "host_decode_step_us": {"value": round(decode_us, 2),
                                "what": "kv_bm_allocate_batch of 256 rows x 1 token + kv_bm_flush"},
        "gpu_launches": args.steps * len(win),
        "gpu_launches_per_window": args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, n, spent = oracle_admission_rate(min(cpu_budget, 10.0))
        result["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                  "sample": f"{n} admissions of one 2048-token request (128 blocks x "
                                            f"{n_caches} caches), {spent:.1f} s (Python + numpy)"}
    del pool, caches
    return result


# ---------------------------------------------------------------- chunked prefill (tcgen05)

def prefill_flops(pw: W.PrefillWorkload) -> int:
    """Multiply-adds x 2 of the visible (query row, key) pairs only: q.K and p.V, D each, for
    every q head; masked pairs the kernel computes anyway are not counted."""
    s = pw.spec
    return int(4 * s.head_dim * s.num_q_heads * pw.visible_keys().sum())


def oracle_prefill_rate(pw: W.PrefillWorkload, budget_s: float, threads: int):
    """The oracle's varlen attention over a growing number of whole sequences until ~budget_s."""
    import oracle
    s = pw.spec
    NB, bs = pw.num_blocks, s.block_size
    kc = pw.pool_k.reshape(NB, bs, s.num_kv_heads, s.head_dim)
    vc = pw.pool_v.reshape(NB, bs, s.num_kv_heads, s.head_dim)
    vis = pw.visible_keys()
    order = np.argsort(pw.seq_lens)  # shortest first, so the sample fits the budget
    flops, spent, done = 0, 0.0, 0
    for b in order:
        if spent >= budget_s:
            break
        t0 = time.perf_counter()
        oracle.paged_attention_varlen(pw.q, s.dtype, kc, vc, s.dtype, pw.block_table, pw.seq_lens,
                                      pw.query_start_loc, s.softmax_scale, s.window, seqs=[int(b)],
                                      threads=threads)
        spent += time.perf_counter() - t0
        lo, hi = pw.query_start_loc[b], pw.query_start_loc[b + 1]
        flops += 4 * s.head_dim * s.num_q_heads * int(vis[lo:hi].sum())
        done += 1
    return flops / spent / 1e12, done, spent


def prefill_config(pw: W.PrefillWorkload) -> dict:
    """The config object of a prefill workload's line (both arms print the same one)."""
    s = pw.spec
    kv_bytes = 2 * int(pw.seq_lens.astype(np.int64).sum()) * s.num_kv_heads * s.head_dim * 2
    q_bytes = pw.num_tokens * s.num_q_heads * s.head_dim * 2
    return {"workload": s.name, "num_seqs": s.num_seqs, "num_q_heads": s.num_q_heads,
            "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size,
            "chunk": s.chunk, "context": s.context, "window": s.window,
            "tokens": pw.num_tokens, "seq_len_mean": round(float(pw.seq_lens.mean()), 1),
            "l2": f"no flush: each step reads {(kv_bytes + q_bytes) / 1e6:.0f} MB of q and cache and "
                  f"writes {q_bytes / 1e6:.0f} MB ({'more' if kv_bytes + q_bytes > 126e6 else 'less'} "
                  f"than the 126 MB L2)"}


def admission_config(layers: int) -> dict:
    """The config object of the block-admission line (both arms print the same one)."""
    a = dict(ADMISSION, layers=layers)
    n_caches = 2 * a["layers"]
    block_bytes = a["block_size"] * a["num_kv_heads"] * a["head_dim"] * 2
    n_new = a["new_requests"] * a["prompt"] // a["block_size"]
    return {"workload": "block_admission", **a, "caches": n_caches, "block_bytes": block_bytes,
            "new_blocks_per_step": n_new,
            "l2": f"no flush: each step writes {n_new * n_caches * block_bytes / 2**30:.2f} GiB of zeros"}


def run_prefill(args, name: str, rank: int, world: int, cpu_budget: float) -> dict:
    import torch
    from paged_kv_cache_block_gb300 import kvcache as kv

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    spec = W.PREFILL_BY_NAME[name]
    if args.num_seqs:
        spec = dataclasses.replace(spec, num_seqs=args.num_seqs)
    pw = W.make_prefill(spec)
    s = pw.spec
    shape = (pw.num_blocks, s.block_size, s.num_kv_heads, s.head_dim)
    kc = to_dev(pw.pool_k, s.dtype, dev).view(shape)
    vc = to_dev(pw.pool_v, s.dtype, dev).view(shape)
    q = to_dev(pw.q, s.dtype, dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    bt = torch.from_numpy(pw.block_table).to(dev)
    L = torch.from_numpy(pw.seq_lens).to(dev)
    qsl = torch.from_numpy(pw.query_start_loc).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    max_L, max_q = int(pw.seq_lens.max()), int(pw.chunks.max())

    def launch():
        kv.paged_attention_prefill(q, kc, vc, bt, L, qsl, max_L, max_q, s.softmax_scale, s.window,
                                   out=out, lse_out=lse, d_err=err)

    launch()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()  # the K timed launches as one graph
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            launch()
    graph.replay()
    torch.cuda.synchronize()
    if err.item() != 0:
        raise RuntimeError(f"device error bits {err.item()}")

    ranks_barrier(world)
    clocks = ClockSampler(pci_of(dev))
    win = timed_windows(graph.replay, 1, stream, world, args.repeats)
    clk = clocks.stop()
    ms = statistics.median(win)
    ranks_barrier(world)

    # end to end: every step's queries and metadata from pinned host memory, its output back
    # (HostPipe: one copy each way, double-buffered on copy streams)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[s.dtype]
    pipe = HostPipe(dev, dict(q=(pw.q, tdt), bt=(pw.block_table, torch.int32), L=(pw.seq_lens, torch.int32),
                              qsl=(pw.query_start_loc, torch.int32)),
                    dict(out=(tdt, tuple(out.shape))))

    def e2e(t):
        kv.paged_attention_prefill(t["q"], kc, vc, t["bt"], t["L"], t["qsl"], max_L, max_q, s.softmax_scale,
                                   s.window, out=t["out"], lse_out=lse, d_err=err)

    pipe.run(max(1, args.warmup), e2e, stream)
    ms_e2e = pipe.run(args.steps, e2e, stream)
    if err.item() != 0:
        raise RuntimeError(f"device error bits {err.item()}")
    if not torch.equal(pipe.output((args.steps - 1) & 1, "out").view(torch.int16), out.cpu().view(torch.int16)):
        raise RuntimeError("end-to-end outputs differ from the resident launch's")
    ms_e2e, = ranks_max([ms_e2e], world, dev)

    flops = prefill_flops(pw)
    tflops = world * flops * args.steps / (ms / 1e3) / 1e12
    peak = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else None
    peak_tf = peak["bf16_tflops"] if peak else 1900.0
    result = {
        "metric": PREFILL_METRIC,
        "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": s.dtype,
        "data": "synthetic (seeded N(0,1), block tables from a seeded permutation)",
        "config": prefill_config(pw),
        "windows": window_summary(win, args.steps),
        "flops_per_step": flops,
        "prefill_tokens_per_s": round(world * pw.num_tokens * args.steps / (ms / 1e3), 1),
        "roofline": {"kernel": "prefill_attention_kernel (tcgen05.mma, TMEM accumulators, TMA), CUDA graph replay",
                     "bound": "tensor", "achieved": round(tflops / world, 2), "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(tflops / world / peak_tf, 4),
                     "peak_source": ("measured (MEASURED_PEAKS.json bf16_tflops, burst)" if peak
                                     else "fallback"),
                     "flops_per_launch": flops, "traffic": None},
        "e2e": {"value": round(world * flops * args.steps / (ms_e2e / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(ms_e2e / args.steps, 4),
                "h2d_bytes_per_step": pipe.h2d_bytes, "d2h_bytes_per_step": pipe.d2h_bytes,
                "how": "eager API call; each step's q, block table, lengths and query offsets in one "
                       "pinned buffer, one upload and one download a step on copy streams, two device "
                       "sets alternating so copies overlap the neighbouring steps"},
        "gpu_launches": args.steps * len(win),
        "gpu_launches_per_window": args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = host_cores()
        tf, n, spent = oracle_prefill_rate(pw, min(cpu_budget, 20.0), threads)
        result["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                  "sample": f"{n} of {s.num_seqs} sequences (shortest first), all heads, "
                                            f"{spent:.1f} s (C, fp64, pthreads)"}
    del q, out, kc, vc, pipe
    return result


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama3_8b",
                    choices=sorted(W.BY_NAME) + sorted(W.PREFILL_BY_NAME) + ["block_admission"])
    ap.add_argument("--workers", type=int, default=0, help="persistent CTAs (0 = one per SM)")
    ap.add_argument("--mode", default=None, choices=["fused", "calls"],
                    help="fused: kv_decode_step, one launch per layer; calls: the three calls "
                         "(default: fused, except calls for INT4 caches, where it measures faster)")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="smaller batch of the same shape (profiling captures only; not a bench line)")
    ap.add_argument("--layers", type=int, default=0,
                    help="block_admission: layers whose K and V caches are zero-filled (default 32)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--other-cpu-budget", type=float, default=4.0,
                    help="seconds of oracle time for each other workload's cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed windows of --steps steps each (at least; more until ~200 ms are timed)")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="the default workload's line without the other workloads' figures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    args.repeats = max(1, args.repeats)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    # the other workloads ride along on the default run (the headline workload at full size)
    args.other_configs = (args.workload == "llama3_8b" and not args.num_seqs and not args.no_other_configs
                          and "--workload" not in sys.argv)

    if args.impl == "reference":
        return run_reference(args, rank, world)

    ranks_init(world)
    result = measure(args, args.workload, rank, world)
    if args.other_configs and world == 1:
        # the other workloads of the specification (and the widened rows), each measured in this
        # same run with its own roofline, end-to-end figure and oracle baseline
        import torch
        others = {}
        for name in OTHER_CONFIGS:
            if name == args.workload:
                continue
            torch.cuda.empty_cache()
            others[name] = summary(measure(args, name, rank, world, cpu_budget=args.other_cpu_budget))
        result["other_configs"] = others
    if rank == 0:
        print(json.dumps(result))
    ranks_done(world)


# the workloads measured beside the headline one: the specification's other decode batches, the
# INT4 cache, chunked prefill and block admission
OTHER_CONFIGS = ["opt125m", "llama70b_fp8", "mistral_hybrid", "llama3_8b_int4", "prefill_llama3_8b",
                 "prefill_prompt_llama3_8b", "block_admission"]


def summary(r: dict) -> dict:
    """The figures of a workload's full result line that the headline line carries for it."""
    keep = ("metric", "value", "unit", "ms_per_step", "dtype", "config", "windows", "roofline", "e2e",
            "cpu_baseline", "clocks", "gpu_launches")
    return {k: r[k] for k in keep if k in r}


def measure(args, name: str, rank: int, world: int, cpu_budget=None) -> dict:
    """One workload's result line (not printed)."""
    if cpu_budget is None:
        cpu_budget = args.cpu_budget
    if name == "block_admission":
        return run_block_admission(args, rank, world, cpu_budget)
    if name in W.PREFILL_BY_NAME:
        return run_prefill(args, name, rank, world, cpu_budget)
    return decode_result(args, name, rank, world, cpu_budget)


def decode_config(wl: W.Workload, args, world: int, attn_bytes: int, mode: str) -> dict:
    """The config object of a decode workload's line (both arms print the same one)."""
    s = wl.spec
    return {"workload": s.name, "num_seqs": s.num_seqs, "q_len": s.q_len,
            "num_q_heads": s.num_q_heads, "num_kv_heads": s.num_kv_heads,
            "head_dim": s.head_dim, "block_size": s.block_size, "num_blocks": wl.num_blocks,
            "seq_len_mean": round(float(wl.seq_lens.mean()), 1), "max_seq_len": wl.max_seq_len,
            "layers": [l.window for l in wl.layers], "num_workers": args.workers or "one per SM",
            "parallelism": f"replicas x{world} (independent batches)",
            "l2": f"no flush: each step reads {attn_bytes / 1e6:.0f} MB of cache, q and table "
                  f"({'more' if attn_bytes > 126e6 else 'less'} than the 126 MB L2)",
            "step": "slot mapping + cache write + paged attention (+ lse merge) per layer",
            "mode": mode}


def decode_mode(args, name: str) -> str:
    if args.mode is not None:
        return args.mode
    return "calls" if W.BY_NAME[name].cache_dtype == "int4" else "fused"


def decode_result(args, name: str, rank: int, world: int, cpu_budget: float) -> dict:
    mode = decode_mode(args, name)
    margs = argparse.Namespace(**{**vars(args), "mode": mode})
    r = run_gpu(margs, name, rank, world)
    wl, clk, layers = r["wl"], r["clk"], r["layers"]
    acc = algorithmic_bytes(wl)
    step_bytes = acc["step"]
    K = args.steps
    ms_total = statistics.median(r["win_step"])
    ms_step = ms_total / K
    value = world * step_bytes * K / (ms_total / 1e3) / 1e9
    tokens = wl.num_tokens
    attn_bytes = sum(l["attention"] for l in acc["layers"])
    n_layers = len(wl.layers)
    # the dominant kernel: the fused step kernel (all of a layer's bytes) or the attention call,
    # its time per launch from the median window of the attention graph
    per_launch_ms = statistics.median(r["win_attn"]) / K / n_layers
    kernel_bytes = step_bytes if mode == "fused" else attn_bytes
    per_launch_bytes = kernel_bytes / n_layers
    peaks = measured_peaks()
    achieved = per_launch_bytes / (per_launch_ms / 1e3) / 1e9
    traffic = profiled_traffic(name)
    s = wl.spec
    # calls: slot mapping; per layer cache write, attention, merge.  fused: per layer the decode
    # kernel (slot mapping, cache write and attention) and the merge
    launches_per_step = 2 * n_layers if mode == "fused" else 1 + 3 * n_layers
    model_layers = MODEL_LAYERS.get(s.name.split("_int4")[0], 1)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": s.dtype if s.cache_dtype == s.dtype else f"{s.dtype}+{s.cache_dtype}",
        "data": "synthetic (seeded N(0,1), block tables from a seeded permutation)",
        "config": decode_config(wl, args, world, attn_bytes, mode),
        "windows": window_summary(r["win_step"], K),
        "step_bytes": step_bytes,
        "attention_bytes_per_step": attn_bytes,
        "decode_tokens_per_s": round(world * tokens * K / (ms_total / 1e3), 1),
        # per attention layer (the step holds n_layers of them), and as context divided by the
        # attention layers of the model the workload is shaped after
        "decode_tokens_per_s_per_layer": round(world * tokens * K * n_layers / (ms_total / 1e3), 1),
        "decode_tokens_per_s_model_layers": {
            "layers": model_layers,
            "value": round(world * tokens * K * n_layers / (ms_total / 1e3) / model_layers, 1)},
        "logical_kv_bytes_per_step": sum(l["logical_kv"] for l in acc["layers"]),
        "write_path_us": {"value": round(r["us_write"], 2),
                          "what": "kv_compute_slot_mapping + cache write of one layer's new tokens, CUDA graph replay"},
        "kernel_ms_per_step": round(per_launch_ms * n_layers, 4),
        "timing": "each timed window replays one CUDA graph of the K steps (value) or of the K steps' "
                  "attention calls (roofline); median over the windows; e2e and eager_ms_per_step are "
                  "plain API calls",
        "eager_ms_per_step": round(r["ms_eager"] / K, 4),
        "pct_hbm_peak_step": round(100 * value / world / peaks["hbm_gbs"], 2),
        "roofline": {"kernel": (("paged_decode_int4_kernel" if s.cache_dtype == "int4" else "paged_decode_kernel") +
                                ", fused step (slot mapping + cache write + attention + merge)"
                                if mode == "fused" else
                                ("kv_paged_attention_decode_int4" if s.cache_dtype == "int4" else
                                 "kv_paged_attention_decode") + " (attention + merge)") + ", CUDA graph replay",
                     "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                     "bytes_per_launch": per_launch_bytes, "traffic": traffic},
        "e2e": {"value": round(world * step_bytes * K / (r["ms_e2e"] / 1e3) / 1e9, 2), "unit": UNIT,
                "ms_per_step": round(r["ms_e2e"] / K, 4), "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"],
                "how": "eager API calls; each step's inputs (table, lengths, positions, q, new K/V) in "
                       "one pinned buffer, one upload and one download a step on copy streams, two "
                       "device sets alternating so copies overlap the neighbouring steps"},
        "gpu_launches": launches_per_step * K * len(r["win_step"]),
        "gpu_launches_per_window": launches_per_step * K,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = host_cores()
        gbs, nseq, spent = oracle_sample_rate(wl, cpu_budget, threads)
        gbs1, nseq1, spent1 = oracle_sample_rate(wl, max(1.0, cpu_budget / 4), 1)
        result["cpu_baseline"] = {"value": round(gbs, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                                  "sample": f"{nseq} of {wl.spec.num_seqs} sequences, every layer, "
                                            f"{spent:.1f} s of oracle time (C, fp64, pthreads)",
                                  "cores_1": {"value": round(gbs1, 4), "unit": UNIT,
                                              "sample": f"{nseq1} of {wl.spec.num_seqs} sequences, every "
                                                        f"layer, {spent1:.1f} s on one thread"}}
    del layers, r
    return result


def run_reference(args, rank: int, world: int):
    """The reference arm: the CPU oracle on the host cores, same workload, metric and unit."""
    if rank != 0:
        return
    if args.workload in W.PREFILL_BY_NAME or args.workload == "block_admission":
        return run_reference_other(args, world)
    wl = W.make_workload(W.BY_NAME[args.workload])
    attn_bytes = sum(l["attention"] for l in algorithmic_bytes(wl)["layers"])
    threads = host_cores()
    times, bytes_done, seqs = [], [], []
    for i in range(args.warmup + args.steps):
        gbs, nseq, spent = oracle_sample_rate(wl, 2.0, threads)
        if i >= args.warmup:
            times.append(spent)
            bytes_done.append(gbs * spent * 1e9)
            seqs.append(nseq)
    value = sum(bytes_done) / sum(times) / 1e9
    s = wl.spec
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * sum(times) / len(times), 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1), block tables from a seeded permutation)",
           "config": decode_config(wl, args, world, attn_bytes, decode_mode(args, args.workload)),
           "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                            "sample": f"each step: {int(np.median(seqs))} of {s.num_seqs} sequences, "
                                      f"{statistics.median(times):.2f} s"},
           "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def run_reference_other(args, world: int):
    """The reference arm for the prefill and block-admission workloads: their oracle rates."""
    threads = host_cores()
    prefill = args.workload in W.PREFILL_BY_NAME
    pw = W.make_prefill(W.PREFILL_BY_NAME[args.workload]) if prefill else None
    rates, times, units = [], [], []
    for i in range(args.warmup + args.steps):
        if prefill:
            rate, n, spent = oracle_prefill_rate(pw, 2.0, threads)
        else:
            rate, n, spent = oracle_admission_rate(2.0)
        if i >= args.warmup:
            rates.append(rate * spent)
            times.append(spent)
            units.append(n)
    value = sum(rates) / sum(times)
    unit = "TFLOP/s" if prefill else "GB/s"
    cores = threads if prefill else 1
    what = "sequences" if prefill else "admissions of one 2048-token request"
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC if prefill else ADMISSION_METRIC,
        "value": round(value, 6), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64" if prefill else "u16 (bytes)", "data": "synthetic",
        "config": prefill_config(pw) if prefill else admission_config(args.layers or ADMISSION["layers"]),
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": f"each step: {int(np.median(units))} {what}, {statistics.median(times):.2f} s"},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


if __name__ == "__main__":
    main()
