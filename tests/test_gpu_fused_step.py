"""kv_decode_step (slot mapping, cache write, attention and merge in one cooperative launch)
against the three separate calls (bit for bit: same slots, same cache bytes, same outputs) and
against the CPU oracle (specification tolerances)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_block_gb300 import workloads as W
from tests import harness as H
from tests.test_gpu_parity import SMALL, _spec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from paged_kv_cache_block_gb300 import kvcache
    return kvcache


def _compare(wl, layer, num_workers=0, seqs=None):
    kc, vc = H.gpu_fill_cache(wl, layer)
    sep = H.gpu_step(wl, layer, kc, vc, num_workers=num_workers)
    kc2, vc2 = H.gpu_fill_cache(wl, layer)
    fus = H.gpu_step_fused(wl, layer, kc2, vc2, num_workers=num_workers)
    assert fus.err == sep.err == 0
    assert torch.equal(fus.slots, sep.slots)
    assert torch.equal(kc2.view(torch.uint8), kc.view(torch.uint8))
    assert torch.equal(vc2.view(torch.uint8), vc.view(torch.uint8))
    assert torch.equal(fus.out, sep.out)
    assert torch.equal(fus.lse, sep.lse)
    o = H.oracle_step(wl, layer, seqs=seqs)
    if seqs is None:
        H.check_whole_cache(fus, o)
    H.check_attention(wl, fus, o, rows=None if seqs is None else H.rows_of(wl, seqs))


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("num_workers", [0, 5])
def test_fused_step_small_configs(kv, name, num_workers):
    wl = W.make_workload(SMALL[name])
    for layer in wl.layers:
        _compare(wl, layer, num_workers)


@pytest.mark.parametrize("kw", [
    dict(block_size=4, head_dim=64, dtype="f16", cache_dtype="f16"),
    dict(block_size=32, head_dim=128, dtype="bf16", cache_dtype="bf16"),
    dict(num_q_heads=32, num_kv_heads=4, q_len=8),
    dict(q_len=4, windows=(37,)),
    dict(dtype="f16", cache_dtype="e4m3", num_q_heads=16, num_kv_heads=2),
    dict(dtype="bf16", cache_dtype="e4m3", num_q_heads=16, num_kv_heads=2, block_size=8, q_len=2),
    dict(dtype="bf16", cache_dtype="e4m3", num_q_heads=64, num_kv_heads=8, block_size=32),
    dict(dtype="bf16", cache_dtype="e4m3", num_q_heads=64, num_kv_heads=8, block_size=16, windows=(100,)),
])
def test_fused_step_shapes(kv, kw):
    wl = W.make_workload(_spec(lengths=("fixed", (9, 40, 333, 1000)), **kw))
    _compare(wl, wl.layers[0], num_workers=11)


@pytest.mark.parametrize("name", ["opt125m", "llama3_8b", "llama70b_fp8", "mistral_hybrid"])
def test_fused_step_full_size_benchmark_configs(kv, name):
    """The benchmark's fused workloads at full size: every layer equal to the separate calls bit
    for bit, the whole cache equal to the oracle's, and every output and lse row against the
    oracle."""
    wl = W.make_workload(W.BY_NAME[name])
    for layer in wl.layers:
        _compare(wl, layer)
        torch.cuda.empty_cache()


def test_fused_step_error_bits_match_separate_calls(kv):
    wl = W.make_workload(_spec(lengths=("fixed", (10, 300, 40, 64)), q_len=2))
    layer = wl.layers[0]
    wl.block_table[1, (300 - 1) // 16] = -5          # the block of sequence 1's new tokens
    kc, vc = H.gpu_fill_cache(wl, layer)
    sep = H.gpu_step(wl, layer, kc, vc)
    kc2, vc2 = H.gpu_fill_cache(wl, layer)
    fus = H.gpu_step_fused(wl, layer, kc2, vc2)
    assert sep.err == fus.err and fus.err & kv.KV_DERR_BAD_BLOCK
    assert torch.equal(fus.slots, sep.slots) and (fus.slots[2:4] == -1).all()
    assert torch.equal(fus.out, sep.out)


def test_fused_step_many_workers(kv):
    """More workers than SMs and than stages: empty shares, sequences cut in many pieces."""
    wl = W.make_workload(_spec(lengths=("fixed", (9, 40, 333, 1000)), q_len=3))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _compare(wl, wl.layers[0], num_workers=sms * 3)
