"""The failure path of the library's waits, on the GPU without a fault: a kernel waits (with the
bounded wait every kernel uses) on an mbarrier phase that nothing completes; after its limit it
must report KV_DERR_TIMEOUT and return, and the device context must stay usable."""
import numpy as np
import pytest
import torch

from paged_kv_cache_block_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from paged_kv_cache_block_gb300 import kvcache
    return kvcache


@pytest.mark.parametrize("limit_us", [2000, 20000])
def test_wait_runs_out_and_reports(kv, limit_us):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kv.selftest_bounded_wait(limit_us, err, waited)
    torch.cuda.synchronize()
    assert err.item() == kv.KV_DERR_TIMEOUT
    assert limit_us <= waited.item() < limit_us + 100000


def test_context_usable_after_a_timeout(kv):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.selftest_bounded_wait(1000, err)
    wl = W.make_workload(W.TINY)
    layer = wl.layers[0]
    kc, vc = H.gpu_fill_cache(wl, layer)
    g = H.gpu_step(wl, layer, kc, vc)
    o = H.oracle_step(wl, layer)
    assert err.item() == kv.KV_DERR_TIMEOUT and g.err == 0
    assert np.array_equal(g.slots.cpu().numpy(), o.slots)
    H.check_attention(wl, g, o)


def test_host_checks(kv):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0, 1000001):
        with pytest.raises(kv.KVError) as e:
            kv.selftest_bounded_wait(bad, err)
        assert e.value.status == kv.KV_ERR_INVALID_ARG
