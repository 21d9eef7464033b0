"""Failure path on the GPU, without a fault: a bounded device-side wait that gives up.

The tensor-core encoder's pipeline waits on mbarriers with a time limit; when a wait runs out the
kernel records MP_ERR_TIMEOUT in the device status word instead of hanging. Here the library's test
hook runs that same bounded wait on a barrier that nothing completes (no copy, no MMA), with a
limit of a few milliseconds; the status must come back once as a timeout, then read clean, and the
next decode must run normally on the same context.
"""
import time

import numpy as np
import pytest
import torch

from workloads import make_hyperplanes, make_layer, small_workload

pytestmark = pytest.mark.gpu

MP_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lsh_sampled_sparse_gb300 as mp
    mp.lib()
    return mp


def test_wait_that_runs_out_reports_a_timeout_and_the_context_stays_usable(mp):
    wl = small_workload(B=1, Hq=8, Hkv=2, n=4000, index=960)
    x = {k: v.cuda() for k, v in make_layer(wl).items()}
    W = make_hyperplanes(wl).cuda()
    c = mp.key_mean(x["keys"])
    codes = mp.build_tables(x["keys"], c, W, wl.K, wl.L)
    args = (wl.K, wl.L, wl.n_sink, wl.n_local)
    before = mp.decode_attention(x["q"], codes, c, W, x["keys"], x["values"], *args)
    assert mp.device_status() == 0
    t0 = time.perf_counter()
    mp.debug_wait_expiry(3000)                          # gives up after 3 ms
    assert mp.device_status() == MP_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.003
    assert mp.device_status() == 0                      # read once, then reset
    after = mp.decode_attention(x["q"], codes, c, W, x["keys"], x["values"], *args)
    torch.cuda.synchronize()
    assert mp.device_status() == 0
    assert torch.equal(before, after)
    assert np.all(np.isfinite(after.cpu().numpy()))


def test_wait_limit_is_checked_on_the_host(mp):
    for bad in (0, -5, 100001):
        with pytest.raises(mp.MagicPIGError):
            mp.debug_wait_expiry(bad)
    assert mp.device_status() == 0
