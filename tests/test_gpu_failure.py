"""Failure reporting without a GPU fault: a bounded in-kernel wait that expires
records KVP_ERR_DEVICE_TIMEOUT in the device status word, the kernel returns,
and the context stays usable (the next calls run and are bit-exact).  The
expired wait is the library's self-test (one thread, a barrier that nothing
arrives on, the kernels' own wait with a 2 ms limit); no kernel traps,
faults or spins without a bound."""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_125_gb300 as kvp

from parity import BF16_NAN, u16

pytestmark = pytest.mark.gpu

TIMEOUT = -5  # KVP_ERR_DEVICE_TIMEOUT


def _store_round_trip(seed):
    """A small kv_store through the C ABI, bit-exact against the oracle."""
    nb, bs, hkv, d, n = 8, 16, 2, 64, 40
    g = torch.Generator().manual_seed(seed)
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int32)
    k = torch.randn((n, hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((n, hkv, d), generator=g).to(torch.bfloat16)
    kc = torch.full((nb, bs, hkv, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    kvp.kv_store(k.cuda(), v.cuda(), slots.cuda(), kc, vc)
    torch.cuda.synchronize()
    kr = np.full((nb, bs, hkv, d), BF16_NAN, np.uint16)
    vr = kr.copy()
    oracle.kv_store(k, v, slots, kr, vr)
    return np.array_equal(u16(kc), kr) and np.array_equal(u16(vc), vr)


def test_wait_that_is_satisfied_records_nothing():
    kvp.device_status()
    kvp.selftest_wait(arrive=True)
    torch.cuda.synchronize()
    assert kvp.device_status() == 0


def test_expired_wait_reports_timeout_and_the_context_stays_usable():
    kvp.device_status()
    t0 = time.perf_counter()
    kvp.selftest_wait(arrive=False)
    torch.cuda.synchronize()  # returns: the wait gave up after its limit
    elapsed = time.perf_counter() - t0
    assert kvp.device_status() == TIMEOUT
    assert elapsed >= 0.002 * 0.9  # it did wait its limit before giving up
    assert kvp.device_status() == 0  # the read cleared the word
    # same stream, same context: later calls run and are exact
    assert _store_round_trip(3)
    assert kvp.device_status() == 0


def test_timeout_is_recorded_once_and_first_error_wins():
    """Two expired waits in a row leave one timeout code; the status word keeps
    the first error until it is read."""
    kvp.device_status()
    kvp.selftest_wait(arrive=False)
    kvp.selftest_wait(arrive=False)
    torch.cuda.synchronize()
    assert kvp.device_status() == TIMEOUT
    assert kvp.device_status() == 0
