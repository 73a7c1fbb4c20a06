"""Failure detection on the GPU without faulting it: a bounded device wait that runs out.

Every TMA / MMA pipeline of the library waits on mbarriers through one bounded wait routine that,
after its limit, records a site code in the library's status word and returns, so the kernel ends
and the context stays usable.  spec_probe_bounded_wait runs that routine on an mbarrier that nothing
arrives at (the failure: a producer that never delivers), with a short limit.
"""
import time

import pytest

import synth
from oracle import bf16 as obf, ops as oops

from gpu_util import assert_close_rel, bf16_dev, f64_of_bf16

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_reports_and_clears(lib):
    lib.spec_device_status()                        # start from a clear status word
    t0 = time.perf_counter()
    lib.spec_probe_bounded_wait(2000, arrive=False)     # 2 ms limit, nothing arrives
    rc, site = lib.spec_device_status_code()
    elapsed = time.perf_counter() - t0
    assert rc == lib.SPEC_ETIMEOUT, rc
    assert site == lib.PROBE_WAIT_SITE
    assert elapsed < 1.0, elapsed                   # the wait gave up; nothing hung
    # reading the status cleared it
    assert lib.spec_device_status_code() == (lib.SPEC_OK, 0)
    # the raising form names the timeout
    lib.spec_probe_bounded_wait(500, arrive=False)
    with pytest.raises(lib.SpecError) as e:
        lib.spec_device_status()
    assert e.value.code == lib.SPEC_ETIMEOUT and "0x1e1" in str(e.value)
    assert lib.spec_device_status_code() == (lib.SPEC_OK, 0)


def test_bounded_wait_that_completes_leaves_status_clear(lib):
    lib.spec_device_status()
    lib.spec_probe_bounded_wait(4000, arrive=True)      # a second warp arrives after ~1 ms
    assert lib.spec_device_status_code() == (lib.SPEC_OK, 0)


def test_context_usable_after_a_timeout(lib):
    lib.spec_probe_bounded_wait(1000, arrive=False)
    assert lib.spec_device_status_code()[0] == lib.SPEC_ETIMEOUT
    M, N, K = 7, 640, 1024
    X = synth.normal_bf16_bits(11, (M, K), 1.0)
    W = synth.normal_bf16_bits(12, (N, K), 0.05)
    Y = lib.spec_verify_linear(bf16_dev(X), bf16_dev(W))
    lib.spec_device_status()
    assert_close_rel(f64_of_bf16(Y), oops.linear(obf.decode(X), obf.decode(W)), "linear after a timeout")
