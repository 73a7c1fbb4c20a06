"""The allocation-free linear entry point against the workspace one and the oracle.

spec_verify_linear_noalloc serves callers that can neither allocate device
memory nor hand the library a workspace (an op living inside a host runtime
that owns the GPU's memory, a plugin given only its inputs and outputs).  Its
split-K scratch is a static device array inside the library, so these checks
run it twice in a row (the array keeps the previous call's contents) and
compare each result with spec_verify_linear on the same inputs and with the
fp64 oracle.  The cases are chosen so that the scratch is really used: the
plans of the default options need none for most small shapes, so each case
states the plan it forces and asserts a non-zero scratch need.  The file is
named to be collected last.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import bf16 as obf, ops as oops

from gpu_util import assert_close_rel, bf16_dev, bits_of, f64_of_bf16

pytestmark = pytest.mark.gpu

LIMIT = 16 << 20


def _case(seed, M, N, K, residual):
    X = synth.normal_bf16_bits(seed, (M, K), 1.0)
    W = synth.normal_bf16_bits(seed + 1, (N, K), 0.02)
    R = synth.normal_bf16_bits(seed + 2, (M, N), 1.0) if residual else None
    oracle = oops.linear(obf.decode(X), obf.decode(W), obf.decode(R) if residual else None)
    return bf16_dev(X), bf16_dev(W), (bf16_dev(R) if residual else None), oracle


class _options:
    """Library knobs set for one case and restored afterwards."""

    def __init__(self, lib, **kw):
        self.lib, self.kw = lib, kw

    def __enter__(self):
        for k, v in self.kw.items():
            self.lib.spec_set_option(k, v)

    def __exit__(self, *exc):
        self.lib.spec_set_option("gemv_max_m", 0)
        self.lib.spec_set_option("linear_cluster", 1)
        self.lib.spec_set_option("linear_pair", 1)
        self.lib.spec_set_option("persistent_grid", 0)


# (M, N, K, options, plan): every case needs 0 < scratch <= 16 MiB
CASES = [
    (32, 4096, 4096, dict(linear_cluster=0), "tensor cores, 32 tiles over 152 CTAs: stream-K pieces + reduce"),
    (16, 4096, 4096, dict(linear_cluster=0), "tensor cores, every tile split about 5 ways"),
    (64, 1000, 4096, dict(linear_cluster=0, persistent_grid=37), "ragged N, forced grid of 37 CTAs"),
    (4, 2048, 12288, dict(gemv_max_m=4), "CUDA cores, K split, arrival counters at the start of the scratch"),
    (1, 4096, 4096, dict(gemv_max_m=4), "CUDA cores at one row"),
]


@pytest.mark.parametrize("M,N,K,opts,plan", CASES)
def test_noalloc_uses_the_static_scratch_and_matches_twice(lib, M, N, K, opts, plan):
    X, W, R, oracle = _case(M + N + K, M, N, K, residual=True)
    with _options(lib, **opts):
        need = lib.spec_linear_workspace_bytes(M, N, K)
        assert 0 < need <= LIMIT, (plan, need)
        ref = lib.spec_verify_linear(X, W, residual=R)
        lib.spec_device_status()
        for _ in range(2):              # the second call finds the scratch the first one left
            Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            lib.spec_verify_linear_noalloc(X, W, Y, residual=R)
            lib.spec_device_status()
            # same plan, same arithmetic: identical bits to the workspace entry point
            assert np.array_equal(bits_of(Y), bits_of(ref)), plan
            assert_close_rel(f64_of_bf16(Y), oracle, f"noalloc {plan}")


@pytest.mark.parametrize("M,N,K", [(3, 1024, 4096), (5, 4096, 4096), (16, 640, 1000)])
def test_noalloc_without_scratch_need(lib, M, N, K):
    """Default plans that need no scratch (cluster split-K sums on chip): still correct twice."""
    X, W, R, oracle = _case(M * 3 + N, M, N, K, residual=True)
    ref = f64_of_bf16(lib.spec_verify_linear(X, W, residual=R))
    for _ in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        lib.spec_verify_linear_noalloc(X, W, Y, residual=R)
        lib.spec_device_status()
        assert_close_rel(f64_of_bf16(Y), ref, f"noalloc M={M} N={N} K={K}")
        assert_close_rel(f64_of_bf16(Y), oracle, f"noalloc vs oracle M={M} N={N} K={K}")


def test_noalloc_back_to_back_different_plans(lib):
    """A CUDA-core split-K call, then a stream-K call, with no host sync in between: each clears
    the counters it needs before its kernels run."""
    a = _case(1, 4, 2048, 12288, residual=False)
    b = _case(2, 40, 4096, 4096, residual=True)
    outs = []
    with _options(lib, gemv_max_m=4, linear_cluster=0):
        assert lib.spec_linear_workspace_bytes(4, 2048, 12288) > 0
        assert lib.spec_linear_workspace_bytes(40, 4096, 4096) > 0
        for X, W, R, _ in (a, b, a):
            Y = torch.empty((X.shape[0], W.shape[0]), dtype=torch.bfloat16, device="cuda")
            outs.append(lib.spec_verify_linear_noalloc(X, W, Y, residual=R))
        lib.spec_device_status()
    for y, (_, _, _, oracle) in zip(outs, (a, b, a)):
        assert_close_rel(f64_of_bf16(y), oracle, "noalloc back to back")
    assert np.array_equal(bits_of(outs[0]), bits_of(outs[2]))


def test_noalloc_rejects_scratch_beyond_the_limit(lib):
    M, N, K = 368, 24576, 4096                         # 192 tiles of 368 rows, stream-K split
    # (the pair plan and the whole tiles + cluster remainder plan need no scratch: both off)
    with _options(lib, linear_cluster=0, linear_pair=0):
        need = lib.spec_linear_workspace_bytes(M, N, K)
        assert need > LIMIT
        big_x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
        big_w = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
        Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(lib.SpecError) as e:
            lib.spec_verify_linear_noalloc(big_x, big_w, Y)
        assert e.value.code == lib.SPEC_EUNSUPPORTED
        torch.cuda.synchronize()
        assert torch.count_nonzero(Y) == 0


def test_noalloc_rejects_bad_arguments_before_any_work(lib):
    """A call rejected by its argument checks enqueues nothing (not even the scratch clear)."""
    X, W, _, _ = _case(5, 32, 4096, 4096, residual=False)
    Y = torch.zeros((32, 4096), dtype=torch.bfloat16, device="cuda")
    R_bad = torch.zeros((32, 4097), dtype=torch.bfloat16, device="cuda")[:, 1:]   # 2 bytes off
    with _options(lib, linear_cluster=0):
        with pytest.raises(lib.SpecError) as e:
            lib.spec_verify_linear_noalloc(X, W, Y, residual=R_bad)
        assert e.value.code == lib.SPEC_EINVAL
        assert lib._lib.spec_launches() == 0
    torch.cuda.synchronize()
    assert torch.count_nonzero(Y) == 0
