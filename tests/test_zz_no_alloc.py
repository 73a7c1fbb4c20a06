"""The allocation-free linear entry point against the workspace one.

spec_verify_linear_noalloc serves callers that can neither allocate device
memory nor hand the library a workspace (an op living inside a host runtime
that owns the GPU's memory, a plugin given only its inputs and outputs).  Its
split-K scratch is a static device array inside the library, so these checks
run it twice in a row (the array keeps the previous call's contents) and
compare each result with spec_verify_linear on the same inputs.  The file is
named to be collected last.
"""
import pytest
import torch

import synth

from gpu_util import assert_close_rel, bf16_dev, f64_of_bf16

pytestmark = pytest.mark.gpu


def _case(seed, M, N, K, residual):
    X = bf16_dev(synth.normal_bf16_bits(seed, (M, K), 1.0))
    W = bf16_dev(synth.normal_bf16_bits(seed + 1, (N, K), 0.02))
    R = bf16_dev(synth.normal_bf16_bits(seed + 2, (M, N), 1.0)) if residual else None
    return X, W, R


@pytest.mark.parametrize("M,N,K", [(3, 1024, 4096), (5, 4096, 4096), (16, 640, 1000)])
def test_noalloc_matches_workspace_entry_point_twice(lib, M, N, K):
    assert lib.spec_linear_workspace_bytes(M, N, K) <= 16 << 20
    X, W, R = _case(M + N, M, N, K, residual=True)
    ref = f64_of_bf16(lib.spec_verify_linear(X, W, residual=R))
    for _ in range(2):                  # the second call reuses the scratch left by the first
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        lib.spec_verify_linear_noalloc(X, W, Y, residual=R)
        lib.spec_device_status()
        assert_close_rel(f64_of_bf16(Y), ref, f"noalloc M={M} N={N} K={K}")


def test_noalloc_back_to_back_different_shapes(lib):
    a = _case(1, 4, 2048, 12288, residual=False)      # CUDA-core path, K split 24 ways
    b = _case(2, 9, 6144, 4096, residual=True)         # tensor-core path, K split
    refs = [f64_of_bf16(lib.spec_verify_linear(X, W, residual=R)) for X, W, R in (a, b)]
    outs = []
    for X, W, R in (a, b):
        Y = torch.empty((X.shape[0], W.shape[0]), dtype=torch.bfloat16, device="cuda")
        outs.append(lib.spec_verify_linear_noalloc(X, W, Y, residual=R))
    lib.spec_device_status()
    for y, r in zip(outs, refs):
        assert_close_rel(f64_of_bf16(y), r, "noalloc back to back")


def test_noalloc_rejects_scratch_beyond_the_limit(lib):
    M, N, K = 368, 24576, 4096                         # 192 tiles of 368 rows, stream-K split
    lib.spec_set_option("linear_cluster", 0)           # (else whole tiles + a cluster remainder: no scratch)
    try:
        need = lib.spec_linear_workspace_bytes(M, N, K)
        assert need > 16 << 20
        _noalloc_over_limit(lib, M, N, K)
    finally:
        lib.spec_set_option("linear_cluster", 1)


def _noalloc_over_limit(lib, M, N, K):
    big_x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    big_w = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.SpecError) as e:
        lib.spec_verify_linear_noalloc(big_x, big_w, Y)
    assert e.value.code == lib.SPEC_EUNSUPPORTED
    assert torch.count_nonzero(Y) == 0
