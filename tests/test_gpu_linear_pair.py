"""GPU parity of the 2-SM pair GEMM (spec_set_option("linear_pair", 1)): 256-row weight tiles on CTA
pairs, each CTA staging half of every MMA's token rows, k-steps split between the pairs of a
cluster and summed on chip.  Every case is checked element by element against the fp64 oracle
(the single-linear bar) and the plan is checked to be the pair kernel's."""
import numpy as np
import pytest

import synth
from oracle import bf16 as obf, ops as oops

from gpu_util import assert_close_chain, assert_close_rel, bf16_dev, bits_of, dev, f64_of_bf16

pytestmark = pytest.mark.gpu


# pairs for every product with 64+ token rows (split-K on pairs for few tiles), or pairs only for
# products with more 128-row tiles than SMs (whole pair tiles, then the rest split); the persistent
# pair kernel (an option for the latter) is off here: its own tests cover it
@pytest.fixture(params=[1, 0], ids=["pairs-everywhere", "many-tiles"])
def pair(lib, request):
    lib.spec_set_option("linear_pair", 1)
    lib.spec_set_option("linear_pair_few", request.param)
    lib.spec_set_option("linear_pair_persistent", 0)
    yield lib
    lib.spec_set_option("linear_pair_few", 0)


SHAPES = [
    # (M, N, K): the Qwen3-8B projections at the benchmark's 368 rows, other token tiles,
    # ragged N (an odd number of 128-row tiles leaves half of the last pair empty), ragged K
    (368, 6144, 4096), (368, 4096, 4096), (368, 4096, 12288), (64, 4096, 4096), (100, 1152, 520),
    (200, 1000, 1024), (256, 2048, 2048), (300, 640, 1000), (384, 512, 256), (129, 3072, 4096),
    # more 128-row tiles than SMs: whole pair tiles, then the rest
    (368, 24576, 1024), (200, 20480, 136), (300, 19584, 520),
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("residual", [False, True])
def test_pair_linear(pair, M, N, K, residual):
    lib = pair
    X = synth.normal_bf16_bits(M + K, (M, K), 1.0)
    W = synth.normal_bf16_bits(N + K, (N, K), 0.02)
    R = synth.normal_bf16_bits(M + N, (M, N), 1.0) if residual else None
    assert lib.spec_linear_workspace_bytes(M, N, K) == 0
    lib.reset_launch_count()
    Y = lib.spec_verify_linear(bf16_dev(X), bf16_dev(W), residual=bf16_dev(R) if residual else None)
    launches = lib.launch_count()
    lib.spec_device_status()
    ref = oops.linear(obf.decode(X), obf.decode(W), obf.decode(R) if residual else None)
    assert_close_rel(f64_of_bf16(Y), ref, f"pair linear M={M} N={N} K={K}")
    assert launches in (1, 2)


@pytest.mark.parametrize("M,I,K", [(368, 12288, 4096), (300, 640, 1000), (128, 1088, 512)])
def test_pair_swiglu(pair, M, I, K):
    lib = pair
    X = synth.normal_bf16_bits(7 + M, (M, K), 1.0)
    Wg = synth.normal_bf16_bits(8 + I, (I, K), 0.05)
    Wu = synth.normal_bf16_bits(9 + I, (I, K), 0.05)
    Wgu = lib.interleave_gate_up(bf16_dev(Wg), bf16_dev(Wu))
    A = lib.spec_verify_linear_swiglu(bf16_dev(X), Wgu)
    lib.spec_device_status()
    x = obf.decode(X)
    ref = oops.silu_mul(oops.linear(x, obf.decode(Wg)), oops.linear(x, obf.decode(Wu)))
    assert_close_rel(f64_of_bf16(A), ref, f"pair swiglu M={M} I={I} K={K}")


@pytest.mark.parametrize("M", [368, 100])
def test_pair_linear_rope(pair, M):
    """QKV projection with the rotation in the pair kernel's epilogue (one launch)."""
    lib = pair
    Hq, Hkv, D, K = 32, 8, 128, 4096
    rng = np.random.default_rng(M)
    B = max(1, M // 6)
    gam = np.full(B, M // B - 1)
    gam[-1] += M - int((gam + 1).sum())
    batch = synth.RaggedBatch(gam, rng.integers(0, 8000, size=B))
    N = (Hq + 2 * Hkv) * D
    X = synth.normal_bf16_bits(M + 1, (M, K), 1.0)
    W = synth.normal_bf16_bits(M + 2, (N, K), 0.02)
    cs = lib.spec_rope_table(dev(batch.cu_rows), dev(batch.ctx_len), M, D, 1e6)
    lib.reset_launch_count()
    Y = lib.spec_verify_linear_rope(bf16_dev(X), bf16_dev(W), cs, Hq + Hkv)
    assert lib.launch_count() == 1
    lib.spec_device_status()
    pos = np.concatenate([batch.ctx_len[b] + np.arange(batch.gammas[b] + 1) for b in range(batch.B)])
    y = oops.linear(obf.decode(X), obf.decode(W))
    ref = y.copy()
    ref[:, :(Hq + Hkv) * D] = oops.rope(y[:, :(Hq + Hkv) * D].reshape(M, Hq + Hkv, D), pos, 1e6).reshape(M, -1)
    assert_close_chain(f64_of_bf16(Y), ref, 1, f"pair linear + rope M={M}")
    assert_close_rel(f64_of_bf16(Y)[:, (Hq + Hkv) * D:], y[:, (Hq + Hkv) * D:], "pair linear (v heads)")


def test_pair_bit_identical_on_repeat_and_with_residual_alias(pair):
    """The on-chip sums run in pair order: repeated calls give the same bits; Y may alias the
    residual exactly."""
    lib = pair
    import torch
    M, N, K = 368, 4096, 4096
    X = bf16_dev(synth.normal_bf16_bits(1, (M, K), 1.0))
    W = bf16_dev(synth.normal_bf16_bits(2, (N, K), 0.02))
    R = synth.normal_bf16_bits(3, (M, N), 1.0)
    a = lib.spec_verify_linear(X, W, residual=bf16_dev(R))
    b = lib.spec_verify_linear(X, W, residual=bf16_dev(R))
    Y = bf16_dev(R).clone()
    lib.spec_verify_linear(X, W, Y=Y, residual=Y)
    lib.spec_device_status()
    assert np.array_equal(bits_of(a), bits_of(b))
    assert np.array_equal(bits_of(a), bits_of(Y))
