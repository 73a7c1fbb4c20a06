"""GPU parity of the persistent GEMM on CTA pairs (tcgen05 2-SM MMA): the LM head (lmhead_pair, the
default) and, as an option (linear_pair_persistent), products with more 128-row weight tiles than
SMs run whole 256-row pair tiles round-robin on the pairs, then the pair tiles left over as
stream-K pieces summed by the reduce kernel (1) or on the pair split-K kernel (2); 0 is the default
two-launch plan.  Every case is
checked element by element against the fp64 oracle (the single-linear bar); the shapes cover odd
numbers of 128-row tiles (the last pair tile's second half lies past N), token tiles rounded up to
a pair build, ragged K, and the folded RMSNorm's row scales."""
import numpy as np
import pytest
import torch

import synth
from oracle import bf16 as obf, ops as oops, sampler as osamp

from gpu_util import PROB_ATOL, assert_close_chain, assert_close_rel, bf16_dev, bits_of, dev, f64_of_bf16

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(params=[1, 2, 0], ids=["stream-k-rest", "split-k-rest", "two-launch"])
def persistent(lib, request):
    lib.spec_set_option("linear_pair", 1)
    lib.spec_set_option("linear_pair_persistent", request.param)
    yield lib, request.param
    lib.spec_set_option("linear_pair_persistent", 0)


SHAPES = [
    # (M, N, K)
    (368, 24576, 1024),   # gate|up rows at the benchmark's 368 rows: 96 pair tiles, 20 left over
    (368, 40000, 256),    # 313 tiles (odd): 157 pair tiles, the last one's second half past N
    (300, 19584, 520),    # NSUB = 2, BN 160, ragged K
    (200, 20480, 136),    # NSUB = 1, BN 208 rounded up to 224
    (100, 20000, 264),    # NSUB = 1, BN 112 rounded up to 128, ragged N
    (64, 19584, 512),     # 64 rows: BN 64
    (384, 38912, 128),    # two k-steps, 152 pair tiles: two whole ones per pair
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("residual", [False, True])
def test_pair_persistent_linear(persistent, M, N, K, residual):
    lib, mode = persistent
    X = synth.normal_bf16_bits(M + K, (M, K), 1.0)
    W = synth.normal_bf16_bits(N + K, (N, K), 0.02)
    R = synth.normal_bf16_bits(M + N, (M, N), 1.0) if residual else None
    lib.reset_launch_count()
    Y = lib.spec_verify_linear(bf16_dev(X), bf16_dev(W), residual=bf16_dev(R) if residual else None)
    launches = lib.launch_count()
    lib.spec_device_status()
    ref = oops.linear(obf.decode(X), obf.decode(W), obf.decode(R) if residual else None)
    assert_close_rel(f64_of_bf16(Y), ref, f"pair persistent ({mode}) M={M} N={N} K={K}")
    assert launches in (1, 2)


@pytest.mark.parametrize("M,N,K", [(368, 40000, 256), (200, 20480, 136)])
def test_pair_persistent_deterministic(persistent, M, N, K):
    """Pieces are summed in CTA order: the same bits on every call, and Y may alias the residual."""
    lib, _ = persistent
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


@pytest.mark.parametrize("M,I,K", [(368, 12288, 512), (300, 9792, 520), (128, 10240, 264)])
def test_pair_persistent_swiglu(persistent, M, I, K):
    lib, mode = persistent
    X = synth.normal_bf16_bits(7 + M, (M, K), 1.0)
    Wg = synth.normal_bf16_bits(8 + I, (I, K), 0.05)
    Wu = synth.normal_bf16_bits(9 + I, (I, K), 0.05)
    Wgu = lib.interleave_gate_up(bf16_dev(Wg), bf16_dev(Wu))
    A = lib.spec_verify_linear_swiglu(bf16_dev(X), Wgu)
    lib.spec_device_status()
    x = obf.decode(X)
    ref = oops.silu_mul(oops.linear(x, obf.decode(Wg)), oops.linear(x, obf.decode(Wu)))
    assert_close_rel(f64_of_bf16(A), ref, f"pair persistent ({mode}) swiglu M={M} I={I} K={K}")


@pytest.mark.parametrize("M,N,K", [(368, 24576, 512), (200, 20480, 136)])
def test_pair_persistent_folded_norm(persistent, M, N, K):
    """h W^T with h = RMSNorm(x): rows scaled by 1 / rms in the epilogue (pieces scaled alike)."""
    lib, mode = persistent
    X = bf16_dev(synth.normal_bf16_bits(M + N, (M, K), 2.0))
    ssq = lib.spec_row_ssq(X)
    W = synth.normal_bf16_bits(M + K, (N, K), 0.02)
    Y = lib.spec_verify_linear(X, bf16_dev(W), norm=lib.row_norm(in_ssq=ssq, eps=EPS))
    lib.spec_device_status()
    h = obf.round_to_bf16(oops.rmsnorm(f64_of_bf16(X), np.ones(K), EPS))
    assert_close_chain(f64_of_bf16(Y), oops.linear(h, obf.decode(W)), 1, f"normed pair persistent ({mode}) M={M}")


@pytest.mark.parametrize("M,K,V,T", [(368, 256, 40000, 0.7), (300, 512, 30000, 1.0), (100, 264, 20000, 0.5)])
def test_pair_lmhead_softmax(lib, M, K, V, T):
    H = synth.normal_bf16_bits(M + V, (M, K), 1.0)
    W = synth.normal_bf16_bits(M + V + 1, (V, K), 0.02)
    P = lib.spec_lmhead_softmax(bf16_dev(H), bf16_dev(W), T).cpu().numpy()
    lib.spec_device_status()
    ref = oops.target_probs(oops.linear(obf.decode(H), obf.decode(W)), T)
    assert np.abs(P.astype(np.float64) - ref).max() < PROB_ATOL
    assert np.allclose(P.sum(axis=1), 1.0, atol=1e-4)


@pytest.mark.parametrize("M,K,V", [(368, 256, 40000), (64, 512, 19968)])
def test_pair_lmhead_greedy(lib, M, K, V):
    H = synth.normal_bf16_bits(3 * M + V, (M, K), 1.0)
    W = synth.normal_bf16_bits(3 * M + V + 1, (V, K), 0.05)
    P = lib.spec_lmhead_softmax(bf16_dev(H), bf16_dev(W), 0.0).cpu().numpy()
    lib.spec_device_status()
    logits = oops.linear(obf.decode(H), obf.decode(W))
    assert np.all(P.sum(axis=1) == 1.0)
    idx = P.argmax(axis=1)
    s = np.sort(logits, axis=1)
    clear = s[:, -1] - s[:, -2] > 1e-4
    assert clear.sum() > M // 2
    assert np.array_equal(idx[clear], np.argmax(logits, axis=1)[clear])


def test_pair_lmhead_sampler_matches_the_one_sm_path(lib):
    """The fused LM head -> sampler on pairs and on the one-SM kernel: the same decisions wherever
    neither side reports a near tie, and both match the oracle there."""
    M, K, V, T = 368, 512, 30000, 0.7
    batch = synth.RaggedBatch([4] * 73 + [2], [100] * 74)
    assert batch.M == M
    H = synth.normal_bf16_bits(21, (M, K), 1.0)
    W = synth.normal_bf16_bits(22, (V, K), 0.25)
    logits = oops.linear(obf.decode(H), obf.decode(W))
    q, drafts = synth.draft_distribution(logits, batch, 0.5, T, seed=23)
    U = synth.uniforms_f32(24, M)
    outs = []
    for pair in (1, 0):
        lib.spec_set_option("lmhead_pair", pair)
        n, t, near = lib.spec_lmhead_reject_sample(bf16_dev(H), bf16_dev(W), T, dev(q), dev(drafts), dev(U),
                                                   dev(batch.cu_rows))
        lib.spec_device_status()
        outs.append((n.cpu().numpy(), t.cpu().numpy(), near.cpu().numpy()))
    lib.spec_set_option("lmhead_pair", 1)
    p_ref = oops.target_probs(logits, T)
    n_ref, t_ref, near_ref = osamp.reject_sample(p_ref, q, drafts, U, batch.cu_rows, 1e-4)
    clear = (outs[0][2] == 0) & (outs[1][2] == 0) & (near_ref == 0)
    assert clear.sum() >= batch.B // 2
    for b in np.nonzero(clear)[0]:
        r0 = batch.cu_rows[b]
        for n, t, _ in outs:
            assert n[b] == n_ref[b], b
            assert np.array_equal(t[r0:r0 + n[b] + 1], t_ref[r0:r0 + n[b] + 1]), b
