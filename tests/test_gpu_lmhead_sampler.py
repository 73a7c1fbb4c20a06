"""GPU parity of spec_lmhead_softmax and spec_reject_sample against the oracle."""
import numpy as np
import pytest
import torch
from scipy import stats

import synth
from oracle import bf16 as obf, formulas as F, ops as oops, sampler as osamp

from gpu_util import PROB_ATOL, bf16_dev, dev

pytestmark = pytest.mark.gpu


def lmhead_case(lib, M, K, V, T, seed, std=0.02):
    H = synth.normal_bf16_bits(seed, (M, K), 1.0)
    W = synth.normal_bf16_bits(seed + 1, (V, K), std)
    P = lib.spec_lmhead_softmax(bf16_dev(H), bf16_dev(W), T)
    lib.spec_device_status()
    logits = oops.linear(obf.decode(H), obf.decode(W))
    return P.cpu().numpy(), logits


@pytest.mark.parametrize("M,K,V,T", [
    (5, 512, 4096, 1.0), (1, 512, 4096, 0.7), (40, 4096, 8192, 1.0), (17, 264, 1000, 0.5),
    (300, 512, 2048, 1.0), (3, 1024, 151936, 0.7),
])
def test_lmhead_softmax_probabilities(lib, M, K, V, T):
    P, logits = lmhead_case(lib, M, K, V, T, seed=M + V)
    ref = oops.target_probs(logits, T)
    err = np.abs(P.astype(np.float64) - ref).max()
    assert err < PROB_ATOL, err
    assert np.allclose(P.sum(axis=1), 1.0, atol=1e-4)


@pytest.mark.parametrize("M,K,V", [(5, 512, 4096), (40, 4096, 8192), (2, 512, 151936)])
def test_lmhead_greedy_one_hot(lib, M, K, V):
    P, logits = lmhead_case(lib, M, K, V, 0.0, seed=3 * M + V, std=0.05)
    assert np.all((P == 0.0) | (P == 1.0)) and np.all(P.sum(axis=1) == 1.0)
    idx = P.argmax(axis=1)
    top = logits.max(axis=1)
    # the argmax is decided on fp32 logits; where the fp64 logits of two tokens lie
    # closer than fp32 accumulation error, either pick is correct
    assert np.all(logits[np.arange(M), idx] >= top - 1e-4 * np.abs(top).max())
    exact = np.argmax(logits, axis=1)
    gap = np.sort(logits, axis=1)[:, -1] - np.sort(logits, axis=1)[:, -2]
    clear = gap > 1e-4
    assert np.array_equal(idx[clear], exact[clear])


@pytest.mark.parametrize("M,K,V,T", [(100, 512, 30000, 1.0), (300, 256, 151936, 0.7), (300, 256, 8200, 0.0)])
def test_lmhead_ragged_vocab_tiles(lib, M, K, V, T):
    """LM head on vocabularies that leave a ragged last 128-row tile, at 100 and 300 rows."""
    P, logits = lmhead_case(lib, M, K, V, T, seed=M + V, std=0.05 if T == 0 else 0.02)
    if T > 0:
        ref = oops.target_probs(logits, T)
        assert np.abs(P.astype(np.float64) - ref).max() < PROB_ATOL
    else:
        idx = P.argmax(axis=1)
        gap = np.sort(logits, axis=1)[:, -1] - np.sort(logits, axis=1)[:, -2]
        clear = gap > 1e-4
        assert np.array_equal(idx[clear], np.argmax(logits, axis=1)[clear])
        assert np.all(P.sum(axis=1) == 1.0)


# ------------------------------------------------------------------ sampler

def sampler_inputs(seed, gammas, V, conc=0.5, zero_frac=0.0):
    rng = np.random.default_rng(seed)
    batch = synth.RaggedBatch(gammas, np.zeros(len(gammas), np.int32))
    P = rng.dirichlet(np.full(V, conc), size=batch.M).astype(np.float32)
    Q = rng.dirichlet(np.full(V, conc), size=batch.n_drafts).astype(np.float32)
    if zero_frac:
        Q[rng.random(Q.shape) < zero_frac] = 0.0
    drafts = np.array([rng.choice(V, p=q.astype(np.float64) / q.astype(np.float64).sum()) for q in Q],
                      np.int32) if batch.n_drafts else np.zeros(0, np.int32)
    U = synth.uniforms_f32(seed + 1, batch.M)
    return batch, P, Q, drafts, U


def gpu_sample(lib, batch, P, Q, drafts, U, tie_eps=1e-5):
    Qd = dev(Q) if Q.size else torch.zeros((1, P.shape[1]), dtype=torch.float32, device="cuda")
    Dd = dev(drafts) if drafts.size else torch.zeros(1, dtype=torch.int32, device="cuda")
    n, t, near = lib.spec_reject_sample(dev(P), Qd, Dd, dev(U), dev(batch.cu_rows), tie_eps)
    lib.spec_device_status()
    return n.cpu().numpy(), t.cpu().numpy(), near.cpu().numpy()


@pytest.mark.parametrize("gammas,V", [
    ([4], 8), ([0, 1, 2, 10], 50), (list(range(0, 12)), 4096), ([3] * 64, 151936),
    ([31, 32, 33, 40], 64),
])
def test_sampler_bit_exact_on_identical_inputs(lib, gammas, V):
    batch, P, Q, drafts, U = sampler_inputs(len(gammas) + V, gammas, V)
    n, t, near = gpu_sample(lib, batch, P, Q, drafts, U)
    n_ref, t_ref, near_ref = osamp.reject_sample(P, Q, drafts, U, batch.cu_rows)
    assert np.array_equal(n, n_ref)
    assert np.array_equal(t, t_ref)
    assert np.array_equal(near, near_ref)


def test_sampler_zero_draft_probabilities_and_fallback(lib):
    # q(x) = 0 accepts; p == q rows make the residual empty and fall back to p
    batch, P, Q, drafts, U = sampler_inputs(3, [5, 5, 5], 16, zero_frac=0.3)
    Q[0:5] = P[0:5]                              # sequence 0: q == p everywhere
    n, t, near = gpu_sample(lib, batch, P, Q, drafts, U)
    n_ref, t_ref, near_ref = osamp.reject_sample(P, Q, drafts, U, batch.cu_rows)
    assert np.array_equal(n, n_ref) and np.array_equal(t, t_ref) and np.array_equal(near, near_ref)


def test_sampler_greedy_prefix_rule(lib):
    rng = np.random.default_rng(4)
    B, gamma, V = 500, 6, 32
    tgt = rng.integers(0, V, size=(B, gamma + 1))
    P = np.zeros((B * (gamma + 1), V), np.float32)
    P[np.arange(B * (gamma + 1)), tgt.reshape(-1)] = 1.0
    Q = rng.dirichlet(np.ones(V), size=B * gamma).astype(np.float32)
    agree = rng.integers(0, gamma + 1, size=B)
    drafts = rng.integers(0, V, size=(B, gamma))
    for b in range(B):
        drafts[b, :agree[b]] = tgt[b, :agree[b]]
        if agree[b] < gamma and drafts[b, agree[b]] == tgt[b, agree[b]]:
            drafts[b, agree[b]] = (tgt[b, agree[b]] + 1) % V
    batch = synth.RaggedBatch([gamma] * B, np.zeros(B, np.int32))
    n, t, _ = gpu_sample(lib, batch, P, Q, drafts.reshape(-1).astype(np.int32), synth.uniforms_f32(5, batch.M))
    assert np.array_equal(n, agree)
    t = t.reshape(B, gamma + 1)
    for b in range(B):
        assert np.array_equal(t[b, :agree[b] + 1], tgt[b, :agree[b] + 1])


def test_sampler_lossless_on_gpu(lib):
    """Chi-square on V = 8 over 1e6 GPU rounds: emitted tokens follow p."""
    rng = np.random.default_rng(11)
    V, gamma, R = 8, 4, 1_000_000
    p = rng.dirichlet(np.full(V, 0.8), size=gamma + 1).astype(np.float32)
    q = rng.dirichlet(np.full(V, 0.8), size=gamma).astype(np.float32)
    ud = synth.uniforms_f32(100, R * gamma).reshape(R, gamma).astype(np.float64)
    cq = np.cumsum(q.astype(np.float64), axis=1)
    drafts = np.stack([np.minimum((cq[i][None, :] <= (ud[:, i] * cq[i, -1])[:, None]).sum(1), V - 1)
                       for i in range(gamma)], axis=1).reshape(-1).astype(np.int32)
    cu = (np.arange(R + 1) * (gamma + 1)).astype(np.int32)
    U = synth.uniforms_f32(107, R * (gamma + 1))
    Pd = dev(np.tile(p, (R, 1)))
    Qd = dev(np.tile(q, (R, 1)))
    n, t, _ = lib.spec_reject_sample(Pd, Qd, dev(drafts), dev(U), dev(cu))
    lib.spec_device_status()
    n = n.cpu().numpy()
    t = t.cpu().numpy().reshape(R, gamma + 1)
    for j in range(gamma + 1):
        reached = n >= j
        counts = np.bincount(t[reached, j], minlength=V).astype(np.float64)
        exp = p[j].astype(np.float64) / p[j].sum() * counts.sum()
        assert stats.chisquare(counts, exp * counts.sum() / exp.sum()).pvalue > 0.01, j
    for i in range(gamma):
        reached = n >= i
        acc = (n[reached] > i).mean()
        alpha = F.acceptance_probability(p[i], q[i])
        assert abs(acc - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / reached.sum())


def test_sampler_empty_batch_and_bad_token_flag(lib):
    batch, P, Q, drafts, U = sampler_inputs(9, [2], 8)
    drafts[0] = 99                                # out of range: clamped and flagged
    Pd, Qd = dev(P), dev(Q)
    lib.spec_reject_sample(Pd, Qd, dev(drafts), dev(U), dev(batch.cu_rows))
    with pytest.raises(lib.SpecError):
        lib.spec_device_status()
    lib.spec_device_status()                      # cleared
    # B = 0: nothing to do, nothing launched
    empty = torch.zeros(1, dtype=torch.int32, device="cuda")
    n, t, near = lib.spec_reject_sample(Pd, Qd, dev(drafts), dev(U), empty)
    assert n.numel() == 0 and near.numel() == 0


@pytest.mark.parametrize("M,T", [(368, 0.7), (300, 0.0), (260, 1.0)])
def test_lmhead_token_tiling_does_not_change_results(lib, M, T):
    """One 384-row token tile (lmhead_nsub 2, the default above 256 rows) or two 192-row tiles
    (lmhead_nsub 1): every logit is the same k-ordered sum and every statistic covers the same 128
    vocabulary rows, so the probabilities come out bit for bit the same; both match the oracle."""
    K, V = 512, 8200
    H = bf16_dev(synth.normal_bf16_bits(M, (M, K), 1.0))
    W = bf16_dev(synth.normal_bf16_bits(M + 1, (V, K), 0.05))
    out = {}
    for nsub in (1, 2):
        lib.spec_set_option("lmhead_nsub", nsub)
        try:
            out[nsub] = lib.spec_lmhead_softmax(H, W, T)
            lib.spec_device_status()
        finally:
            lib.spec_set_option("lmhead_nsub", 2)
    assert torch.equal(out[1], out[2])
    logits = oops.linear(obf.decode(synth.normal_bf16_bits(M, (M, K), 1.0)),
                         obf.decode(synth.normal_bf16_bits(M + 1, (V, K), 0.05)))
    ref = oops.target_probs(logits, T)
    if T > 0:
        assert np.abs(out[2].cpu().numpy().astype(np.float64) - ref).max() < PROB_ATOL
    else:
        top2 = np.sort(logits, axis=1)
        clear = (top2[:, -1] - top2[:, -2]) > 1e-3
        assert np.array_equal(out[2].cpu().numpy().argmax(1)[clear], logits.argmax(1)[clear])
