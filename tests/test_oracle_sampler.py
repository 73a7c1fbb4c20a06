"""Pins of oracle.sampler against what the pages fix about the accept/reject rule.

* lossless: every emitted position is distributed as the target's p
  ("How Speculative Decoding Works (and When It Doesn't)", "Why the output
  doesn't change": min(p, q) + max(0, p - q) = p);
* per-position acceptance = sum_x min(p, q) (same section);
* tokens per round = (1 - a^(g+1)) / (1 - a) under i.i.d. acceptance
  ("Speculative Decoding Spends Arithmetic You May Not Have", "Why γ has a
  ceiling");
* temperature 0: longest argmax-matching prefix plus one ("Exactness is a
  choice");
* structure: 1..gamma+1 tokens, truncation at the first rejection
  (Algorithm 1, "What one iteration actually does").

Mutation tests plant a plausible mistake in the oracle (on the CPU) and
check that these pins catch it.
"""
import numpy as np
import pytest
from scipy import stats

import synth
from oracle import formulas as F
from oracle import sampler as S

V = 8
ROUNDS = 1_000_000


def _dists(seed, gamma):
    rng = np.random.default_rng(seed)
    P = rng.dirichlet(np.full(V, 0.8), size=gamma + 1).astype(np.float32)
    Q = rng.dirichlet(np.full(V, 0.8), size=gamma).astype(np.float32)
    return P, Q


def _rounds(P, Q, n_rounds, seed):
    """n_rounds independent rounds of one sequence shape sharing (p, q)."""
    gamma = Q.shape[0]
    cu = np.arange(n_rounds + 1, dtype=np.int64) * (gamma + 1)
    Pb = np.tile(P, (n_rounds, 1))
    Qb = np.tile(Q, (n_rounds, 1))
    # drafts x_i ~ q_i by inverse CDF on their own Philox stream
    ud = synth.uniforms_f32(seed, n_rounds * gamma).reshape(n_rounds, gamma).astype(np.float64)
    cq = np.cumsum(Q.astype(np.float64), axis=1)
    drafts = np.stack([np.minimum((cq[i][None, :] <= (ud[:, i] * cq[i, -1])[:, None]).sum(1), V - 1)
                       for i in range(gamma)], axis=1).reshape(-1)
    U = synth.uniforms_f32(seed + 7, n_rounds * (gamma + 1))
    n_acc, out, near = S.reject_sample(Pb, Qb, drafts, U, cu)
    return n_acc, out.reshape(n_rounds, gamma + 1), near


def _chi2_pvalue(samples, probs):
    counts = np.bincount(samples, minlength=len(probs)).astype(np.float64)
    pr = probs.astype(np.float64)
    keep = pr > 0
    assert np.all(counts[~keep] == 0), "token with p = 0 was emitted"
    exp = pr[keep] / pr[keep].sum() * counts[keep].sum()
    exp *= counts[keep].sum() / exp.sum()
    return stats.chisquare(counts[keep], exp).pvalue


def check_lossless(n_acc, out, P, min_p=0.01):
    """Position j's token, given the round reached it, is distributed as p_j."""
    gamma = P.shape[0] - 1
    pvals = []
    for j in range(gamma + 1):
        reached = n_acc >= j
        pv = _chi2_pvalue(out[reached, j], P[j])
        pvals.append(pv)
    return min(pvals) > min_p, pvals


@pytest.fixture(scope="module")
def big_run():
    P, Q = _dists(11, 4)
    n_acc, out, near = _rounds(P, Q, ROUNDS, seed=100)
    return P, Q, n_acc, out, near


def test_lossless_chi_square(big_run):
    P, Q, n_acc, out, _ = big_run
    ok, pvals = check_lossless(n_acc, out, P)
    assert ok, pvals


def test_acceptance_rate_is_shared_mass(big_run):
    P, Q, n_acc, out, _ = big_run
    gamma = Q.shape[0]
    for i in range(gamma):
        reached = n_acc >= i
        k = reached.sum()
        acc = (n_acc[reached] > i).mean()
        alpha = F.acceptance_probability(P[i], Q[i])
        sigma = np.sqrt(alpha * (1 - alpha) / k)
        assert abs(acc - alpha) < 4 * sigma + 1e-9, (i, acc, alpha)


def test_mean_tokens_matches_closed_form():
    # i.i.d. acceptance: the same (p, q) at every position
    rng = np.random.default_rng(5)
    p = rng.dirichlet(np.full(V, 0.8)).astype(np.float32)
    q = rng.dirichlet(np.full(V, 0.8)).astype(np.float32)
    for gamma in (1, 4, 7):
        P = np.tile(p, (gamma + 1, 1))
        Q = np.tile(q, (gamma, 1))
        n_acc, _, _ = _rounds(P, Q, 400_000, seed=200 + gamma)
        emitted = n_acc + 1.0
        alpha = F.acceptance_probability(p, q)
        want = F.expected_tokens(alpha, gamma)
        sigma = emitted.std() / np.sqrt(len(emitted))
        assert abs(emitted.mean() - want) < 4 * sigma, (gamma, emitted.mean(), want)


def test_structure_and_truncation(big_run):
    P, Q, n_acc, out, _ = big_run
    gamma = Q.shape[0]
    assert n_acc.min() >= 0 and n_acc.max() <= gamma
    emitted = n_acc + 1
    assert emitted.min() >= 1 and emitted.max() <= gamma + 1
    cols = np.arange(gamma + 1)[None, :]
    assert np.all(out[cols > n_acc[:, None]] == -1)
    assert np.all(out[cols <= n_acc[:, None]] >= 0)


def test_greedy_special_case():
    # T = 0: p is one-hot at the target argmax; any draft q with q(x) > 0.
    rng = np.random.default_rng(9)
    B, gamma = 2000, 6
    tgt = rng.integers(0, V, size=(B, gamma + 1))
    P = np.zeros((B * (gamma + 1), V), np.float32)
    P[np.arange(B * (gamma + 1)), tgt.reshape(-1)] = 1.0
    Q = rng.dirichlet(np.ones(V), size=B * gamma).astype(np.float32)
    # drafts agree with the target argmax on a random prefix
    drafts = rng.integers(0, V, size=(B, gamma))
    agree = rng.integers(0, gamma + 1, size=B)
    for b in range(B):
        drafts[b, :agree[b]] = tgt[b, :agree[b]]
        if agree[b] < gamma and drafts[b, agree[b]] == tgt[b, agree[b]]:
            drafts[b, agree[b]] = (tgt[b, agree[b]] + 1) % V
    cu = np.arange(B + 1) * (gamma + 1)
    U = synth.uniforms_f32(1, B * (gamma + 1))
    n_acc, out, near = S.reject_sample(P, Q, drafts.reshape(-1), U, cu)
    out = out.reshape(B, gamma + 1)
    assert np.array_equal(n_acc, agree)
    for b in range(B):
        n = agree[b]
        assert np.array_equal(out[b, :n], tgt[b, :n])
        assert out[b, n] == tgt[b, n]          # correction / bonus is the argmax
    # a rejected draft with tiny q(x) is within tie_eps of p = 0: counted, result still exact
    assert near.sum() <= B // 100


def test_full_acceptance_when_q_equals_p():
    rng = np.random.default_rng(2)
    p = rng.dirichlet(np.ones(V)).astype(np.float32)
    P = np.tile(p, (5, 1)); Q = np.tile(p, (4, 1))
    n_acc, out, _ = _rounds(P, Q, 20000, seed=3)
    assert np.all(n_acc == 4)                  # u * q <= p always holds when q == p


def test_zero_residual_falls_back_to_p():
    # p == q but a forced reject (u * q > p impossible) -> use a draft token with q > p instead
    p = np.array([[0.25, 0.25, 0.25, 0.25]] * 2, np.float32)
    q = np.array([[0.25, 0.25, 0.25, 0.25]], np.float32)
    r = S.correction_distribution(p[0], q[0])
    assert np.allclose(r, p[0])
    # single-draft exact case: x has q > p, residual puts mass only where p > q
    P = np.array([[0.5, 0.5, 0.0, 0.0], [0.1, 0.2, 0.3, 0.4]], np.float32)
    Q = np.array([[0.0, 0.25, 0.75, 0.0]], np.float32)
    n_acc, out, near = S.reject_sample(P, Q, np.array([2]), np.array([0.5, 0.3], np.float32),
                                       np.array([0, 2]))
    assert n_acc[0] == 0 and out[0] == 0 and out[1] == -1   # residual [0.5, 0.25, 0, 0]


def test_ragged_batch_and_near_ties():
    P = np.array([[0.2, 0.8], [0.5, 0.5], [0.9, 0.1], [0.3, 0.7], [0.6, 0.4]], np.float32)
    Q = np.array([[0.4, 0.6], [0.5, 0.5], [0.5, 0.5]], np.float32)
    drafts = np.array([1, 0, 1])
    cu = np.array([0, 2, 5])
    U = np.array([0.5, 0.1, 0.999, 1.0 / 3.0, 0.5], np.float32)
    n_acc, out, near = S.reject_sample(P, Q, drafts, U, cu)
    # seq 0: 0.5*0.6 = 0.3 <= 0.8 accept; bonus from P[1] with u=0.1 -> token 0
    assert n_acc[0] == 1 and list(out[:2]) == [1, 0]
    # seq 1: 0.999*0.5 > 0.9? no -> accept x=0; 0.333*0.5 = 0.1667 <= 0.7 accept; bonus P[4], u=.5 -> 0.3 <= 0.6: token 0
    assert n_acc[1] == 2 and list(out[2:]) == [0, 1, 0]
    assert near.sum() == 0
    # a decision exactly at the boundary counts as a near tie
    n_acc, out, near = S.reject_sample(np.array([[0.25, 0.75], [0.5, 0.5]], np.float32),
                                       np.array([[0.5, 0.5]], np.float32),
                                       np.array([0]), np.array([0.5, 0.9], np.float32),
                                       np.array([0, 2]))
    assert n_acc[0] == 1 and near[0] == 1


# ---------------------------------------------------------------- mutation pins

def _mutant_run(monkeypatch, name, fn):
    monkeypatch.setattr(S, name, fn)
    P, Q = _dists(11, 3)
    n_acc, out, _ = _rounds(P, Q, 300_000, seed=300)
    return P, Q, n_acc, out


def test_mutation_correction_from_p_is_caught(monkeypatch):
    # mistake: after a rejection, resample from p instead of the residual
    P, Q, n_acc, out = _mutant_run(monkeypatch, "correction_distribution",
                                   lambda p, q: np.asarray(p, np.float64))
    ok, _ = check_lossless(n_acc, out, P)
    assert not ok


def test_mutation_inverted_ratio_is_caught(monkeypatch):
    # mistake: accept with probability min(1, q/p)
    P, Q, n_acc, out = _mutant_run(monkeypatch, "accept_mask",
                                   lambda p, q, u: np.asarray(u, np.float64) * p <= q)
    ok, _ = check_lossless(n_acc, out, P)
    assert not ok


def test_mutation_unclipped_residual_is_caught(monkeypatch):
    # mistake: residual p - q without the max(0, .) clip (negative weights)
    P, Q, n_acc, out = _mutant_run(
        monkeypatch, "correction_distribution",
        lambda p, q: np.abs(np.asarray(p, np.float64) - np.asarray(q, np.float64)))
    ok, _ = check_lossless(n_acc, out, P)
    assert not ok
