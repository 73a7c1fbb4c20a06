"""Pins of the typical-acceptance oracle ("How Speculative Decoding Works (and When It Doesn't)",
"Exactness is a choice").  The page's threshold formula was lost in extraction, so these pin
the reading's closed-form cases and the page's stated properties, not the formula itself:
entropy of uniform / one-hot / two-point rows, the threshold's floor and its entropy slope,
greedy equivalence on one-hot rows (temperature 0), and the final token drawn from the target
row itself (no residual)."""
import numpy as np
import pytest
from scipy import stats

import synth
from oracle import sampler as S
from oracle import typical as T


def test_entropy_closed_forms():
    for k in (1, 2, 5, 64):
        row = np.zeros(100)
        row[:k] = 1.0 / k
        assert abs(T.entropy(row) - np.log(k)) < 1e-12
    a = 0.3
    assert abs(T.entropy(np.array([a, 1 - a, 0.0])) - (-(a * np.log(a) + (1 - a) * np.log(1 - a)))) < 1e-15
    rng = np.random.default_rng(0)
    p = rng.dirichlet(np.full(50, 0.4))
    assert abs(T.entropy(p) - stats.entropy(p)) < 1e-12


def test_threshold_floor_and_entropy_slope():
    one_hot = np.zeros(10)
    one_hot[3] = 1.0
    assert T.threshold(one_hot, 0.05, 0.3) == pytest.approx(0.3)        # H = 0: max(eps, delta)
    assert T.threshold(one_hot, 0.5, 0.3) == pytest.approx(0.5)
    for k in (2, 4, 25, 1000):
        row = np.full(k, 1.0 / k)
        assert T.threshold(row, 0.05, 0.3) == pytest.approx(max(0.05, 0.3 / k), rel=1e-12)
    # the bar falls as the entropy rises, and never below the floor
    rows = [np.full(k, 1.0 / k) for k in (1, 2, 3, 8, 50, 400)]
    taus = [float(T.threshold(r, 0.01, 0.4)) for r in rows]
    assert all(a >= b for a, b in zip(taus, taus[1:])) and min(taus) == pytest.approx(0.01)


def _one_seq(P_rows, drafts, u_final, eps, delta):
    gamma = len(drafts)
    cu = np.array([0, gamma + 1], np.int32)
    U = np.full(gamma + 1, 0.5, np.float32)
    U[gamma] = u_final
    return T.typical_accept_sample(np.asarray(P_rows, np.float32), np.asarray(drafts, np.int32), U, cu, eps, delta)


def test_uniform_rows_accept_by_closed_form():
    V = 32
    def row(k):
        r = np.zeros(V, np.float32)
        r[:k] = 1.0 / k
        return r
    # eps 0.05, delta 0.3: k = 4 -> tau = max(0.05, 0.075), 1/4 passes; k = 25 -> tau = 0.05, 1/25 fails
    n, out, _ = _one_seq([row(4), row(4), row(25), row(2)], [1, 2, 3], 0.3, 0.05, 0.3)
    assert n[0] == 2 and list(out[:2]) == [1, 2]
    # natural log, not log2: k = 4, delta = 1.2 -> tau = 0.3 > 1/4 (log2 would give 0.16 and accept)
    n, _, _ = _one_seq([row(4), row(4)], [0], 0.3, 0.01, 1.2)
    assert n[0] == 0
    # a draft outside the support has p = 0 and always fails
    n, _, _ = _one_seq([row(4), row(4)], [10], 0.3, 0.0, 0.0)
    assert n[0] == 0


def test_one_hot_rows_reduce_to_greedy():
    """Temperature 0: the target rows are one-hot, both rules keep exactly the drafts that equal
    the argmax and then emit the argmax (the page's closing remark in the section)."""
    rng = np.random.default_rng(3)
    B, gamma, V = 200, 5, 16
    tgt = rng.integers(0, V, size=(B, gamma + 1))
    P = np.zeros((B * (gamma + 1), V), np.float32)
    P[np.arange(B * (gamma + 1)), tgt.reshape(-1)] = 1.0
    agree = rng.integers(0, gamma + 1, size=B)
    drafts = rng.integers(0, V, size=(B, gamma))
    for b in range(B):
        drafts[b, :agree[b]] = tgt[b, :agree[b]]
        if agree[b] < gamma and drafts[b, agree[b]] == tgt[b, agree[b]]:
            drafts[b, agree[b]] = (tgt[b, agree[b]] + 1) % V
    cu = (np.arange(B + 1) * (gamma + 1)).astype(np.int32)
    U = synth.uniforms_f32(4, B * (gamma + 1))
    Q = rng.dirichlet(np.ones(V), size=B * gamma).astype(np.float32)
    n, out, _ = T.typical_accept_sample(P, drafts.reshape(-1).astype(np.int32), U, cu, 0.09, 0.3)
    n_ex, out_ex, _ = S.reject_sample(P, Q, drafts.reshape(-1).astype(np.int32), U, cu)
    assert np.array_equal(n, agree) and np.array_equal(n, n_ex) and np.array_equal(out, out_ex)


def test_final_token_comes_from_the_target_row():
    """The first draft always fails (p_1(x_1) = 0), so the emitted token is a draw from p_1 itself
    (the row the failing draft was tested against): chi-square over 20000 rounds."""
    V, R = 6, 20000
    p1 = np.array([0.0, 0.1, 0.15, 0.2, 0.25, 0.3])
    p2 = np.full(V, 1.0 / V)
    P = np.tile(np.stack([p1, p2]).astype(np.float32), (R, 1))
    drafts = np.zeros(R, np.int32)                 # token 0 has p = 0 in row 0
    cu = (np.arange(R + 1) * 2).astype(np.int32)
    U = synth.uniforms_f32(9, 2 * R)
    n, out, _ = T.typical_accept_sample(P, drafts, U, cu, 0.01, 0.3)
    assert np.all(n == 0)
    counts = np.bincount(out[0::2], minlength=V).astype(np.float64)
    assert counts[0] == 0
    assert stats.chisquare(counts[1:], p1[1:] * R).pvalue > 0.001


def test_every_draft_accepted_takes_the_bonus_row():
    V = 8
    sure = np.zeros(V, np.float32)
    sure[2] = 1.0
    bonus = np.zeros(V, np.float32)
    bonus[5] = 1.0
    n, out, near = _one_seq([sure, sure, bonus], [2, 2], 0.7, 0.05, 0.3)
    assert n[0] == 2 and list(out) == [2, 2, 5] and near[0] == 0


def test_near_ties_are_counted():
    V = 4
    row = np.full(V, 0.25, np.float32)
    # tau = max(eps, delta / 4) = 0.25 + 1e-7: p(x) = 0.25 fails, inside the 1e-5 band
    n, _, near = _one_seq([row, row], [0], 0.5, 0.25 + 1e-7, 0.0)
    assert n[0] == 0 and near[0] >= 1
