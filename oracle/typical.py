"""Typical acceptance, the lossy accept rule (test infrastructure only; parity unpinned).

Follows "How Speculative Decoding Works (and When It Doesn't)", section
"Exactness is a choice": rejection sampling is dropped for a single test per
draft token: keep x_i when the target gives it a probability above a
threshold, and let the threshold depend on the entropy of the target
distribution, "with epsilon a hard floor and delta setting how fast the bar
moves with entropy"; a confident target (low entropy) sets a high bar, an
uncertain one a low bar.

The page's formula did not survive extraction.  Reading adopted (the plainest
one its words support):

    H_i   = -sum_x p_i(x) ln p_i(x)                 (natural log, 0 ln 0 = 0)
    tau_i = max(epsilon, delta * exp(-H_i))          (epsilon: the floor)
    accept x_i  iff  p_i(x_i) > tau_i

Medusa's own rule (the page's source) writes the threshold as
min(epsilon, delta * exp(-H)), with epsilon as a cap instead; with a floor
the page's wording is followed.  Where the exact formula decides the outcome
this function is parity unpinned: only its closed-form special cases are
checked (one-hot rows behave like greedy decoding, as the page states for
temperature 0; uniform rows have H = ln k).

After the accepted prefix x_1 .. x_n (n = first failing test, else gamma),
the next token is drawn from the target row p_{n+1} itself: with no
rejection sampling there is no residual; when every draft passes, p_{gamma+1}
is the bonus distribution as in the exact rule.  The draw uses the same
inverse CDF in token-index order as the exact sampler, with the uniform of
row gamma (rows 0 .. gamma - 1 of U are not used).

Near ties: a test with |p_i(x_i) - tau_i| < tie_eps, and a final pick whose
CDF boundary lies within tie_eps * sum(p) of u * sum(p), are counted per
sequence.
"""
import numpy as np

from .sampler import inverse_cdf_pick


def entropy(p_rows: np.ndarray) -> np.ndarray:
    """H = -sum p ln p along the last axis (fp64; 0 ln 0 = 0).  Rows need not be normalised:
    the rows are the target's probabilities as given."""
    p = np.asarray(p_rows, np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(p > 0.0, p * np.log(np.where(p > 0.0, p, 1.0)), 0.0)
    return -t.sum(axis=-1)


def threshold(p_rows: np.ndarray, eps: float, delta: float) -> np.ndarray:
    """tau = max(eps, delta * exp(-H(p)))."""
    return np.maximum(np.float64(eps), np.float64(delta) * np.exp(-entropy(p_rows)))


def typical_accept_sample(P, drafts, U, cu_rows, eps: float, delta: float, tie_eps: float = 1e-5):
    """One verify round under typical acceptance for a ragged batch.

    P [M, V]: target probabilities of every verify row (packed as for the exact
    sampler); drafts [sum gamma]; U [M] (row gamma_b of each sequence is the draw
    for the final token); cu_rows [B + 1].  Returns n_acc [B], out_tok [M]
    (sequence b emits out_tok[cu_rows[b] : cu_rows[b] + n_acc[b] + 1], later slots
    -1) and near_tie [B], all int32.
    """
    P = np.asarray(P)
    drafts = np.asarray(drafts, np.int64)
    U = np.asarray(U)
    cu = np.asarray(cu_rows, np.int64)
    B = len(cu) - 1
    M = int(cu[-1]) if B else 0
    n_acc = np.zeros(B, np.int64)
    near = np.zeros(B, np.int64)
    out = np.full(M, -1, np.int64)
    for b in range(B):
        r0 = int(cu[b])
        gamma = int(cu[b + 1] - cu[b] - 1)
        q0 = r0 - b
        n = gamma
        for i in range(gamma):
            row = P[r0 + i]
            x = int(drafts[q0 + i])
            px = np.float64(row[x])
            tau = threshold(row, eps, delta)
            if abs(px - tau) < tie_eps:
                near[b] += 1
            if not px > tau:
                n = i
                break
        t, near_pick = inverse_cdf_pick(np.asarray(P[r0 + n], np.float64)[None, :], np.asarray([U[r0 + gamma]]),
                                        tie_eps)
        near[b] += int(near_pick[0])
        n_acc[b] = n
        out[r0:r0 + n] = drafts[q0:q0 + n]
        out[r0 + n] = int(t[0])
    return n_acc.astype(np.int32), out.astype(np.int32), near.astype(np.int32)
