"""Leviathan-style rejection sampler for one verify round (test infrastructure only).

Follows the steps of Algorithm 1 on "Speculative Decoding Spends Arithmetic
You May Not Have" (section "What one iteration actually does"), in its
order, for a ragged batch of sequences:

1. draw r_1 .. r_gamma ~ U(0, 1)                       (caller-supplied)
2. n = (first i with r_i > p_i(x_i) / q_i(x_i)) - 1, else gamma
3. p' = norm(max(0, p_{n+1} - q_{n+1})) if n < gamma, else p' = p_{gamma+1}
4. emit x_1 .. x_n and t ~ p'

Readings of the points the pages leave open:

* the test is done without division: accept x_i iff u_i * q_i(x_i) <= p_i(x_i)
  (the rejection condition of Algorithm 1 multiplied by q > 0; q = 0 accepts);
  the product is exact in fp64 for fp32 inputs;
* uniforms are packed one per verify row: rows 0 .. gamma-1 of a sequence
  carry r_1 .. r_gamma, row gamma carries the draw for t;
* t is drawn by inverse CDF in token-index order over the *unnormalised*
  p': t = smallest x with sum_{y<=x} p'(y) > u * sum_y p'(y), all in fp64;
* if the residual max(0, p - q) sums to zero (p == q up to rounding), t is
  drawn from p_{n+1} itself;
* the bonus distribution is p_{gamma+1} of the same verify pass
  ("How Speculative Decoding Works (and When It Doesn't)", "How speculative
  decoding works": a fully accepted draft of k tokens commits k + 1).

Near ties: a decision with |u*q - p| < tie_eps, and a final pick whose CDF
boundary lies within tie_eps * sum(p') of u * sum(p'), is counted per
sequence.  Those are the only places where two correct implementations that
round differently may disagree.
"""
import numpy as np


def accept_mask(p_x: np.ndarray, q_x: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Accept draft i iff u_i * q_i(x_i) <= p_i(x_i) (fp64; exact for fp32 inputs)."""
    return np.asarray(u, np.float64) * np.asarray(q_x, np.float64) <= np.asarray(p_x, np.float64)


def correction_distribution(p_row: np.ndarray, q_row: np.ndarray) -> np.ndarray:
    """Unnormalised residual max(0, p - q) (fp64), rows along the last axis.

    Rows whose residual mass is zero fall back to p itself.
    """
    p = np.asarray(p_row, np.float64)
    r = np.maximum(0.0, p - np.asarray(q_row, np.float64))
    empty = r.sum(axis=-1) <= 0.0
    if np.any(empty):
        r = np.where(empty[..., None], p, r)
    return r


def inverse_cdf_pick(weights: np.ndarray, u: np.ndarray, tie_eps: float):
    """Smallest index x with cumsum(w)[x] > u * sum(w), per row (fp64).

    Returns (index, near_tie) where near_tie flags picks whose bracketing
    CDF values lie within tie_eps * sum(w) of the threshold.
    """
    w = np.asarray(weights, np.float64)
    c = np.cumsum(w, axis=-1)
    total = c[..., -1]
    thr = np.asarray(u, np.float64) * total
    idx = np.sum(c <= thr[..., None], axis=-1)
    V = w.shape[-1]
    # u < 1 keeps the threshold below the total; guard against a zero row
    idx = np.minimum(idx, V - 1)
    rows = np.arange(w.shape[0])
    hi = c[rows, idx]
    lo = np.where(idx > 0, c[rows, np.maximum(idx - 1, 0)], 0.0)
    band = tie_eps * total
    near = (np.abs(hi - thr) < band) | ((idx > 0) & (np.abs(lo - thr) < band))
    return idx.astype(np.int64), near


def reject_sample(P, Q, drafts, U, cu_rows, tie_eps: float = 1e-5):
    """One verify round's acceptance for a ragged batch.

    P [M, V]: target probabilities of every verify row (row 0 of sequence b
    is its last committed token, rows 1..gamma_b its drafts); Q [sum gamma, V]:
    draft probabilities, sequence b's rows start at cu_rows[b] - b; drafts
    [sum gamma]: x_1..x_gamma per sequence; U [M]: uniforms (see module doc);
    cu_rows [B + 1].

    Returns n_acc [B] int32, out_tok [M] int32 (sequence b emits
    out_tok[cu_rows[b] : cu_rows[b] + n_acc[b] + 1]; the remaining slots are
    -1) and near_tie [B] int32.
    """
    P = np.asarray(P)
    Q = np.asarray(Q)
    drafts = np.asarray(drafts, np.int64)
    U = np.asarray(U)
    cu = np.asarray(cu_rows, np.int64)
    B = len(cu) - 1
    M = int(cu[-1])
    gam = (cu[1:] - cu[:-1] - 1).astype(np.int64)
    if np.any(gam < 0):
        raise ValueError("every sequence needs at least one verify row")
    r0 = cu[:-1]
    q0 = r0 - np.arange(B)
    n_acc = gam.copy()
    decided = np.zeros(B, dtype=bool)
    near = np.zeros(B, dtype=np.int64)
    gmax = int(gam.max()) if B else 0
    for i in range(gmax):
        live = (~decided) & (i < gam)
        if not np.any(live):
            break
        b = np.nonzero(live)[0]
        x = drafts[q0[b] + i]
        p_x = P[r0[b] + i, x]
        q_x = Q[q0[b] + i, x]
        u = U[r0[b] + i]
        gap = np.asarray(u, np.float64) * np.asarray(q_x, np.float64) - np.asarray(p_x, np.float64)
        near[b] += (np.abs(gap) < tie_eps)
        acc = accept_mask(p_x, q_x, u)
        rej = b[~acc]
        n_acc[rej] = i
        decided[rej] = True
    # final distribution per sequence: residual at the first rejection, else the bonus row
    t = np.zeros(B, dtype=np.int64)
    if B:
        rejected = n_acc < gam
        fin_rows = r0 + n_acc
        u_fin = U[r0 + gam]
        W = np.empty((B, P.shape[1]), dtype=np.float64)
        if np.any(rejected):
            rb = np.nonzero(rejected)[0]
            W[rb] = correction_distribution(P[fin_rows[rb]], Q[q0[rb] + n_acc[rb]])
        if np.any(~rejected):
            ab = np.nonzero(~rejected)[0]
            W[ab] = np.asarray(P[fin_rows[ab]], np.float64)
        t, near_pick = inverse_cdf_pick(W, u_fin, tie_eps)
        near += near_pick
    out = np.full(M, -1, dtype=np.int64)
    for k in range(gmax + 1):
        b = np.nonzero(k < n_acc)[0]
        out[r0[b] + k] = drafts[q0[b] + k]
        b = np.nonzero(k == n_acc)[0]
        out[r0[b] + k] = t[b]
    return n_acc.astype(np.int32), out.astype(np.int32), near.astype(np.int32)
