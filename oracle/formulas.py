"""Closed forms the pages print about a verify round (test infrastructure only).

These serve the reporting side (mean tokens per round, acceptance metrics,
break-even lines) and pin the sampler statistically.
"""
import numpy as np


def expected_tokens(alpha: float, gamma: int) -> float:
    """E[tokens per round] = (1 - alpha^(gamma+1)) / (1 - alpha) under i.i.d. acceptance.

    "Speculative Decoding Spends Arithmetic You May Not Have", "Why gamma has
    a ceiling" (printed as alpha^gamma+1, read as alpha^(gamma+1)); equal to
    1 + alpha + ... + alpha^gamma ("05 · Speculative Decoding", "The
    economics — one formula that decides everything").
    """
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def arithmetic_increase(alpha: float, gamma: int, c_hat: float) -> float:
    """Theorem 3.11's expected increase in arithmetic: (1-a)(g c + g + 1)/(1 - a^(g+1)).

    "Speculative Decoding Spends Arithmetic You May Not Have", "The speedup is
    borrowed, and there is a lender".
    """
    return (1.0 - alpha) * (gamma * c_hat + gamma + 1) / (1.0 - alpha ** (gamma + 1))


def speedup_model(alpha: float, k: int, c: float) -> float:
    """speedup = (1 + alpha + ... + alpha^k) / (1 + k c).

    "05 · Speculative Decoding", "The economics — one formula that decides
    everything".
    """
    return sum(alpha ** i for i in range(k + 1)) / (1.0 + k * c)


def break_even_alpha(k: int, c: float, iters: int = 60) -> float:
    """Smallest alpha with speedup_model(alpha, k, c) >= 1, by bisection on [0, 1]."""
    lo, hi = 0.0, 1.0
    if speedup_model(0.0, k, c) >= 1.0:
        return 0.0
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if speedup_model(mid, k, c) < 1.0:
            lo = mid
        else:
            hi = mid
    return lo


def verify_cost_rate(p: float, t_verify_ms: float, t_draft_ms: float) -> float:
    """Tokens per ms of single-draft speculation: (1 + p) / (T_verify + T_draft).

    Speculative decoding verify cost (ariaki.me), section 2 "The division".
    """
    return (1.0 + p) / (t_verify_ms + t_draft_ms)


def verify_speedup(p: float, t_decode_ms: float, t_verify_ms: float, t_draft_ms: float) -> float:
    """speedup = (1 + p) T_decode / (T_verify + T_draft) (same section)."""
    return (1.0 + p) * t_decode_ms / (t_verify_ms + t_draft_ms)


def verify_break_even_ms(p: float, t_decode_ms: float, t_draft_ms: float) -> float:
    """Largest T_verify that still breaks even: (1 + p) T_decode - T_draft (section 2.2)."""
    return (1.0 + p) * t_decode_ms - t_draft_ms


def acceptance_probability(p: np.ndarray, q: np.ndarray) -> float:
    """alpha = sum_x min(p(x), q(x)) = 1 - TV(p, q).

    "How Speculative Decoding Works (and When It Doesn't)", "Why the output
    doesn't change": the accepted mass is what the two distributions share.
    """
    return float(np.minimum(np.asarray(p, np.float64), np.asarray(q, np.float64)).sum())


def spec_metrics(n_acc: np.ndarray, gammas: np.ndarray) -> dict:
    """vLLM-style acceptance metrics over a set of rounds.

    Mean acceptance length = 1 + accepted / rounds; acceptance rate =
    accepted / drafted; per-position rate i = rounds whose first i+1 drafts
    were all accepted / rounds (counted over every round, so unconditional).
    ("Speculative Decoding Spends Arithmetic You May Not Have", "Checking it
    on a real system".)
    """
    n_acc = np.asarray(n_acc, np.int64)
    gammas = np.asarray(gammas, np.int64)
    rounds = len(n_acc)
    accepted = int(n_acc.sum())
    drafted = int(gammas.sum())
    gmax = int(gammas.max()) if rounds else 0
    per_pos = [float(np.sum(n_acc > i)) / rounds for i in range(gmax)]
    return {
        "rounds": rounds,
        "accepted": accepted,
        "drafted": drafted,
        "mean_acceptance_length": 1.0 + accepted / rounds if rounds else 0.0,
        "acceptance_rate": accepted / drafted if drafted else 0.0,
        "per_position": per_pos,
    }
