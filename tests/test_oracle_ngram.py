"""Pins of the n-gram prompt-lookup drafter oracle (reading stated in oracle/ngram.py)."""
import numpy as np
import pytest

import synth
from oracle import ngram as NG


def brute(h, k, n_min, n_max):
    """Every start j and window n by plain loops, longest window first, latest start kept."""
    h = list(int(x) for x in h)
    L = len(h)
    for n in range(n_max, n_min - 1, -1):
        best = None
        for j in range(0, L):
            if j + n > L - 1:
                break
            if all(h[j + t] == h[L - n + t] for t in range(n)):
                best = j
        if best is not None:
            return h[best + n:best + n + k]
    return []


def test_hand_worked_cases():
    # pattern "7 8" (n = 2) last seen at j = 3 (j = 1 is earlier): copies 9 5 7 8
    assert list(NG.propose([1, 7, 8, 7, 8, 9, 5, 7, 8], 4, 1, 2)) == [9, 5, 7, 8]
    # k past the end of the history: "4 4" latest at j = 1 of [3 4 4 4]: only h[3] = 4 follows
    assert list(NG.propose([3, 4, 4, 4], 5, 2, 2)) == [4]
    h = [1, 7, 8, 2, 7, 8, 9, 5, 7, 8]
    # n = 3 "5 7 8" never occurred before; n = 2 "7 8" at j = 1 and j = 4 -> latest j = 4 -> 9 5 7 8
    assert list(NG.propose(h, 4, 2, 3)) == [9, 5, 7, 8]
    assert list(NG.propose(h, 2, 2, 3)) == [9, 5]
    # no earlier occurrence of any window: no drafts
    assert list(NG.propose([1, 2, 3, 4, 5], 4, 1, 3)) == []
    # the longer window wins over a later match of a shorter one: "3 1 2" at j = 0 (n = 3) -> 9;
    # the latest "1 2" (n = 2) would be j = 5 -> 4
    h = [3, 1, 2, 9, 9, 1, 2, 4, 3, 1, 2]
    assert list(NG.propose(h, 1, 2, 3)) == [9]
    assert list(NG.propose(h, 1, 2, 2)) == [4]
    # overlapping occurrences of a repeated token: "5 5" latest at j = 2 -> copies h[4] = 5
    assert list(NG.propose([5, 5, 5, 5, 5], 3, 2, 2)) == [5]
    # a history too short for any window
    assert list(NG.propose([4], 3, 1, 2)) == []


def test_matches_brute_force_on_small_alphabets():
    rng = np.random.default_rng(0)
    for trial in range(400):
        L = int(rng.integers(1, 60))
        h = rng.integers(0, int(rng.integers(2, 5)), size=L)
        k = int(rng.integers(1, 6))
        n_min = int(rng.integers(1, 4))
        n_max = n_min + int(rng.integers(0, 4))
        assert list(NG.propose(h, k, n_min, n_max)) == brute(h, k, n_min, n_max), (h, k, n_min, n_max)


def test_drafts_copy_what_followed_an_occurrence():
    rng = np.random.default_rng(1)
    for _ in range(200):
        h = rng.integers(0, 3, size=int(rng.integers(5, 80)))
        d = NG.propose(h, 5, 2, 4)
        if len(d) == 0:
            continue
        L = len(h)
        # some window n in [2, 4] and start j reproduce the pattern and are followed by d
        ok = any(j + n <= L - 1 and np.array_equal(h[j:j + n], h[L - n:]) and
                 np.array_equal(h[j + n:j + n + len(d)], d) for n in range(2, 5) for j in range(L))
        assert ok and 1 <= len(d) <= 5


def test_batch_packing_and_padding():
    hs = [[1, 2, 1, 2], [9], [4, 4, 4, 4, 4, 4]]
    cu = np.cumsum([0] + [len(h) for h in hs]).astype(np.int32)
    drafts, n = NG.propose_batch(np.concatenate(hs).astype(np.int32), cu, 3, 1, 2)
    for b, h in enumerate(hs):
        d = NG.propose(h, 3, 1, 2)
        assert n[b] == len(d) and list(drafts[b, :n[b]]) == list(d) and np.all(drafts[b, n[b]:] == -1)


def test_copy_heavy_synthetic_histories_match_often():
    """The generator's copy-heavy histories (spans repeated from earlier context) give drafts for
    most sequences; the uniform-random ones over a large vocabulary almost never do."""
    rng_seed = 3
    tokens, cu = synth.ngram_histories(rng_seed, B=32, len_lo=256, len_hi=1024, vocab=50000, copy_frac=0.8)
    _, n = NG.propose_batch(tokens, cu, 4, 3, 8)
    assert (n > 0).mean() > 0.5
    tokens, cu = synth.ngram_histories(rng_seed, B=32, len_lo=256, len_hi=1024, vocab=50000, copy_frac=0.0)
    _, n = NG.propose_batch(tokens, cu, 4, 3, 8)
    assert (n > 0).mean() < 0.2
