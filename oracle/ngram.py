"""n-gram prompt-lookup drafter (test infrastructure only).

A drafter with no weights ("Speculative Decoding Spends Arithmetic You May Not
Have", the ladder and "Why a better draft model can be a worse deal"; "05 ·
Speculative Decoding", "Under the Hood" table row "N-gram": it matches the
recent context against earlier text and copies what followed; "Cheat Sheet":
num_speculative_tokens k and the match window prompt_lookup_min /
prompt_lookup_max).

Reading adopted for what the pages leave open, per sequence with token
history h[0 .. L-1]:

* window sizes are tried from n_max down to n_min, the first n that matches
  wins (longer matches are the more reliable guess);
* the pattern is the last n tokens, h[L-n .. L-1]; an occurrence is a start j
  with h[j .. j+n-1] equal to it and at least one token after it, j + n <= L-1
  (which excludes the pattern itself); overlapping occurrences count;
* of several occurrences the most recent one (largest j) is taken;
* the drafts are the tokens that followed it, h[j+n .. min(j+n+k, L) - 1]: up
  to k of them, fewer when the history ends first; no occurrence for any n
  gives no drafts.
"""
import numpy as np


def propose(history, k: int, n_min: int, n_max: int):
    """Drafts (int64 array, length 0 .. k) for one token history."""
    h = np.asarray(history, np.int64)
    L = len(h)
    for n in range(n_max, n_min - 1, -1):
        if n <= 0 or L - 1 - n < 0:
            continue
        pattern = h[L - n:]
        windows = np.lib.stride_tricks.sliding_window_view(h[:L - 1], n)   # starts 0 .. L-1-n
        hits = np.nonzero((windows == pattern).all(axis=1))[0]
        if hits.size:
            j = int(hits.max())
            return h[j + n:min(j + n + k, L)].copy()
    return np.zeros(0, np.int64)


def propose_batch(tokens, cu_len, k: int, n_min: int, n_max: int):
    """Packed histories (tokens [sum L], cu_len [B+1]) -> drafts [B, k] int32 (-1 padded) and
    n_drafts [B] int32."""
    tokens = np.asarray(tokens)
    cu = np.asarray(cu_len, np.int64)
    B = len(cu) - 1
    drafts = np.full((B, k), -1, np.int32)
    n = np.zeros(B, np.int32)
    for b in range(B):
        d = propose(tokens[cu[b]:cu[b + 1]], k, n_min, n_max)
        drafts[b, :len(d)] = d
        n[b] = len(d)
    return drafts, n
