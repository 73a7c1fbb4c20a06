"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds *no* arithmetic of the verify method (no linear layer, no
attention, no target softmax, no acceptance rule).  It only draws random
numbers and packs them into the layouts the library and the oracle both read:

* bf16 tensors are returned as ``uint16`` bit patterns (numpy), so each side
  decodes them with its own code;
* uniforms for the acceptance test and the final draw are fp32 values in
  (0, 1) built from a Philox-4x64 stream: ``u = (2*(bits >> 41) + 1) * 2**-24``,
  which is exact in fp32 and never 0 or 1;
* ragged verify batches are described by ``gammas`` (drafts per sequence),
  ``cu_rows`` (prefix sum of gamma_b + 1) and ``ctx_len`` (committed context).

The draft distribution ``q`` is the draft model's output, an *input* of the
verify step.  ``draft_distribution`` builds it from logits handed in by the
caller (target-like logits plus Gaussian noise), with its own softmax; the
draft tokens are drawn from ``q`` by inverse CDF on a separate Philox stream.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "philox",
    "uniforms_f32",
    "normal_bf16_bits",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "ragged_batch",
    "draft_distribution",
    "RaggedBatch",
]


def philox(seed: int) -> np.random.Generator:
    """numpy Generator on the Philox-4x64-10 bit generator, keyed by ``seed``."""
    return np.random.Generator(np.random.Philox(int(seed)))


def uniforms_f32(seed: int, n: int) -> np.ndarray:
    """``n`` fp32 uniforms in (0, 1) from Philox(seed): (2*(b>>41)+1)*2^-24."""
    bits = philox(seed).bit_generator.random_raw(int(n)).astype(np.uint64)
    k = (bits >> np.uint64(41)).astype(np.float64)
    return ((2.0 * k + 1.0) * 2.0 ** -24).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((b >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((b + rounding) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16_bits(seed: int, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) samples rounded to bf16, as uint16 bit patterns."""
    x = philox(seed).standard_normal(size=shape, dtype=np.float32) * np.float32(std)
    return f32_to_bf16_bits(x)


class RaggedBatch:
    """Shape of one verify round: per-sequence draft counts and contexts."""

    def __init__(self, gammas, ctx_len, cap: int | None = None):
        self.gammas = np.asarray(gammas, dtype=np.int32)
        self.ctx_len = np.asarray(ctx_len, dtype=np.int32)
        rows = self.gammas + 1
        self.cu_rows = np.zeros(len(rows) + 1, dtype=np.int32)
        self.cu_rows[1:] = np.cumsum(rows)
        self.B = int(len(rows))
        self.M = int(self.cu_rows[-1])
        self.n_drafts = int(self.gammas.sum())
        self.max_rows = int(rows.max()) if self.B else 0
        need = int((self.ctx_len + rows).max()) if self.B else 0
        self.cap = int(cap) if cap is not None else need
        if self.cap < need:
            raise ValueError("cache capacity below ctx_len + gamma + 1")

    @property
    def q_rows(self) -> np.ndarray:
        """Index of each sequence's first draft row in the packed q/draft arrays."""
        return (self.cu_rows[:-1] - np.arange(self.B, dtype=np.int32)).astype(np.int32)


def ragged_batch(seed: int, B: int, gamma_lo: int, gamma_hi: int,
                 ctx_lo: int, ctx_hi: int, cap: int | None = None) -> RaggedBatch:
    """gamma_b ~ U{gamma_lo..gamma_hi}, ctx_b ~ U{ctx_lo..ctx_hi}, seeded."""
    g = philox(seed)
    gammas = g.integers(gamma_lo, gamma_hi + 1, size=B)
    ctx = g.integers(ctx_lo, ctx_hi + 1, size=B)
    return RaggedBatch(gammas, ctx, cap)


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def draft_distribution(logits: np.ndarray, batch: RaggedBatch, sigma: float,
                       temperature: float, seed: int):
    """Draft-model stand-in: q = softmax((z + N(0, sigma^2)) / T) per draft row.

    ``logits`` are target-like logits for all M verify rows (fp64 or fp32,
    shape [M, V]); draft row i of sequence b uses verify row cu_rows[b] + i.
    With T == 0 the draft is greedy (one-hot at the argmax of z + noise).
    Returns q [n_drafts, V] fp32 and the draft tokens [n_drafts] int32 drawn
    from q by inverse CDF with uniforms from Philox(seed + 1).
    """
    V = logits.shape[1]
    rows = np.concatenate([np.arange(batch.cu_rows[b], batch.cu_rows[b] + batch.gammas[b])
                           for b in range(batch.B)]) if batch.n_drafts else np.zeros(0, np.int64)
    z = logits[rows].astype(np.float64)
    noise = philox(seed).standard_normal(size=z.shape)
    z = z + sigma * noise
    if temperature == 0.0:
        q = np.zeros_like(z)
        q[np.arange(len(rows)), np.argmax(z, axis=1)] = 1.0
    else:
        q = _softmax_rows(z / temperature)
    q32 = q.astype(np.float32)
    c = np.cumsum(q32.astype(np.float64), axis=1)
    u = uniforms_f32(seed + 1, len(rows)).astype(np.float64) * c[:, -1]
    tok = np.minimum((c <= u[:, None]).sum(axis=1), V - 1)
    # never draft a token the draft itself gives zero probability
    for i in np.nonzero(q32[np.arange(len(rows)), tok] == 0)[0]:
        tok[i] = int(np.argmax(q32[i]))
    return q32, tok.astype(np.int32)


def ngram_histories(seed: int, B: int, len_lo: int, len_hi: int, vocab: int, copy_frac: float):
    """Packed token histories for the n-gram drafter: tokens [sum L] int32 and cu_len [B+1].

    Each history (length ~ U[len_lo, len_hi]) is built from segments of 8..64 tokens; a segment
    is, with probability copy_frac, a span copied from earlier in the same history (the
    copy-heavy regime: editing, quoting, repeating the prompt), else fresh uniform tokens.
    """
    rng = philox(seed)
    lens = rng.integers(len_lo, len_hi + 1, size=B)
    out = []
    for L in lens:
        h = []
        while len(h) < L:
            seg = int(rng.integers(8, 65))
            if h and len(h) > 16 and rng.random() < copy_frac:
                start = int(rng.integers(0, len(h) - 8))
                span = h[start:start + seg]
                h.extend(span)
            else:
                h.extend(int(t) for t in rng.integers(0, vocab, size=seg))
        out.append(np.asarray(h[:L], np.int32))
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum([len(x) for x in out])
    return np.concatenate(out) if out else np.zeros(0, np.int32), cu
