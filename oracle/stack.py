"""fp64 verify pass of a Qwen3-8B-shaped decoder stack (test infrastructure only).

The pages fix the target's shape (36 layers, 8 key/value heads with grouped
query attention, "Speculative Decoding Spends Arithmetic You May Not Have",
"Why a better draft model can be a worse deal") and that all gamma+1 rows go
through ONE forward pass (Algorithm 1).  The layer internals are this
project's reading: pre-RMSNorm (eps 1e-6), RoPE (theta 1e6, rotate-half) on
q and k, causal GQA attention over the cache, SwiGLU MLP, residual adds, a
final RMSNorm and the LM head.

bf16 rounding (one reading, fixed whatever plan a kernel takes): a layer is the
chain of steps RMSNorm -> QKV projection with RoPE -> attention -> O projection
+ residual -> RMSNorm -> gate/up projection with the SwiGLU activation -> down
projection + residual, and exactly the tensors one step hands to the next are
rounded to bf16: h, q / k / v (q and k after their rotation), o, x, h, the
activation a, x.  Quantities inside a step (the unrotated q and k, gate and
up, attention scores and weights) stay in fp64.  The logits are left
unrounded.  A kernel plan that stores more (gate|up between two launches, q
and k before a separate rotation) or less (a norm folded into the next
product) rounds elsewhere; the GPU tests hold every plan to this one reading
within the chain tolerance that tests/test_oracle_chain_tolerance.py derives
and pins on the CPU.
"""
from dataclasses import dataclass, field

import numpy as np

from . import ops
from .bf16 import decode, round_to_bf16 as r16


@dataclass
class Dims:
    d: int = 4096
    Hq: int = 32
    Hkv: int = 8
    D: int = 128
    I: int = 12288
    V: int = 151936
    layers: int = 36
    eps: float = 1e-6
    theta: float = 1e6


@dataclass
class LayerWeights:
    """bf16 bit patterns (uint16); decoded per matrix on use."""
    w_qkv: np.ndarray            # [(Hq + 2 Hkv) D, d]
    w_o: np.ndarray              # [d, Hq D]
    w_gu: np.ndarray             # [2 I, d]   gate rows then up rows
    w_down: np.ndarray           # [d, I]
    attn_norm: np.ndarray        # [d]
    mlp_norm: np.ndarray         # [d]


@dataclass
class StackWeights:
    layers: list = field(default_factory=list)
    final_norm: np.ndarray | None = None
    w_lm: np.ndarray | None = None   # [V, d]


def layer_forward(x, lw: LayerWeights, dims: Dims, cu_rows, ctx_len, Kc, Vc):
    """One decoder layer over the packed verify rows.

    x [M, d] (bf16 values, fp64); Kc/Vc [B, Hkv, cap, D] this layer's cache.
    Returns (x', Kc', Vc').
    """
    M = x.shape[0]
    Hq, Hkv, D = dims.Hq, dims.Hkv, dims.D
    pos = np.concatenate([ctx_len[b] + np.arange(cu_rows[b + 1] - cu_rows[b])
                          for b in range(len(cu_rows) - 1)]) if M else np.zeros(0)
    h = r16(ops.rmsnorm(x, decode(lw.attn_norm), dims.eps))
    qkv = ops.linear(h, decode(lw.w_qkv))
    q = qkv[:, :Hq * D].reshape(M, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(M, Hkv, D)
    v = r16(qkv[:, (Hq + Hkv) * D:]).reshape(M, Hkv, D)
    q = r16(ops.rope(q, pos, dims.theta))
    k = r16(ops.rope(k, pos, dims.theta))
    o, Kc, Vc = ops.verify_attention(q, k, v, cu_rows, Kc, Vc, ctx_len, 1.0 / np.sqrt(D))
    o = r16(o)
    x = r16(ops.linear(o.reshape(M, Hq * D), decode(lw.w_o), residual=x))
    h = r16(ops.rmsnorm(x, decode(lw.mlp_norm), dims.eps))
    gu = ops.linear(h, decode(lw.w_gu))
    a = r16(ops.silu_mul(gu[:, :dims.I], gu[:, dims.I:]))
    x = r16(ops.linear(a, decode(lw.w_down), residual=x))
    return x, Kc, Vc


def head_logits(x, sw: StackWeights, dims: Dims):
    """Final RMSNorm and LM head: logits [M, V] in fp64 (unrounded)."""
    h = r16(ops.rmsnorm(x, decode(sw.final_norm), dims.eps))
    return ops.linear(h, decode(sw.w_lm))


def verify_pass(x0, sw: StackWeights, dims: Dims, cu_rows, ctx_len, Kcaches, Vcaches,
                n_layers: int | None = None):
    """Run the stack once over all packed verify rows.

    Returns (final hidden x [M, d], logits [M, V] or None if there is no LM
    head, updated caches).
    """
    x = np.asarray(x0, dtype=np.float64)
    Kc = list(Kcaches)
    Vc = list(Vcaches)
    L = len(sw.layers) if n_layers is None else n_layers
    for li in range(L):
        x, Kc[li], Vc[li] = layer_forward(x, sw.layers[li], dims, cu_rows, ctx_len, Kc[li], Vc[li])
    logits = head_logits(x, sw, dims) if sw.w_lm is not None else None
    return x, logits, Kc, Vc


def decode_steps(x0, sw: StackWeights, dims: Dims, cu_rows, ctx_len, Kcaches, Vcaches):
    """The same rows as gamma_b+1 sequential single-position decode steps.

    Step j feeds row j of every sequence that has one, at context ctx_b + j,
    with the cache written by steps 0..j-1.  Returns (x [M, d], logits or None,
    caches) in the packed row order of ``verify_pass``.
    """
    x0 = np.asarray(x0, dtype=np.float64)
    cu = np.asarray(cu_rows)
    ctx = np.asarray(ctx_len)
    B = len(cu) - 1
    rows = cu[1:] - cu[:-1]
    Kc = [np.array(k, dtype=np.float64, copy=True) for k in Kcaches]
    Vc = [np.array(v, dtype=np.float64, copy=True) for v in Vcaches]
    X = np.zeros_like(x0)
    logits = None
    for j in range(int(rows.max())):
        seqs = np.nonzero(rows > j)[0]
        idx = cu[seqs] + j
        sub_cu = np.arange(len(seqs) + 1)
        sub_ctx = ctx[seqs] + j
        x = x0[idx]
        sub_K = [k[seqs] for k in Kc]
        sub_V = [v[seqs] for v in Vc]
        x, lg, sub_K, sub_V = verify_pass(x, sw, dims, sub_cu, sub_ctx, sub_K, sub_V)
        for li in range(len(Kc)):
            Kc[li][seqs] = sub_K[li]
            Vc[li][seqs] = sub_V[li]
        X[idx] = x
        if lg is not None:
            if logits is None:
                logits = np.zeros((x0.shape[0], lg.shape[1]))
            logits[idx] = lg
    return X, logits, Kc, Vc


def draft_decode(tok0, table, sw: StackWeights, dims: Dims, ctx_len, Kcaches, Vcaches, U, temperature: float,
                 gamma: int):
    """gamma autoregressive decode steps of a (draft-shaped) stack for B sequences, one row each.

    The step before the verify pass ("Speculative Decoding Spends Arithmetic You May Not Have",
    Algorithm 1: the draft model proposes x_1 .. x_gamma one at a time, keeping q_1 .. q_gamma).
    Step i feeds the embedding row of each sequence's current token (table [V, d] bf16 bits;
    the last committed token at step 0) at position ctx_b + i, runs the stack and the LM head
    (sw.w_lm), forms q = softmax(logits / T) (one-hot argmax at T = 0) and draws the next token
    with the sampler's inverse CDF and U[i, b].  Returns (q [B, gamma, V] fp64, drafts [B, gamma]
    int64, logits [B, gamma, V] fp64, caches).
    """
    from . import ops
    from .sampler import inverse_cdf_pick
    tok = np.asarray(tok0, np.int64).copy()
    B = len(tok)
    emb = decode(np.asarray(table))
    cu = np.arange(B + 1)
    ctx = np.asarray(ctx_len, np.int64)
    Kc = [np.array(k, dtype=np.float64, copy=True) for k in Kcaches]
    Vc = [np.array(v, dtype=np.float64, copy=True) for v in Vcaches]
    V = emb.shape[0]
    q = np.zeros((B, gamma, V))
    logits = np.zeros((B, gamma, V))
    drafts = np.zeros((B, gamma), np.int64)
    for i in range(gamma):
        x = emb[tok]
        _, lg, Kc, Vc = verify_pass(x, sw, dims, cu, ctx + i, Kc, Vc)
        p = ops.target_probs(lg, temperature)
        t, _ = inverse_cdf_pick(p, np.asarray(U[i], np.float64), 0.0)
        q[:, i] = p
        logits[:, i] = lg
        drafts[:, i] = t
        tok = t
    return q, drafts, logits, Kc, Vc
