"""Exact fp64 definitions of the verify pass's operations (test infrastructure only).

Inputs are float64 arrays holding bf16 values (decode them with
``oracle.bf16.decode``).  Outputs are float64 and unrounded; callers that
chain operations round with ``oracle.bf16.round_to_bf16`` where the CUDA
path stores bf16.
"""
import numpy as np


def linear(X: np.ndarray, W: np.ndarray, residual: np.ndarray | None = None) -> np.ndarray:
    """Y = X W^T (+ residual), W in nn.Linear layout [N, K].

    One weight read serves all M rows of the verify pass: the pass scores the
    gamma+1 positions together ("Speculative Decoding Spends Arithmetic You
    May Not Have", "The speedup is borrowed, and there is a lender"; "How
    Speculative Decoding Works (and When It Doesn't)", "Prefill and Decode":
    the layer cost scales with M, the weight read does not).
    """
    X = np.asarray(X, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    if X.shape[1] != W.shape[1]:
        raise ValueError("inner dimensions differ")
    Y = X @ W.T
    if residual is not None:
        Y = Y + np.asarray(residual, dtype=np.float64)
    return Y


def rmsnorm(x: np.ndarray, weight: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * weight, per row (last axis)."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(weight, dtype=np.float64)


def rope(x: np.ndarray, positions: np.ndarray, theta: float = 1e6) -> np.ndarray:
    """Rotary position embedding, rotate-half pairing (i, i + D/2).

    x: [M, H, D]; positions: [M] absolute token positions.  Frequency of
    pair i is theta^(-2i/D).
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / D)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu_mul(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """SwiGLU activation: silu(gate) * up, silu(g) = g / (1 + exp(-g))."""
    g = np.asarray(gate, dtype=np.float64)
    return g / (1.0 + np.exp(-g)) * np.asarray(up, dtype=np.float64)


def verify_attention(Q, Knew, Vnew, cu_rows, Kcache, Vcache, ctx_len, scale):
    """Causal GQA attention of each sequence's gamma_b+1 verify rows.

    Row j of sequence b sits at position ctx_b + j.  It attends the ctx_b
    committed keys in the cache plus new keys 0..j of its own block, so the
    rows see exactly what gamma+1 sequential decode steps would see
    ("Speculative Decoding Spends Arithmetic You May Not Have", Algorithm 1:
    p_1 .. p_{gamma+1} from Mp(prefix) .. Mp(prefix + [x_1..x_gamma]); the
    cache read serves every query position, "The speedup is borrowed").

    Q [M, Hq, D]; Knew/Vnew [M, Hkv, D]; Kcache/Vcache [B, Hkv, cap, D].
    Query head h reads kv head h // (Hq // Hkv).
    Returns (O [M, Hq, D], Kcache', Vcache') with the new keys/values
    written at positions ctx_b .. ctx_b + gamma_b.
    """
    Q = np.asarray(Q, dtype=np.float64)
    Knew = np.asarray(Knew, dtype=np.float64)
    Vnew = np.asarray(Vnew, dtype=np.float64)
    Kc = np.array(Kcache, dtype=np.float64, copy=True)
    Vc = np.array(Vcache, dtype=np.float64, copy=True)
    M, Hq, D = Q.shape
    Hkv = Knew.shape[1]
    group = Hq // Hkv
    O = np.zeros((M, Hq, D), dtype=np.float64)
    B = len(cu_rows) - 1
    for b in range(B):
        r0, r1 = int(cu_rows[b]), int(cu_rows[b + 1])
        ctx = int(ctx_len[b])
        n = r1 - r0
        Kc[b, :, ctx:ctx + n, :] = Knew[r0:r1].transpose(1, 0, 2)
        Vc[b, :, ctx:ctx + n, :] = Vnew[r0:r1].transpose(1, 0, 2)
        for h in range(Hq):
            kv = h // group
            keys = Kc[b, kv, :ctx + n, :]
            vals = Vc[b, kv, :ctx + n, :]
            s = (Q[r0:r1, h, :] @ keys.T) * scale          # [n, ctx + n]
            # row j may see keys 0 .. ctx + j
            visible = np.arange(ctx + n)[None, :] <= (ctx + np.arange(n))[:, None]
            s = np.where(visible, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            w = np.exp(s)
            w = w / w.sum(axis=1, keepdims=True)
            O[r0:r1, h, :] = w @ vals
    return O, Kc, Vc


def target_probs(logits: np.ndarray, temperature: float) -> np.ndarray:
    """p = softmax(z / T) per row; T == 0 is greedy: one-hot at argmax(z).

    Greedy ties go to the lowest index.  ("How Speculative Decoding Works
    (and When It Doesn't)", "Exactness is a choice": at temperature zero the
    target distribution collapses to its argmax.)
    """
    z = np.asarray(logits, dtype=np.float64)
    if temperature == 0.0:
        p = np.zeros_like(z)
        p[np.arange(z.shape[0]), np.argmax(z, axis=1)] = 1.0   # argmax: first max
        return p
    s = z / temperature
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=1, keepdims=True)
