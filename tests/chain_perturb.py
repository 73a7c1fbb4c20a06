"""Perturbation model of a verify layer, for deriving the chain tolerance (CPU tests only).

The oracle (oracle.stack) computes one reading of a layer in fp64, rounding to bf16 exactly at
the tensors one step hands to the next.  A GPU plan differs from it in ways that are all correct
arithmetic: fp32 sums instead of fp64, softmax weights rounded to bf16 before the P.V product,
and rounding points of its own (gate|up stored between two launches, q and k stored before a
separate rotation, a norm folded into the next product so h is never stored).  This module
re-composes one layer from the oracle's primitives with those differences switched on one by
one, so that a test can measure how far correct plans drift from the reading after L layers, and
plants mistakes (off-by-one positions, a rotation the wrong way, a wrong attention scale, a
dropped residual, gate and up swapped) so that it can check the bar still catches real errors.
It imports the oracle; nothing outside tests/ uses it.
"""
import numpy as np

from oracle import bf16 as obf, ops as oops

r16 = obf.round_to_bf16
dec = obf.decode


def _f32(a):
    return np.asarray(a, np.float32)


def layer(x, lw, dims, cu, ctx, Kc, Vc, f32=False, p_bf16=False, gu_round=False, qk_round=False,
          fold_norm=False, mistake=None):
    """One layer with the chosen plan differences (see the module docstring)."""
    M = x.shape[0]
    Hq, Hkv, D = dims.Hq, dims.Hkv, dims.D
    pos = np.concatenate([ctx[b] + np.arange(cu[b + 1] - cu[b]) for b in range(len(cu) - 1)])
    if mistake == "position":
        pos = pos + 1

    def lin(a, w, res=None):
        y = (_f32(a) @ _f32(dec(w)).T).astype(np.float64) if f32 else a @ dec(w).T
        return y if res is None else y + res

    def norm(a, w):
        if not f32:
            return oops.rmsnorm(a, dec(w), dims.eps)
        a32 = _f32(a)
        ms = np.mean(a32 * a32, axis=-1, keepdims=True, dtype=np.float32)
        return (a32 / np.sqrt(ms + np.float32(dims.eps)) * _f32(dec(w))).astype(np.float64)

    hn = norm(x, lw.attn_norm)
    h = hn if fold_norm else r16(hn)
    qkv = lin(h, lw.w_qkv)
    if qk_round:
        qkv = r16(qkv)
    q = qkv[:, :Hq * D].reshape(M, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(M, Hkv, D)
    v = r16(qkv[:, (Hq + Hkv) * D:]).reshape(M, Hkv, D)
    q = r16(oops.rope(q, -pos if mistake == "rotation" else pos, dims.theta))
    k = r16(oops.rope(k, pos, dims.theta))
    scale = 1.0 / D if mistake == "scale" else 1.0 / np.sqrt(D)
    if f32 or p_bf16:
        Kc, Vc = np.array(Kc, copy=True), np.array(Vc, copy=True)
        O = np.zeros((M, Hq, D))
        G = Hq // Hkv
        for b in range(len(cu) - 1):
            r0, r1, c = int(cu[b]), int(cu[b + 1]), int(ctx[b])
            n = r1 - r0
            Kc[b, :, c:c + n] = k[r0:r1].transpose(1, 0, 2)
            Vc[b, :, c:c + n] = v[r0:r1].transpose(1, 0, 2)
            for hh in range(Hq):
                kv = hh // G
                s = (_f32(q[r0:r1, hh]) @ _f32(Kc[b, kv, :c + n]).T) * np.float32(scale)
                vis = np.arange(c + n)[None, :] <= (c + np.arange(n))[:, None]
                s = np.where(vis, s, -np.inf).astype(np.float32)
                w = np.exp(s - s.max(axis=1, keepdims=True)).astype(np.float32)
                l = w.sum(axis=1, keepdims=True, dtype=np.float32)
                P = r16(w) if p_bf16 else w.astype(np.float64)
                O[r0:r1, hh] = (_f32(P) @ _f32(Vc[b, kv, :c + n])).astype(np.float64) / l
        o = O
    else:
        o, Kc, Vc = oops.verify_attention(q, k, v, cu, Kc, Vc, ctx, scale)
    o = r16(o)
    x1 = r16(lin(o.reshape(M, Hq * D), lw.w_o, None if mistake == "residual" else x))
    hn = norm(x1, lw.mlp_norm)
    h = hn if fold_norm else r16(hn)
    gu = lin(h, lw.w_gu)
    if gu_round:
        gu = r16(gu)
    g, u = gu[:, :dims.I], gu[:, dims.I:]
    if mistake == "gate_up":
        g, u = u, g
    if f32:
        g32 = _f32(g)
        a = (g32 / (np.float32(1) + np.exp(-g32)) * _f32(u)).astype(np.float64)
    else:
        a = oops.silu_mul(g, u)
    x2 = r16(lin(r16(a), lw.w_down, x1))
    return x2, Kc, Vc


def stack(x0, sw, dims, cu, ctx, Kcs, Vcs, **plan):
    x, Kc, Vc = np.asarray(x0, np.float64), list(Kcs), list(Vcs)
    for li, lw in enumerate(sw.layers):
        x, Kc[li], Vc[li] = layer(x, lw, dims, cu, ctx, Kc[li], Vc[li], **plan)
    return x, Kc, Vc


# the GPU-like plans: fp32 arithmetic and bf16 P throughout, plus each plan's own rounding points
PLANS = {
    "fp32 sums, bf16 P": dict(f32=True, p_bf16=True),
    "+ gate|up stored": dict(f32=True, p_bf16=True, gu_round=True),
    "+ q, k stored before RoPE": dict(f32=True, p_bf16=True, qk_round=True),
    "+ norm folded": dict(f32=True, p_bf16=True, fold_norm=True),
    "all of them": dict(f32=True, p_bf16=True, gu_round=True, qk_round=True, fold_norm=True),
}
MISTAKES = ("position", "rotation", "scale", "residual", "gate_up")


def floor_needed(got, ref, rel):
    """Smallest c with |got - ref| <= rel |ref| + c rms(ref) element-wise."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max((np.abs(got - ref) - rel * np.abs(ref)) / rms))
