"""Pins of oracle.bf16 / oracle.ops / oracle.stack against definitions, invariants and brute force.

Each test is chosen so that a plausible slip (a transposed weight, an
off-by-one causal mask, a wrong GQA head map, a missing scale, a rotation in
the wrong direction, a dropped epsilon) fails it.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import bf16, ops, stack


# ------------------------------------------------------------------ bf16

def test_bf16_round_matches_library_conversion():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * s for s in (1e-3, 1.0, 1e3)])
    x = np.concatenate([x, np.float32([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38, 1e-40])])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = bf16.round_to_bf16(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_ties_to_even_and_decode():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even (1)
    assert bf16.round_to_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert bf16.round_to_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert bf16.round_to_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -30]))[0] == 1 + 2.0 ** -7
    assert bf16.decode(np.array([0x3F80, 0xC000, 0x0000], np.uint16)).tolist() == [1.0, -2.0, 0.0]
    bits = synth.f32_to_bf16_bits(np.float32([1.5, -0.1]))
    assert np.array_equal(bf16.decode(bits), bf16.round_to_bf16(np.array([1.5, np.float32(-0.1)])))


# ------------------------------------------------------------------ linear

def test_linear_exact_on_integers_bruteforce():
    rng = np.random.default_rng(1)
    M, N, K = 3, 5, 7                     # non-square: a transposed operand cannot fit
    X = rng.integers(-8, 9, size=(M, K))
    W = rng.integers(-8, 9, size=(N, K))
    R = rng.integers(-8, 9, size=(M, N))
    Y = ops.linear(X.astype(float), W.astype(float), R.astype(float))
    for m in range(M):
        for n in range(N):
            assert Y[m, n] == sum(int(X[m, k]) * int(W[n, k]) for k in range(K)) + int(R[m, n])
    with pytest.raises(ValueError):
        ops.linear(X.astype(float), W.T.astype(float))


# ------------------------------------------------------------------ glue

def test_rmsnorm_known_values():
    x = np.array([[3.0, 4.0]])
    y = ops.rmsnorm(x, np.array([1.0, 2.0]), eps=0.0)
    r = math.sqrt((9 + 16) / 2)
    assert np.allclose(y, [[3 / r, 8 / r]], rtol=0, atol=1e-15)
    # eps enters under the root
    y = ops.rmsnorm(np.array([[0.0, 0.0]]), np.ones(2), eps=1e-6)
    assert np.all(y == 0)
    y = ops.rmsnorm(np.array([[1e-3, 1e-3]]), np.ones(2), eps=1e-6)
    assert np.allclose(y, 1e-3 / math.sqrt(1e-6 + 1e-6), atol=1e-15)


def test_rope_rotation_properties():
    rng = np.random.default_rng(2)
    D = 16
    x = rng.standard_normal((6, 3, D))
    pos = np.array([0, 1, 5, 17, 400, 8191])
    y = ops.rope(x, pos, theta=1e6)
    assert np.allclose(y[0], x[0])                                   # position 0: identity
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1))   # rotation
    # pair 0 turns by exactly `pos` radians (frequency theta^0 = 1), counter-clockwise
    a, b = x[2, 0, 0], x[2, 0, D // 2]
    assert np.isclose(y[2, 0, 0], a * math.cos(5) - b * math.sin(5))
    assert np.isclose(y[2, 0, D // 2], b * math.cos(5) + a * math.sin(5))
    # pair i turns by pos * theta^(-2i/D)
    i = 3
    ang = 17 * 1e6 ** (-2 * i / D)
    assert np.isclose(y[3, 1, i], x[3, 1, i] * math.cos(ang) - x[3, 1, i + D // 2] * math.sin(ang))
    # relative property: <rope(q, m), rope(k, n)> depends on m - n only
    q = rng.standard_normal((1, 1, D)); k = rng.standard_normal((1, 1, D))
    d1 = np.sum(ops.rope(q, [10]) * ops.rope(k, [3]))
    d2 = np.sum(ops.rope(q, [1007]) * ops.rope(k, [1000]))
    assert np.isclose(d1, d2)


def test_silu_mul_values():
    g = np.array([0.0, 1.0, -1.0, 30.0])
    u = np.array([5.0, 2.0, 2.0, 1.0])
    y = ops.silu_mul(g, u)
    assert y[0] == 0.0
    assert np.isclose(y[1], 2.0 / (1 + math.exp(-1)))
    assert np.isclose(y[2], -2.0 / (1 + math.e))
    assert np.isclose(y[3], 30.0)


def test_target_probs():
    z = np.array([[0.0, math.log(2.0)], [1.0, 1.0]])
    p = ops.target_probs(z, 1.0)
    assert np.allclose(p[0], [1 / 3, 2 / 3]) and np.allclose(p[1], [0.5, 0.5])
    # temperature divides the logits
    assert np.allclose(ops.target_probs(z, 0.5), ops.target_probs(2 * z, 1.0))
    # shift invariance, and no overflow
    assert np.allclose(ops.target_probs(z + 1000.0, 1.0), p)
    # greedy: one-hot at argmax, ties to the lowest index
    g = ops.target_probs(np.array([[0.1, 0.9, 0.9, -1.0]]), 0.0)
    assert g.tolist() == [[0.0, 1.0, 0.0, 0.0]]


# ------------------------------------------------------------------ attention

def _attn_case(seed, gammas, ctx, Hq=4, Hkv=2, D=8, cap=None):
    rng = np.random.default_rng(seed)
    batch = synth.RaggedBatch(gammas, ctx, cap)
    M, B = batch.M, batch.B
    Q = rng.standard_normal((M, Hq, D))
    Kn = rng.standard_normal((M, Hkv, D))
    Vn = rng.standard_normal((M, Hkv, D))
    Kc = rng.standard_normal((B, Hkv, batch.cap, D))
    Vc = rng.standard_normal((B, Hkv, batch.cap, D))
    return batch, Q, Kn, Vn, Kc, Vc


def _bruteforce_row(q, keys, vals, scale):
    s = [scale * sum(q[d] * k[d] for d in range(len(q))) for k in keys]
    mx = max(s)
    w = [math.exp(v - mx) for v in s]
    tot = sum(w)
    return [sum(w[i] * vals[i][d] for i in range(len(keys))) / tot for d in range(len(q))]


def test_attention_bruteforce_small():
    batch, Q, Kn, Vn, Kc, Vc = _attn_case(3, [2, 0, 3], [3, 1, 0])
    O, Kc2, Vc2 = ops.verify_attention(Q, Kn, Vn, batch.cu_rows, Kc, Vc, batch.ctx_len, 0.5)
    for b in range(batch.B):
        r0 = batch.cu_rows[b]
        ctx = batch.ctx_len[b]
        for j in range(batch.gammas[b] + 1):
            for h in range(Q.shape[1]):
                kv = h // 2
                keys = [Kc[b, kv, t] for t in range(ctx)] + [Kn[r0 + t, kv] for t in range(j + 1)]
                vals = [Vc[b, kv, t] for t in range(ctx)] + [Vn[r0 + t, kv] for t in range(j + 1)]
                want = _bruteforce_row(Q[r0 + j, h], keys, vals, 0.5)
                assert np.allclose(O[r0 + j, h], want, atol=1e-12)
        # cache gets the new block at ctx .. ctx + gamma, the rest untouched
        n = batch.gammas[b] + 1
        assert np.array_equal(Kc2[b, :, ctx:ctx + n], Kn[r0:r0 + n].transpose(1, 0, 2))
        assert np.array_equal(Vc2[b, :, :ctx], Vc[b, :, :ctx])


def test_attention_causality_and_gqa_map():
    batch, Q, Kn, Vn, Kc, Vc = _attn_case(4, [4], [5], Hq=6, Hkv=3)
    O, _, _ = ops.verify_attention(Q, Kn, Vn, batch.cu_rows, Kc, Vc, batch.ctx_len, 0.3)
    # perturbing new key/value j changes rows >= j only
    for j in range(5):
        Kp = Kn.copy(); Vp = Vn.copy()
        Kp[j] += 1.0; Vp[j] -= 2.0
        O2, _, _ = ops.verify_attention(Q, Kp, Vp, batch.cu_rows, Kc, Vc, batch.ctx_len, 0.3)
        changed = np.any(np.abs(O2 - O) > 1e-12, axis=(1, 2))
        assert changed.tolist() == [r >= j for r in range(5)]
    # perturbing kv head 1 changes query heads 2, 3 only (group size 2)
    Kp = Kn.copy(); Kp[:, 1] += 1.0
    O2, _, _ = ops.verify_attention(Q, Kp, Vn, batch.cu_rows, Kc, Vc, batch.ctx_len, 0.3)
    changed = np.any(np.abs(O2 - O) > 1e-12, axis=(0, 2))
    assert changed.tolist() == [False, False, True, True, False, False]
    # cache positions >= ctx are ignored (stale entries never leak in)
    Kc2 = Kc.copy(); Kc2[:, :, 5:] = 1e9
    O2, _, _ = ops.verify_attention(Q, Kn, Vn, batch.cu_rows, Kc2, Vc, batch.ctx_len, 0.3)
    assert np.allclose(O2, O)


def test_attention_special_cases():
    # identical keys -> uniform weights -> mean of the visible values
    batch, Q, Kn, Vn, Kc, Vc = _attn_case(5, [2], [3], Hq=2, Hkv=1)
    Kc[:] = 0.7; Kn[:] = 0.7
    O, _, _ = ops.verify_attention(Q, Kn, Vn, batch.cu_rows, Kc, Vc, batch.ctx_len, 1.0)
    for j in range(3):
        vis = np.concatenate([Vc[0, 0, :3], Vn[:j + 1, 0]])
        assert np.allclose(O[j, 0], vis.mean(axis=0))
    # a single visible key (ctx 0, row 0) returns its value exactly
    batch, Q, Kn, Vn, Kc, Vc = _attn_case(6, [0], [0], Hq=2, Hkv=1)
    O, _, _ = ops.verify_attention(Q, Kn, Vn, batch.cu_rows, Kc, Vc, batch.ctx_len, 1.0)
    assert np.allclose(O[0, 0], Vn[0, 0]) and np.allclose(O[0, 1], Vn[0, 0])


# ------------------------------------------------------------------ stack

def _tiny_stack(seed, dims, L):
    sw = stack.StackWeights()
    qkv_rows = (dims.Hq + 2 * dims.Hkv) * dims.D
    for li in range(L):
        s = seed + 10 * li
        sw.layers.append(stack.LayerWeights(
            w_qkv=synth.normal_bf16_bits(s + 1, (qkv_rows, dims.d), 0.2),
            w_o=synth.normal_bf16_bits(s + 2, (dims.d, dims.Hq * dims.D), 0.2),
            w_gu=synth.normal_bf16_bits(s + 3, (2 * dims.I, dims.d), 0.2),
            w_down=synth.normal_bf16_bits(s + 4, (dims.d, dims.I), 0.2),
            attn_norm=synth.f32_to_bf16_bits(np.ones(dims.d, np.float32)),
            mlp_norm=synth.f32_to_bf16_bits(np.ones(dims.d, np.float32))))
    sw.final_norm = synth.f32_to_bf16_bits(np.ones(dims.d, np.float32))
    sw.w_lm = synth.normal_bf16_bits(seed + 999, (dims.V, dims.d), 0.2)
    return sw


def test_verify_pass_equals_sequential_decode():
    """One pass over gamma+1 rows == gamma+1 single-row decode steps (Algorithm 1's parallel line)."""
    dims = stack.Dims(d=32, Hq=4, Hkv=2, D=8, I=48, V=50, layers=2)
    sw = _tiny_stack(7, dims, 2)
    batch = synth.RaggedBatch([3, 0, 5], [4, 9, 1], cap=16)
    x0 = bf16.decode(synth.normal_bf16_bits(8, (batch.M, dims.d)))
    rng = np.random.default_rng(9)
    Kc = [bf16.round_to_bf16(rng.standard_normal((batch.B, dims.Hkv, batch.cap, dims.D))) for _ in range(2)]
    Vc = [bf16.round_to_bf16(rng.standard_normal((batch.B, dims.Hkv, batch.cap, dims.D))) for _ in range(2)]
    xv, lv, Kv, Vv = stack.verify_pass(x0, sw, dims, batch.cu_rows, batch.ctx_len, Kc, Vc)
    xd, ld, Kd, Vd = stack.decode_steps(x0, sw, dims, batch.cu_rows, batch.ctx_len, Kc, Vc)
    assert np.array_equal(xv, xd)
    assert np.allclose(lv, ld, rtol=0, atol=1e-12)
    for li in range(2):
        assert np.array_equal(Kv[li], Kd[li]) and np.array_equal(Vv[li], Vd[li])
    # and the positions matter: shifting every context by one changes the result
    xs, _, _, _ = stack.verify_pass(x0, sw, dims, batch.cu_rows, batch.ctx_len + 1, Kc, Vc)
    assert not np.allclose(xs, xv)
