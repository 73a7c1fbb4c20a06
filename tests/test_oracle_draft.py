"""Pins of the oracle's draft decode loop (oracle/stack.py draft_decode)."""
import numpy as np

import synth
from oracle import bf16 as obf, ops as oops, sampler as osamp, stack as ostack


def _stack(seed, L=2, d=32, Hq=4, Hkv=2, D=8, I=48, V=40):
    dims = ostack.Dims(d=d, Hq=Hq, Hkv=Hkv, D=D, I=I, V=V, layers=L)
    ones = synth.f32_to_bf16_bits(np.ones(d, np.float32))
    layers = []
    for li in range(L):
        s = seed + 10 * li
        layers.append(ostack.LayerWeights(
            synth.normal_bf16_bits(s + 1, ((Hq + 2 * Hkv) * D, d), 0.2), synth.normal_bf16_bits(s + 2, (d, Hq * D), 0.2),
            synth.normal_bf16_bits(s + 3, (2 * I, d), 0.2), synth.normal_bf16_bits(s + 4, (d, I), 0.2), ones, ones))
    table = synth.normal_bf16_bits(seed + 99, (V, d), 0.5)
    return dims, ostack.StackWeights(layers, ones, table), table


def test_draft_steps_equal_one_pass_over_the_drafted_rows():
    """q_i of step i equals the stack's distribution at row i of ONE pass over the rows
    [tok0, x_1 .. x_{gamma-1}] with the same caches (the pinned decode == verify equivalence),
    and each draft is the inverse-CDF pick of its own q row with U[i]."""
    dims, sw, table = _stack(5)
    B, gamma, cap = 3, 4, 16
    ctx = np.array([2, 5, 0])
    kc = [obf.decode(synth.normal_bf16_bits(50 + i, (B, dims.Hkv, cap, dims.D), 1.0)) for i in range(dims.layers)]
    vc = [obf.decode(synth.normal_bf16_bits(60 + i, (B, dims.Hkv, cap, dims.D), 1.0)) for i in range(dims.layers)]
    tok0 = np.array([1, 7, 30])
    U = synth.uniforms_f32(8, gamma * B).reshape(gamma, B)
    q, drafts, lg, _, _ = ostack.draft_decode(tok0, table, sw, dims, ctx, kc, vc, U, 0.9, gamma)
    emb = obf.decode(table)
    rows = np.concatenate([np.concatenate([[tok0[b]], drafts[b, :-1]]) for b in range(B)])
    cu = np.arange(B + 1) * gamma
    _, lg_pass, _, _ = ostack.verify_pass(emb[rows], sw, dims, cu, ctx, kc, vc)
    assert np.allclose(lg_pass.reshape(B, gamma, -1), lg, rtol=0, atol=1e-12)
    assert np.allclose(q, oops.target_probs(lg.reshape(B * gamma, -1), 0.9).reshape(B, gamma, -1))
    for i in range(gamma):
        t, _ = osamp.inverse_cdf_pick(q[:, i], U[i].astype(np.float64), 0.0)
        assert np.array_equal(t, drafts[:, i])


def test_greedy_drafts_follow_the_argmax_chain():
    dims, sw, table = _stack(9)
    B, gamma, cap = 2, 3, 8
    ctx = np.array([1, 3])
    kc = [np.zeros((B, dims.Hkv, cap, dims.D)) for _ in range(dims.layers)]
    vc = [np.zeros((B, dims.Hkv, cap, dims.D)) for _ in range(dims.layers)]
    U = synth.uniforms_f32(3, gamma * B).reshape(gamma, B)
    q, drafts, lg, _, _ = ostack.draft_decode(np.array([4, 5]), table, sw, dims, ctx, kc, vc, U, 0.0, gamma)
    assert np.array_equal(drafts, lg.argmax(axis=2))
    assert np.all(q.max(axis=2) == 1.0) and np.all(q.sum(axis=2) == 1.0)
