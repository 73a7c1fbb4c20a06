"""GPU parity of the layer glue, a small end-to-end stack, and the smallest verify round."""
import numpy as np
import pytest
import torch

import synth
from oracle import bf16 as obf, ops as oops, sampler as osamp, stack as ostack

from gpu_util import (PROB_ATOL, STACK_PROB_BOUND, assert_close_chain, assert_close_rel, bf16_dev, bits_of, dev,
                      f64_of_bf16)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N", [(1, 4096), (5, 512), (37, 4096), (3, 16384), (2, 8)])
def test_rmsnorm(lib, M, N):
    X = synth.normal_bf16_bits(M + N, (M, N), 3.0)
    w = synth.normal_bf16_bits(M + N + 1, (N,), 1.0)
    Y = lib.spec_rmsnorm(bf16_dev(X), bf16_dev(w), 1e-6)
    ref = oops.rmsnorm(obf.decode(X), obf.decode(w), 1e-6)
    assert_close_rel(f64_of_bf16(Y), ref, "rmsnorm", rel=1e-2)


def test_rope(lib):
    batch = synth.RaggedBatch([4, 0, 10], [8190, 0, 333])
    Hq, Hkv, D = 32, 8, 128
    Qb = synth.normal_bf16_bits(1, (batch.M, Hq * D), 1.0)
    Kb = synth.normal_bf16_bits(2, (batch.M, Hkv * D), 1.0)
    Qd, Kd = bf16_dev(Qb), bf16_dev(Kb)
    lib.spec_rope(Qd, Kd, dev(batch.cu_rows), dev(batch.ctx_len), D, 1e6)
    pos = np.concatenate([batch.ctx_len[b] + np.arange(batch.gammas[b] + 1) for b in range(batch.B)])
    qr = oops.rope(obf.decode(Qb).reshape(batch.M, Hq, D), pos, 1e6).reshape(batch.M, -1)
    kr = oops.rope(obf.decode(Kb).reshape(batch.M, Hkv, D), pos, 1e6).reshape(batch.M, -1)
    assert_close_rel(f64_of_bf16(Qd), qr, "rope q", rel=1e-2)
    assert_close_rel(f64_of_bf16(Kd), kr, "rope k", rel=1e-2)


def test_rope_unaligned_heads(lib):
    """Head size 72 and rows starting 2 bytes into the buffer: the element-by-element path."""
    batch = synth.RaggedBatch([3, 1], [100, 4000])
    Hq, Hkv, D = 4, 2, 72
    Qb = synth.normal_bf16_bits(5, (batch.M, Hq * D + 1), 1.0)
    Kb = synth.normal_bf16_bits(6, (batch.M, Hkv * D + 1), 1.0)
    Qd, Kd = bf16_dev(Qb), bf16_dev(Kb)
    lib.spec_rope(Qd[:, 1:], Kd[:, 1:], dev(batch.cu_rows), dev(batch.ctx_len), D, 1e4)
    pos = np.concatenate([batch.ctx_len[b] + np.arange(batch.gammas[b] + 1) for b in range(batch.B)])
    qr = oops.rope(obf.decode(Qb[:, 1:]).reshape(batch.M, Hq, D), pos, 1e4).reshape(batch.M, -1)
    kr = oops.rope(obf.decode(Kb[:, 1:]).reshape(batch.M, Hkv, D), pos, 1e4).reshape(batch.M, -1)
    assert_close_rel(f64_of_bf16(Qd[:, 1:]), qr, "rope q (unaligned)", rel=1e-2)
    assert_close_rel(f64_of_bf16(Kd[:, 1:]), kr, "rope k (unaligned)", rel=1e-2)
    assert np.array_equal(bits_of(Qd[:, :1]), Qb[:, :1])


@pytest.mark.parametrize("std", [2.0, 60.0])
def test_silu_mul(lib, std):
    """std 60 puts many gate values past +-88, where e^-g overflows or underflows in fp32."""
    M, inter = 7, 12288
    GU = synth.normal_bf16_bits(3, (M, 2 * inter), std)
    A = lib.spec_silu_mul(bf16_dev(GU))
    g = obf.decode(GU)
    ref = oops.silu_mul(g[:, :inter], g[:, inter:])
    assert_close_rel(f64_of_bf16(A), ref, "silu_mul", rel=1e-2)


def _tiny_stack(L, seed, d=512, Hq=4, Hkv=2, I=1024, V=1024, std=0.05):
    from speculative_decoding_verify_05_gb300 import engine as E
    dims = E.Dims(d=d, Hq=Hq, Hkv=Hkv, D=128, I=I, V=V, layers=L)
    od = ostack.Dims(d=d, Hq=Hq, Hkv=Hkv, D=128, I=I, V=V, layers=L)
    ones = synth.f32_to_bf16_bits(np.ones(d, np.float32))
    olayers, glayers = [], []
    for li in range(L):
        s = seed + 10 * li
        w = [synth.normal_bf16_bits(s + 1, (dims.qkv, d), std), synth.normal_bf16_bits(s + 2, (d, Hq * 128), std),
             synth.normal_bf16_bits(s + 3, (2 * I, d), std), synth.normal_bf16_bits(s + 4, (d, I), std)]
        olayers.append(ostack.LayerWeights(*w, ones, ones))
        glayers.append(E.LayerW(*[bf16_dev(x) for x in w], bf16_dev(ones), bf16_dev(ones)))
    wl = synth.normal_bf16_bits(seed + 999, (V, d), std)
    osw = ostack.StackWeights(olayers, ones, wl)
    gsw = E.StackW(glayers, bf16_dev(ones), bf16_dev(wl))
    return dims, od, osw, gsw


@pytest.mark.parametrize("L,gammas,ctx,T", [(2, [3, 0, 5], [40, 9, 0], 1.0), (1, [4], [130], 0.0)])
@pytest.mark.parametrize("fused", [True, False])
def test_small_stack_end_to_end(lib, L, gammas, ctx, T, fused):
    from speculative_decoding_verify_05_gb300 import engine as E
    dims, od, osw, gsw = _tiny_stack(L, 50 + L)
    # one oracle reading for both plans (the split plan also stores gate|up as bf16 in between)
    batch = synth.RaggedBatch(gammas, ctx, cap=160)
    kc = [synth.normal_bf16_bits(200 + i, (batch.B, dims.Hkv, batch.cap, 128), 1.0) for i in range(L)]
    vc = [synth.normal_bf16_bits(300 + i, (batch.B, dims.Hkv, batch.cap, 128), 1.0) for i in range(L)]
    x0 = synth.normal_bf16_bits(7, (batch.M, dims.d), 1.0)
    eng = E.VerifyEngine(dims, gsw, [bf16_dev(k) for k in kc], [bf16_dev(v) for v in vc],
                         max_M=batch.M, max_rows=batch.max_rows, fused_swiglu=fused)
    P = eng.verify_pass(bf16_dev(x0), dev(batch.cu_rows), dev(batch.ctx_len), T)
    lib.spec_device_status()
    xr, lg, Kr, Vr = ostack.verify_pass(obf.decode(x0), osw, od, batch.cu_rows, batch.ctx_len,
                                        [obf.decode(k) for k in kc], [obf.decode(v) for v in vc])
    # hidden state after the stack: the chain bar of L layers, element by element
    assert_close_chain(f64_of_bf16(eng.x[:batch.M]), xr, L, f"final hidden (fused={fused})")
    p = P.cpu().numpy().astype(np.float64)
    if T > 0:
        pr = oops.target_probs(lg, T)
        assert np.abs(p - pr).max() < STACK_PROB_BOUND       # end-to-end through L layers
    else:
        top2 = np.sort(lg, axis=1)
        clear = (top2[:, -1] - top2[:, -2]) > 0.05
        assert np.array_equal(p.argmax(1)[clear], lg.argmax(1)[clear])
    # caches: every layer appended exactly its new block
    for li in range(L):
        got = obf.decode(eng.kc[li].contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
        for b in range(batch.B):
            c = batch.ctx_len[b]
            assert np.array_equal(got[b, :, :c], obf.decode(kc[li])[b, :, :c])
        assert_close_chain(got.reshape(-1, 128), Kr[li].reshape(-1, 128), L, "cache after pass")


def test_stack_verify_equals_sequential_decode_on_gpu(lib):
    """One verify pass over gamma+1 rows == gamma+1 single-row passes (same caches)."""
    from speculative_decoding_verify_05_gb300 import engine as E
    dims, od, osw, gsw = _tiny_stack(2, 70)
    gammas, ctx = [4, 2, 0], [33, 5, 80]
    batch = synth.RaggedBatch(gammas, ctx, cap=96)
    kc = [bf16_dev(synth.normal_bf16_bits(400 + i, (3, dims.Hkv, 96, 128), 1.0)) for i in range(2)]
    vc = [bf16_dev(synth.normal_bf16_bits(500 + i, (3, dims.Hkv, 96, 128), 1.0)) for i in range(2)]
    x0 = bf16_dev(synth.normal_bf16_bits(8, (batch.M, dims.d), 1.0))
    ev = E.VerifyEngine(dims, gsw, [k.clone() for k in kc], [v.clone() for v in vc], batch.M, batch.max_rows)
    Pv = ev.verify_pass(x0, dev(batch.cu_rows), dev(batch.ctx_len), 1.0).clone()
    ed = E.VerifyEngine(dims, gsw, [k.clone() for k in kc], [v.clone() for v in vc], batch.M, 1)
    Pd = torch.zeros_like(Pv)
    rows = batch.gammas + 1
    for j in range(int(rows.max())):
        seqs = np.nonzero(rows > j)[0]
        idx = batch.cu_rows[seqs] + j
        # single-row decode step for the sequences that have row j, against the full caches
        cu = np.arange(len(seqs) + 1, dtype=np.int32)
        kcs = [k[seqs] for k in ed.kc]
        vcs = [v[seqs] for v in ed.vc]
        sub = E.VerifyEngine(dims, gsw, kcs, vcs, len(seqs), 1)
        P1 = sub.verify_pass(x0[idx], dev(cu), dev((batch.ctx_len[seqs] + j).astype(np.int32)), 1.0)
        Pd[idx] = P1
        for li in range(2):
            ed.kc[li][seqs] = sub.kc[li]
            ed.vc[li][seqs] = sub.vc[li]
    lib.spec_device_status()
    assert (Pv - Pd).abs().max().item() < 1e-3
    for li in range(2):
        assert torch.equal(ev.kc[li][:, :, :40], ed.kc[li][:, :, :40]) or \
            (ev.kc[li].float() - ed.kc[li].float()).abs().max().item() < 0.1


def test_config1_round(lib):
    """B=1, gamma=4, d=512, V=4096, T=1, Philox seed 0: LM head + softmax + sampler vs the oracle."""
    d, V, gamma = 512, 4096, 4
    batch = synth.RaggedBatch([gamma], [0])
    w_bits = synth.normal_bf16_bits(1, (V, d), 0.02)
    x_bits = synth.normal_bf16_bits(2, (batch.M, d), 1.0)
    logits = oops.linear(obf.decode(x_bits), obf.decode(w_bits))
    p_ref = oops.target_probs(logits, 1.0)
    q, drafts = synth.draft_distribution(logits, batch, 1.0, 1.0, seed=3)
    U = synth.uniforms_f32(0, batch.M)
    P = lib.spec_lmhead_softmax(bf16_dev(x_bits), bf16_dev(w_bits), 1.0)
    n, t, near = lib.spec_reject_sample(P, dev(q), dev(drafts), dev(U), dev(batch.cu_rows))
    lib.spec_device_status()
    Ph = P.cpu().numpy()
    assert np.abs(Ph.astype(np.float64) - p_ref).max() < PROB_ATOL
    # decisions on the oracle's own p agree except where counted as near ties
    n_ref, t_ref, near_ref = osamp.reject_sample(p_ref, q, drafts, U, batch.cu_rows)
    if near.cpu().numpy()[0] == 0 and near_ref[0] == 0:
        assert int(n.cpu()[0]) == int(n_ref[0])
        assert np.array_equal(t.cpu().numpy(), t_ref)


def test_rope_table(lib):
    batch = synth.RaggedBatch([4, 0, 10, 2], [8190, 0, 333, 70000])
    D, theta = 128, 1e6
    cs = lib.spec_rope_table(dev(batch.cu_rows), dev(batch.ctx_len), batch.M, D, theta)
    lib.spec_device_status()
    pos = np.concatenate([batch.ctx_len[b] + np.arange(batch.gammas[b] + 1) for b in range(batch.B)])
    ang = pos[:, None].astype(np.float64) * theta ** (-2.0 * np.arange(D // 2) / D)[None, :]
    got = cs.cpu().numpy().astype(np.float64)
    assert np.abs(got[..., 0] - np.cos(ang)).max() < 2e-6
    assert np.abs(got[..., 1] - np.sin(ang)).max() < 2e-6


@pytest.mark.parametrize("M,Hq,Hkv,K", [(368, 32, 8, 4096), (5, 32, 8, 4096), (37, 8, 4, 512)])
def test_linear_rope_fused(lib, M, Hq, Hkv, K):
    """Q/K heads rotated by the projection (cluster epilogue at 368 rows, GEMM + rotate otherwise)."""
    rng = np.random.default_rng(M)
    B = max(1, M // 6)
    gam = np.full(B, M // B - 1)
    gam[-1] += M - int((gam + 1).sum())
    batch = synth.RaggedBatch(gam, rng.integers(0, 8000, size=B))
    D = 128
    N = (Hq + 2 * Hkv) * D
    X = synth.normal_bf16_bits(M + 1, (M, K), 1.0)
    W = synth.normal_bf16_bits(M + 2, (N, K), 0.02)
    cs = lib.spec_rope_table(dev(batch.cu_rows), dev(batch.ctx_len), M, D, 1e6)
    lib.reset_launch_count()
    Y = lib.spec_verify_linear_rope(bf16_dev(X), bf16_dev(W), cs, Hq + Hkv)
    fused = lib.launch_count() == 1          # rotated in the epilogue; else GEMM, then rotate
    lib.spec_device_status()
    pos = np.concatenate([batch.ctx_len[b] + np.arange(batch.gammas[b] + 1) for b in range(batch.B)])
    # one reading for both plans: q and k rotated from the fp64 sums.  A projection followed by a
    # rotation is a two-step chain (the unfused plan stores q and k in between), so it is held to the
    # chain bar of one layer
    y = oops.linear(obf.decode(X), obf.decode(W))
    ref = y.copy()
    qk = y[:, :(Hq + Hkv) * D].reshape(M, Hq + Hkv, D)
    ref[:, :(Hq + Hkv) * D] = oops.rope(qk, pos, 1e6).reshape(M, -1)
    assert_close_chain(f64_of_bf16(Y), ref, 1, f"linear + rope M={M} (fused={fused})")
    # the V heads are a plain projection: the single-linear bar
    assert_close_rel(f64_of_bf16(Y)[:, (Hq + Hkv) * D:], y[:, (Hq + Hkv) * D:], f"linear (v heads) M={M}")


def test_captured_round_replays_the_eager_round(lib):
    """VerifyEngine.capture_round: after new inputs are written into the captured buffers (same M
    and B, different ragged split, contexts, draft tokens and uniforms) a replay returns exactly
    what the eager verify_round returns on those inputs, cache writes included."""
    from speculative_decoding_verify_05_gb300 import engine as E
    L = 2
    dims, od, osw, gsw = _tiny_stack(L, 70)
    V = dims.V

    def inputs(seed, gammas, ctx):
        batch = synth.RaggedBatch(gammas, ctx, cap=200)
        rng = np.random.default_rng(seed)
        x0 = synth.normal_bf16_bits(seed, (batch.M, dims.d), 1.0)
        q = rng.dirichlet(np.full(V, 0.5), size=batch.M - batch.B).astype(np.float32)
        drafts = np.array([rng.choice(V, p=r.astype(np.float64) / r.astype(np.float64).sum()) for r in q], np.int32)
        U = synth.uniforms_f32(seed + 1, batch.M)
        return batch, x0, q, drafts, U

    bA, xA, qA, dA, uA = inputs(5, [3, 0, 5], [40, 9, 0])        # M = 11
    bB, xB, qB, dB, uB = inputs(6, [1, 6, 1], [100, 3, 57])      # M = 11, another split
    assert bA.M == bB.M and bA.B == bB.B
    kc = [synth.normal_bf16_bits(200 + i, (bA.B, dims.Hkv, 200, 128), 1.0) for i in range(L)]
    vc = [synth.normal_bf16_bits(300 + i, (bA.B, dims.Hkv, 200, 128), 1.0) for i in range(L)]
    eng = E.VerifyEngine(dims, gsw, [bf16_dev(k) for k in kc], [bf16_dev(v) for v in vc], max_M=bA.M, max_rows=7)
    bufs = [bf16_dev(xA), dev(bA.cu_rows), dev(bA.ctx_len), dev(qA), dev(dA), dev(uA)]
    out = (torch.empty(bA.B, dtype=torch.int32, device="cuda"), torch.empty(bA.M, dtype=torch.int32, device="cuda"),
           torch.empty(bA.B, dtype=torch.int32, device="cuda"))
    replay = eng.capture_round(*bufs, 0.8, out)
    lib.spec_device_status()
    # eager round on inputs B (fresh tensors), then the same inputs copied into the captured buffers
    n1, t1, z1 = eng.verify_round(bf16_dev(xB), dev(bB.cu_rows), dev(bB.ctx_len), dev(qB), dev(dB), dev(uB), 0.8)
    n1, t1, z1 = n1.cpu(), t1.cpu(), z1.cpu()
    cache1 = [bits_of(k) for k in eng.kc]
    for buf, host in zip(bufs, (bf16_dev(xB), dev(bB.cu_rows), dev(bB.ctx_len), dev(qB), dev(dB), dev(uB))):
        buf.copy_(host)
    replay()
    lib.spec_device_status()
    assert torch.equal(out[0].cpu(), n1) and torch.equal(out[1].cpu(), t1) and torch.equal(out[2].cpu(), z1)
    for k_after, k_eager in zip(eng.kc, cache1):
        assert np.array_equal(bits_of(k_after), k_eager)
