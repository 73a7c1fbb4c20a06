"""GPU parity of the RMSNorm folded into the verify linears.

A pre-norm product h W^T with h = RMSNorm(x) (unit norm weight, or the weight folded into W) is
(x W^T) / rms(x): the product that stores x leaves per-row, per-128-column sums of squares of what
it stored (out_ssq), and the product that reads x scales its rows by 1 / rms (in_ssq).  The oracle's
reading rounds h to bf16 before the product; the fused epilogue does not (the "norm folded" plan of
the chain tolerance), so single products are held to the chain bar of one layer.  Plans whose
epilogue cannot scale rows fall back to a normalised copy of X.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import bf16 as obf, ops as oops, sampler as osamp

from gpu_util import assert_close_chain, assert_close_rel, bf16_dev, bits_of, dev, f64_of_bf16

pytestmark = pytest.mark.gpu

EPS = 1e-6


def ssq_ref(Y):
    """Per row and 128-column tile sums of squares of the stored bf16 values (fp64)."""
    y = f64_of_bf16(Y)
    M, N = y.shape
    t = (N + 127) // 128
    pad = np.zeros((M, t * 128))
    pad[:, :N] = y
    return (pad.reshape(M, t, 128) ** 2).sum(axis=2)


@pytest.mark.parametrize("M,N", [(1, 4096), (368, 4096), (37, 1000), (5, 12288)])
def test_row_ssq(lib, M, N):
    X = bf16_dev(synth.normal_bf16_bits(M + N, (M, N), 3.0))
    out = lib.spec_row_ssq(X)
    lib.spec_device_status()
    ref = ssq_ref(X)
    assert np.allclose(out.cpu().numpy(), ref, rtol=2e-6, atol=0)


@pytest.mark.parametrize("M,N,K", [(368, 4096, 4096), (368, 4096, 12288), (5, 4096, 4096), (40, 640, 1024)])
def test_out_ssq_of_the_residual_stream(lib, M, N, K):
    """O / down projections (+ residual): Y within the linear bar, and the sums of squares of what
    they stored (fused in the split-K epilogue, or a separate pass for other plans)."""
    X = synth.normal_bf16_bits(M + 1, (M, K), 1.0)
    W = synth.normal_bf16_bits(M + 2, (N, K), 0.02)
    R = synth.normal_bf16_bits(M + 3, (M, N), 1.0)
    ssq = torch.full((M, (N + 127) // 128), -1.0, dtype=torch.float32, device="cuda")
    Y = bf16_dev(R).clone()
    lib.spec_verify_linear(bf16_dev(X), bf16_dev(W), Y=Y, residual=Y, norm=lib.row_norm(out_ssq=ssq))
    lib.spec_device_status()
    assert_close_rel(f64_of_bf16(Y), oops.linear(obf.decode(X), obf.decode(W), obf.decode(R)), "product")
    assert np.allclose(ssq.cpu().numpy(), ssq_ref(Y), rtol=2e-6, atol=0)


def _x_and_ssq(lib, seed, M, K):
    X = bf16_dev(synth.normal_bf16_bits(seed, (M, K), 2.0))
    return X, lib.spec_row_ssq(X)


@pytest.mark.parametrize("M,N,K", [(368, 6144, 4096), (5, 6144, 4096), (64, 1024, 512), (200, 20480, 136)])
def test_in_ssq_linear(lib, M, N, K):
    """h W^T with h = RMSNorm(x): scaled in the epilogue (split-K plans) or a normalised copy."""
    X, ssq = _x_and_ssq(lib, M + N, M, K)
    W = synth.normal_bf16_bits(M + K, (N, K), 0.02)
    Y = lib.spec_verify_linear(X, bf16_dev(W), norm=lib.row_norm(in_ssq=ssq, eps=EPS))
    lib.spec_device_status()
    h = obf.round_to_bf16(oops.rmsnorm(f64_of_bf16(X), np.ones(K), EPS))
    assert_close_chain(f64_of_bf16(Y), oops.linear(h, obf.decode(W)), 1, f"normed linear M={M}")


@pytest.mark.parametrize("M,I,K", [(368, 12288, 4096), (40, 12288, 4096), (5, 1024, 512)])
def test_in_ssq_swiglu(lib, M, I, K):
    X, ssq = _x_and_ssq(lib, M + I, M, K)
    Wg = synth.normal_bf16_bits(M + 1, (I, K), 0.05)
    Wu = synth.normal_bf16_bits(M + 2, (I, K), 0.05)
    Wgu = lib.interleave_gate_up(bf16_dev(Wg), bf16_dev(Wu))
    A = lib.spec_verify_linear_swiglu(X, Wgu, norm=lib.row_norm(in_ssq=ssq, eps=EPS))
    lib.spec_device_status()
    h = obf.round_to_bf16(oops.rmsnorm(f64_of_bf16(X), np.ones(K), EPS))
    ref = oops.silu_mul(oops.linear(h, obf.decode(Wg)), oops.linear(h, obf.decode(Wu)))
    assert_close_chain(f64_of_bf16(A), ref, 1, f"normed swiglu M={M}")


@pytest.mark.parametrize("M", [368, 100, 8])
def test_in_ssq_linear_rope(lib, M):
    Hq, Hkv, D, K = 32, 8, 128, 4096
    rng = np.random.default_rng(M)
    B = max(1, M // 6)
    gam = np.full(B, M // B - 1)
    gam[-1] += M - int((gam + 1).sum())
    batch = synth.RaggedBatch(gam, rng.integers(0, 8000, size=B))
    N = (Hq + 2 * Hkv) * D
    X, ssq = _x_and_ssq(lib, M + 7, M, K)
    W = synth.normal_bf16_bits(M + 8, (N, K), 0.02)
    cs = lib.spec_rope_table(dev(batch.cu_rows), dev(batch.ctx_len), M, D, 1e6)
    Y = lib.spec_verify_linear_rope(X, bf16_dev(W), cs, Hq + Hkv, norm=lib.row_norm(in_ssq=ssq, eps=EPS))
    lib.spec_device_status()
    pos = np.concatenate([batch.ctx_len[b] + np.arange(batch.gammas[b] + 1) for b in range(batch.B)])
    h = obf.round_to_bf16(oops.rmsnorm(f64_of_bf16(X), np.ones(K), EPS))
    y = oops.linear(h, obf.decode(W))
    ref = y.copy()
    ref[:, :(Hq + Hkv) * D] = oops.rope(y[:, :(Hq + Hkv) * D].reshape(M, Hq + Hkv, D), pos, 1e6).reshape(M, -1)
    assert_close_chain(f64_of_bf16(Y), ref, 1, f"normed linear + rope M={M}")


@pytest.mark.parametrize("M,V,T", [(40, 8192, 0.7), (40, 8192, 0.0), (368, 20480, 0.7), (368, 20480, 0.0)])
def test_in_ssq_lmhead_sampler(lib, M, V, T):
    """The LM head -> sampler on the residual stream x with the final norm folded: the same
    decisions as the oracle wherever they are not near ties of either side.  This checks the op
    against its own definition (the product's rows scaled by 1 / rms: the normed rows are not
    rounded), on rows peaked by a W of std 0.25 (logits of std ~5.7), where a bf16 rounding of the
    normed rows alone would move p by a few percent; the layer-level reading, which rounds them, is
    held to the chain bar by the stack tests.  At 368 rows and 160 vocabulary tiles the LM head runs
    on CTA pairs."""
    K = 512
    batch = synth.RaggedBatch([4] * 8, [100] * 8) if M == 40 else synth.RaggedBatch([4] * 73 + [2], [100] * 74)
    assert batch.M == M
    X, ssq = _x_and_ssq(lib, 5, M, K)
    W = synth.normal_bf16_bits(6, (V, K), 0.25)
    h = oops.rmsnorm(f64_of_bf16(X), np.ones(K), EPS)
    logits = oops.linear(h, obf.decode(W))
    q, drafts = synth.draft_distribution(logits, batch, 0.5, T if T > 0 else 1.0, seed=9)
    U = synth.uniforms_f32(11, M)
    n, t, near = lib.spec_lmhead_reject_sample(X, bf16_dev(W), T, dev(q), dev(drafts), dev(U), dev(batch.cu_rows),
                                               norm=lib.row_norm(in_ssq=ssq, eps=EPS))
    lib.spec_device_status()
    p_ref = oops.target_probs(logits, T)
    n_ref, t_ref, near_ref = osamp.reject_sample(p_ref, q, drafts, U, batch.cu_rows, 1e-4)
    n, t, near = n.cpu().numpy(), t.cpu().numpy(), near.cpu().numpy()
    clear = (near == 0) & (near_ref == 0)
    if T == 0:
        top2 = np.sort(logits, axis=1)
        gap_ok = np.array([np.all(top2[batch.cu_rows[b]:batch.cu_rows[b + 1], -1] -
                                  top2[batch.cu_rows[b]:batch.cu_rows[b + 1], -2] > 0.05) for b in range(batch.B)])
        clear &= gap_ok
    assert clear.sum() >= batch.B // 2
    for b in np.nonzero(clear)[0]:
        assert n[b] == n_ref[b], b
        r0 = batch.cu_rows[b]
        assert np.array_equal(t[r0:r0 + n[b] + 1], t_ref[r0:r0 + n[b] + 1]), b


@pytest.mark.parametrize("fold", [True, False])
def test_stack_with_and_without_folded_norms(lib, fold):
    """The same 2-layer stack through the engine with the norms folded (the products carry them) and
    with the RMSNorm kernel: both within the chain bar of the oracle."""
    from speculative_decoding_verify_05_gb300 import engine as E
    from oracle import stack as ostack
    from test_gpu_glue_stack import _tiny_stack
    dims, od, osw, gsw = _tiny_stack(2, 52)
    batch = synth.RaggedBatch([3, 0, 5], [40, 9, 0], cap=160)
    kc = [synth.normal_bf16_bits(200 + i, (batch.B, dims.Hkv, batch.cap, 128), 1.0) for i in range(2)]
    vc = [synth.normal_bf16_bits(300 + i, (batch.B, dims.Hkv, batch.cap, 128), 1.0) for i in range(2)]
    x0 = synth.normal_bf16_bits(7, (batch.M, dims.d), 1.0)
    eng = E.VerifyEngine(dims, gsw, [bf16_dev(k) for k in kc], [bf16_dev(v) for v in vc], max_M=batch.M,
                         max_rows=batch.max_rows, fold_norms=fold)
    lib.reset_launch_count()
    eng.verify_pass(bf16_dev(x0), dev(batch.cu_rows), dev(batch.ctx_len), 1.0)
    launches = lib.launch_count()
    lib.spec_device_status()
    xr, _, _, _ = ostack.verify_pass(obf.decode(x0), osw, od, batch.cu_rows, batch.ctx_len,
                                     [obf.decode(k) for k in kc], [obf.decode(v) for v in vc])
    assert_close_chain(f64_of_bf16(eng.x[:batch.M]), xr, 2, f"final hidden (folded norms={fold})")
    assert launches > 0
