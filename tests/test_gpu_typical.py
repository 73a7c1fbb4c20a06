"""GPU parity of spec_typical_sample (typical acceptance) against the oracle on identical inputs.

The threshold formula is the oracle's reading of a page whose formula was lost (parity
unpinned beyond its closed forms); what is checked here is that the CUDA path computes that
same reading: equal acceptance counts and tokens for every sequence neither side flags as a
near tie, and greedy behaviour on one-hot rows.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import typical as otyp

from gpu_util import dev

pytestmark = pytest.mark.gpu


def typical_inputs(seed, gammas, V, conc):
    """Target rows of varied entropy (Dirichlet, concentration per sequence) and drafts drawn
    from the target rows themselves, so that some pass and some fail the threshold."""
    rng = np.random.default_rng(seed)
    batch = synth.RaggedBatch(gammas, np.zeros(len(gammas), np.int32))
    P = np.empty((batch.M, V), np.float32)
    for b in range(batch.B):
        c = conc[b % len(conc)]
        P[batch.cu_rows[b]:batch.cu_rows[b + 1]] = rng.dirichlet(np.full(V, c), size=batch.gammas[b] + 1)
    drafts = []
    for b in range(batch.B):
        for i in range(batch.gammas[b]):
            row = P[batch.cu_rows[b] + i].astype(np.float64)
            drafts.append(rng.choice(V, p=row / row.sum()))
    drafts = np.asarray(drafts, np.int32) if drafts else np.zeros(0, np.int32)
    U = synth.uniforms_f32(seed + 1, batch.M)
    return batch, P, drafts, U


def gpu_typical(lib, batch, P, drafts, U, eps, delta):
    Dd = dev(drafts) if drafts.size else torch.zeros(1, dtype=torch.int32, device="cuda")
    n, t, near = lib.spec_typical_sample(dev(P), Dd, dev(U), dev(batch.cu_rows), eps, delta)
    lib.spec_device_status()
    return n.cpu().numpy(), t.cpu().numpy(), near.cpu().numpy()


@pytest.mark.parametrize("gammas,V,conc,eps,delta", [
    ([4, 0, 7, 2] * 6, 64, [0.05, 0.3, 2.0], 0.05, 0.3),
    (list(range(0, 12)) * 2, 4096, [0.01, 0.1], 0.01, 0.5),
    ([3] * 8, 151936, [0.001, 0.01], 0.001, 0.4),
    ([40, 33], 256, [0.02], 0.02, 0.3),
])
def test_typical_matches_oracle(lib, gammas, V, conc, eps, delta):
    batch, P, drafts, U = typical_inputs(len(gammas) + V, gammas, V, conc)
    n, t, near = gpu_typical(lib, batch, P, drafts, U, eps, delta)
    n_ref, t_ref, near_ref = otyp.typical_accept_sample(P, drafts, U, batch.cu_rows, eps, delta)
    clean = (near == 0) & (near_ref == 0)
    assert clean.mean() >= 0.6
    assert np.array_equal(n[clean], n_ref[clean])
    for b in np.nonzero(clean)[0]:
        r0, r1 = batch.cu_rows[b], batch.cu_rows[b + 1]
        assert np.array_equal(t[r0:r1], t_ref[r0:r1]), b
    # both branches occur: some drafts kept, some sequences stopped early
    assert n.sum() > 0 and np.any(n < batch.gammas)


def test_typical_one_hot_rows_equal_exact_greedy(lib):
    rng = np.random.default_rng(8)
    B, gamma, V = 300, 5, 32
    tgt = rng.integers(0, V, size=(B, gamma + 1))
    P = np.zeros((B * (gamma + 1), V), np.float32)
    P[np.arange(B * (gamma + 1)), tgt.reshape(-1)] = 1.0
    agree = rng.integers(0, gamma + 1, size=B)
    drafts = rng.integers(0, V, size=(B, gamma))
    for b in range(B):
        drafts[b, :agree[b]] = tgt[b, :agree[b]]
        if agree[b] < gamma and drafts[b, agree[b]] == tgt[b, agree[b]]:
            drafts[b, agree[b]] = (tgt[b, agree[b]] + 1) % V
    drafts = drafts.reshape(-1).astype(np.int32)
    batch = synth.RaggedBatch([gamma] * B, np.zeros(B, np.int32))
    U = synth.uniforms_f32(6, batch.M)
    n, t, _ = gpu_typical(lib, batch, P, drafts, U, 0.09, 0.3)
    Q = rng.dirichlet(np.ones(V), size=B * gamma).astype(np.float32)
    n2, t2, _ = lib.spec_reject_sample(dev(P), dev(Q), dev(drafts), dev(U), dev(batch.cu_rows))
    assert np.array_equal(n, agree) and np.array_equal(n, n2.cpu().numpy())
    assert np.array_equal(t, t2.cpu().numpy())


def test_typical_bad_token_flag_and_empty_batch(lib):
    batch, P, drafts, U = typical_inputs(2, [2], 16, [0.5])
    drafts[0] = -3
    lib.spec_typical_sample(dev(P), dev(drafts), dev(U), dev(batch.cu_rows), 0.05, 0.3)
    with pytest.raises(lib.SpecError):
        lib.spec_device_status()
    lib.spec_device_status()
    empty = torch.zeros(1, dtype=torch.int32, device="cuda")
    n, _, near = lib.spec_typical_sample(dev(P), dev(drafts), dev(U), empty, 0.05, 0.3)
    assert n.numel() == 0 and near.numel() == 0
