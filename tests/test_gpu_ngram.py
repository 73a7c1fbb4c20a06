"""GPU parity of spec_ngram_propose against the oracle: integer work, so bit-exact."""
import numpy as np
import pytest
import torch

import synth
from oracle import ngram as NG

from gpu_util import dev

pytestmark = pytest.mark.gpu


def pack(hs):
    cu = np.zeros(len(hs) + 1, np.int32)
    cu[1:] = np.cumsum([len(h) for h in hs])
    tokens = np.concatenate([np.asarray(h, np.int32) for h in hs]) if cu[-1] else np.zeros(1, np.int32)
    return tokens, cu


def check(lib, tokens, cu, k, n_min, n_max):
    drafts, n = lib.spec_ngram_propose(dev(tokens), dev(cu), k, n_min, n_max)
    lib.spec_device_status()
    d_ref, n_ref = NG.propose_batch(tokens, cu, k, n_min, n_max)
    assert np.array_equal(n.cpu().numpy(), n_ref)
    assert np.array_equal(drafts.cpu().numpy(), d_ref)
    return n_ref


@pytest.mark.parametrize("alphabet,k,n_min,n_max", [(2, 4, 1, 3), (3, 5, 2, 4), (4, 1, 1, 1), (5, 8, 3, 8)])
def test_small_alphabet_histories(lib, alphabet, k, n_min, n_max):
    rng = np.random.default_rng(alphabet * 10 + k)
    hs = [rng.integers(0, alphabet, size=int(rng.integers(0, 700))) for _ in range(200)]
    tokens, cu = pack(hs)
    n = check(lib, tokens, cu, k, n_min, n_max)
    assert (n > 0).mean() > 0.5


@pytest.mark.parametrize("copy_frac", [0.8, 0.0])
def test_copy_heavy_histories_at_full_context(lib, copy_frac):
    """B = 64 histories of 128..8192 tokens over a 151936-token vocabulary (the verify
    workload's context range), copy-heavy or uniform."""
    tokens, cu = synth.ngram_histories(11, B=64, len_lo=128, len_hi=8192, vocab=151936, copy_frac=copy_frac)
    n = check(lib, tokens, cu, 4, 3, 8)
    if copy_frac > 0:
        assert (n > 0).mean() > 0.5


def test_edge_cases(lib):
    hs = [[], [7], [7, 7], [1, 2, 1], [9] * 300, list(range(100)) + list(range(100))]
    tokens, cu = pack(hs)
    check(lib, tokens, cu, 3, 1, 2)
    check(lib, tokens, cu, 1000, 1, 64)          # k past every history, the widest window
    check(lib, tokens, cu, 5, 64, 64)
    rng = np.random.default_rng(5)
    many = [rng.integers(0, 3, size=int(rng.integers(1, 40))) for _ in range(1000)]
    tokens, cu = pack(many)
    check(lib, tokens, cu, 4, 2, 5)


def test_negative_length_is_flagged(lib):
    tokens, cu = pack([[1, 2, 1, 2], [3, 3, 3]])
    cu_bad = cu.copy()
    cu_bad[1] = 6                                 # sequence 1 now has length 7 - 6 = 1, sequence 0 has 6
    cu_bad[2] = 5                                 # and sequence 1 length -1
    drafts, n = lib.spec_ngram_propose(dev(tokens), dev(cu_bad[:3]), 2, 1, 2)
    with pytest.raises(lib.SpecError):
        lib.spec_device_status()
    lib.spec_device_status()
    assert n.cpu().numpy()[1] == 0 and np.all(drafts.cpu().numpy()[1] == -1)
