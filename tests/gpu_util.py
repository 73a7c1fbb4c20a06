"""Helpers shared by the GPU parity tests: move seeded numpy inputs to the
device and compare device results with the oracle within the stated bars."""
import numpy as np
import torch

from oracle import bf16 as obf

DEV = torch.device("cuda")

# spec bars: linear / attention outputs 2e-2 relative (bf16 out, fp32
# accumulate), probabilities 1e-5 absolute.  An element passes when
# |gpu - ref| <= REL * |ref| + FLOOR * rms(ref): the floor covers outputs
# that are tiny next to their row (bf16 rounding is relative to the value;
# fp32 accumulation error scales with the row's magnitude).
REL = 2e-2
FLOOR = 1e-3
PROB_ATOL = 1e-5


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64_of_bf16(t: torch.Tensor) -> np.ndarray:
    return obf.decode(bits_of(t))


def assert_close_rel(got: np.ndarray, ref: np.ndarray, what: str, rel=REL, floor=FLOOR):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    scale = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = rel * np.abs(ref) + floor * scale
    bad = err > bound
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} / {bad.size} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} (rms {scale:.3g})")


# Attention outputs are softmax-weighted sums of values.  The probabilities
# enter the tensor-core PV product rounded to bf16 (relative error <= 2^-9
# each), so an output element can move by up to 2^-9 * sum_i w_i |v_i|, the
# magnitude of the terms it sums, however small the (cancelling) result is.
# Bar: |gpu - ref| <= 2e-2 |ref| + 2 * 2^-9 * sum_i w_i |v_i|.
ATTN_ABS = 2.0 * 2.0 ** -9


def assert_close_attn(got, ref, mag, what: str, rel=REL, abs_frac=ATTN_ABS):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    mag = np.asarray(mag, np.float64)
    assert got.shape == ref.shape == mag.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = rel * np.abs(ref) + abs_frac * mag
    bad = err > bound
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} / {bad.size} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} magnitude {mag[i]!r}")


# Chains of L layers (hidden state, caches): every bf16 rounding point moves a tensor by up to 2^-9
# of each element; once that tensor has gone through a linear map and the residual add, the
# differences are absolute errors of the order of 2^-9 rms per element, and independent rounding
# differences add up like sqrt(L).  The floor CHAIN_FLOOR sqrt(L) rms(ref) is derived and pinned on
# the CPU (tests/test_oracle_chain_tolerance.py): correct plans of the arithmetic (fp32 sums,
# bf16 softmax weights in P.V, other rounding points) stay below it with margin >= 1.5, and planted
# mistakes exceed it at least 5-fold.
CHAIN_FLOOR = 0.03


def chain_floor(L: int) -> float:
    return CHAIN_FLOOR * float(np.sqrt(max(L, 1)))


def assert_close_chain(got, ref, L: int, what: str):
    """Element-wise |gpu - ref| <= 2e-2 |ref| + CHAIN_FLOOR sqrt(L) rms(ref)."""
    assert_close_rel(got, ref, what, rel=REL, floor=chain_floor(L))


# The draft engine's q rows after two layers of a peaked draft stack (tied table of std 0.2:
# p up to ~0.9): the oracle's own perturbation to GPU-like arithmetic moves q by up to 0.025
# (tests/test_oracle_chain_tolerance.py), so the GPU is held to 1.6 times that.
DRAFT_PROB_BOUND = 4e-2


# Probabilities at the end of a stack of up to 2 layers (the tiny GPU stacks, T > 0): correct plans
# move them by up to 1.1e-3 on the oracle itself, about half of this bound (pinned in
# test_oracle_chain_tolerance.py); the 1e-5 bar applies to the LM-head softmax on identical logits,
# which the op tests check.
STACK_PROB_BOUND = 2e-3
