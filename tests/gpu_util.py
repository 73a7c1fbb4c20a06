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


def assert_rows_close_l2(got, ref, what: str, rel=REL):
    """Row-wise ||gpu - ref|| / ||ref|| <= rel: the bar for chains of several bf16 ops."""
    got = np.asarray(got, np.float64).reshape(len(got), -1)
    ref = np.asarray(ref, np.float64).reshape(len(ref), -1)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    r = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert r.max() <= rel, f"{what}: worst row relative L2 error {r.max():.3g} (row {int(r.argmax())})"
