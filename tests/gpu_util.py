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
