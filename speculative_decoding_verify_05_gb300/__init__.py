"""GB300-native speculative-decoding verify round.

The compute lives in ``libspecverify.so`` (hand-written CUDA for sm_103a,
C ABI in ``include/spec_verify.h``); :mod:`.binding` marshals torch tensors
into it and :mod:`.engine` drives a Qwen3-8B-shaped verify pass through it.
"""
import os

PACKAGE_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PACKAGE_DIR, "libspecverify.so")


def build(verbose: bool = False) -> str:
    """Compile the CUDA library in-tree (needs nvcc)."""
    from .build import build as _build
    return _build(verbose=verbose)
