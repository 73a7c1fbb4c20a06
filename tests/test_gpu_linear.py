"""GPU parity of spec_verify_linear (CUDA-core and tcgen05 paths) against the oracle."""
import numpy as np
import pytest

import synth
from oracle import bf16 as obf, ops as oops

from gpu_util import assert_close_rel, bf16_dev, bits_of, f64_of_bf16

pytestmark = pytest.mark.gpu

SHAPES = [
    # (M, N, K): ragged tails in every dimension, several M tiles, split-K on and off
    (1, 256, 512), (2, 384, 1000), (3, 200, 264), (4, 1024, 4096),
    (5, 512, 4096), (7, 136, 72), (16, 640, 264), (17, 256, 520), (40, 1024, 512),
    (100, 256, 768), (256, 384, 128), (300, 384, 512), (368, 6144, 4096), (513, 128, 256),
    (1030, 640, 320),
    (200, 20480, 136),   # 160 tiles: 152 whole, the last 8 split over mostly empty stream-K ranges
]


def run_case(lib, M, N, K, residual, seed, gemv_max_m=4, grid=0, std=0.05):
    X = synth.normal_bf16_bits(seed, (M, K), 1.0)
    W = synth.normal_bf16_bits(seed + 1, (N, K), std)
    R = synth.normal_bf16_bits(seed + 2, (M, N), 1.0) if residual else None
    lib.spec_set_option("gemv_max_m", gemv_max_m)
    lib.spec_set_option("persistent_grid", grid)
    try:
        Y = lib.spec_verify_linear(bf16_dev(X), bf16_dev(W), residual=bf16_dev(R) if residual else None)
        lib.spec_device_status()
    finally:
        lib.spec_set_option("gemv_max_m", 0)
        lib.spec_set_option("persistent_grid", 0)
    ref = oops.linear(obf.decode(X), obf.decode(W), obf.decode(R) if residual else None)
    assert_close_rel(f64_of_bf16(Y), ref, f"linear M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("residual", [False, True])
def test_linear_default_path(lib, M, N, K, residual):
    run_case(lib, M, N, K, residual, seed=M * 7 + N + K)


@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_linear_tensor_core_path_at_tiny_m(lib, M):
    run_case(lib, M, 768, 1024, True, seed=40 + M, gemv_max_m=0)


@pytest.mark.parametrize("grid", [1, 2, 3, 7, 50, 333])
def test_linear_forced_grid(lib, grid):
    """Persistent grids that split tiles between CTAs in many different ways."""
    run_case(lib, 24, 512, 1536, True, seed=90 + grid, gemv_max_m=0, grid=grid)
    run_case(lib, 300, 640, 1000, True, seed=91 + grid, gemv_max_m=0, grid=grid)


def test_linear_residual_aliases_output(lib):
    import torch
    M, N, K = 6, 256, 512
    X = synth.normal_bf16_bits(5, (M, K), 1.0)
    W = synth.normal_bf16_bits(6, (N, K), 0.05)
    R = synth.normal_bf16_bits(7, (M, N), 1.0)
    Yd = bf16_dev(R).clone()
    lib.spec_verify_linear(bf16_dev(X), bf16_dev(W), Y=Yd, residual=Yd)
    lib.spec_device_status()
    ref = oops.linear(obf.decode(X), obf.decode(W), obf.decode(R))
    assert_close_rel(f64_of_bf16(Yd), ref, "aliased residual")


def test_linear_repeat_reuses_workspace(lib):
    """Counters return to zero: the same workspace serves many split-K calls."""
    ws = lib.Workspace()
    X = synth.normal_bf16_bits(8, (5, 4096), 1.0)
    W = synth.normal_bf16_bits(9, (4096, 4096), 0.02)
    ref = oops.linear(obf.decode(X), obf.decode(W))
    Xd, Wd = bf16_dev(X), bf16_dev(W)
    lib.spec_set_option("gemv_max_m", 0)
    try:
        for _ in range(3):
            Y = lib.spec_verify_linear(Xd, Wd, ws=ws)
            assert_close_rel(f64_of_bf16(Y), ref, "repeat")
    finally:
        lib.spec_set_option("gemv_max_m", 0)
    lib.spec_device_status()


def test_linear_strided_output_slice(lib):
    """Y written into a column slice of a wider buffer (leading dimension > N)."""
    import torch
    M, N, K = 9, 256, 384
    X = synth.normal_bf16_bits(11, (M, K), 1.0)
    W = synth.normal_bf16_bits(12, (N, K), 0.05)
    big = torch.zeros((M, 3 * N), dtype=torch.bfloat16, device="cuda")
    lib.spec_verify_linear(bf16_dev(X), bf16_dev(W), Y=big[:, N:2 * N])
    lib.spec_device_status()
    ref = oops.linear(obf.decode(X), obf.decode(W))
    assert_close_rel(f64_of_bf16(big[:, N:2 * N]), ref, "strided Y")
    assert torch.count_nonzero(big[:, :N]) == 0 and torch.count_nonzero(big[:, 2 * N:]) == 0


def test_linear_launch_accounting(lib):
    """One kernel when every tile is finished by one CTA, two when split tiles need the reduce."""
    X = bf16_dev(synth.normal_bf16_bits(3, (368, 4096), 1.0))
    W = bf16_dev(synth.normal_bf16_bits(4, (6144, 4096), 0.02))
    lib.reset_launch_count()
    lib.spec_verify_linear(X, W)
    assert lib.launch_count() == (2 if lib.spec_linear_workspace_bytes(368, 6144, 4096) > 0 else 1)
    lib.spec_set_option("persistent_grid", 1)      # one CTA: every tile whole, no workspace
    try:
        assert lib.spec_linear_workspace_bytes(368, 6144, 4096) == 0
        lib.reset_launch_count()
        lib.spec_verify_linear(X, W)
        assert lib.launch_count() == 1
    finally:
        lib.spec_set_option("persistent_grid", 0)
    lib.spec_device_status()


@pytest.mark.parametrize("M,N,K", [(368, 4096, 4096), (300, 4096, 1000), (200, 4096, 520), (17, 6144, 4096),
                                   (513, 4096, 4096), (64, 2048, 12288), (5, 512, 4096), (8, 256, 256),
                                   (33, 1024, 4096), (48, 384, 264)])
def test_linear_cluster_split_k(lib, M, N, K):
    """Few weight tiles: the cluster split-K kernel (pieces summed over distributed shared
    memory) and the stream-K path both match the oracle."""
    for cluster in (1, 0):
        lib.spec_set_option("linear_cluster", cluster)
        try:
            run_case(lib, M, N, K, True, seed=M + N + K + cluster, gemv_max_m=0)
        finally:
            lib.spec_set_option("linear_cluster", 1)


@pytest.mark.parametrize("M,N,K", [(368, 4096, 4096), (368, 4096, 12288), (300, 4096, 1000), (260, 2048, 520)])
def test_linear_cluster_half_row_tiles(lib, M, N, K):
    """Few weight tiles at 257..384 rows: the cluster plan on two half-row tiles (the planner's
    choice where its exchange model says it pays) and on one two-MMA tile both match the oracle,
    each in one launch without workspace."""
    for split in (1, 0):
        lib.spec_set_option("linear_split_rows", split)
        try:
            assert lib.spec_linear_workspace_bytes(M, N, K) == 0
            lib.reset_launch_count()
            run_case(lib, M, N, K, True, seed=M + N + K + split, gemv_max_m=0)
            assert lib.launch_count() == 1
        finally:
            lib.spec_set_option("linear_split_rows", 1)


# --------------------------------------------------------------------------- fused gate/up + SwiGLU
def run_swiglu(lib, M, I, K, seed, gemv_max_m=4, grid=0, std=0.05):
    """A = silu(X Wg^T) * (X Wu^T) through spec_verify_linear_swiglu vs the oracle in fp64
    (gate and up unrounded, as the fused kernel takes them from its fp32 accumulators)."""
    X = synth.normal_bf16_bits(seed, (M, K), 1.0)
    Wg = synth.normal_bf16_bits(seed + 1, (I, K), std)
    Wu = synth.normal_bf16_bits(seed + 2, (I, K), std)
    Wgu = lib.interleave_gate_up(bf16_dev(Wg), bf16_dev(Wu))
    lib.spec_set_option("gemv_max_m", gemv_max_m)
    lib.spec_set_option("persistent_grid", grid)
    try:
        A = lib.spec_verify_linear_swiglu(bf16_dev(X), Wgu)
        lib.spec_device_status()
    finally:
        lib.spec_set_option("gemv_max_m", 0)
        lib.spec_set_option("persistent_grid", 0)
    x = obf.decode(X)
    ref = oops.silu_mul(oops.linear(x, obf.decode(Wg)), oops.linear(x, obf.decode(Wu)))
    assert_close_rel(f64_of_bf16(A), ref, f"swiglu linear M={M} I={I} K={K}")


SWIGLU_SHAPES = [
    # CUDA-core path (M <= 4), the smallest interleave block, ragged K, one and two
    # sub-tiles, several M tiles, and the Qwen3-8B MLP (I = 12288, d = 4096)
    (1, 1024, 512), (3, 64, 264), (4, 12288, 4096), (5, 12288, 4096), (37, 1024, 520),
    (300, 640, 1000), (368, 12288, 4096), (513, 128, 256), (1030, 320, 320),
]


@pytest.mark.parametrize("M,I,K", SWIGLU_SHAPES)
def test_linear_swiglu(lib, M, I, K):
    run_swiglu(lib, M, I, K, seed=3 * M + I + K)


@pytest.mark.parametrize("M", [1, 2, 4])
def test_linear_swiglu_tensor_core_at_tiny_m(lib, M):
    run_swiglu(lib, M, 768, 1024, seed=60 + M, gemv_max_m=0)


@pytest.mark.parametrize("grid", [1, 3, 7, 50, 333])
def test_linear_swiglu_forced_grid(lib, grid):
    """Split tiles summed by the reduce kernel, which applies the activation itself."""
    run_swiglu(lib, 24, 512, 1536, seed=120 + grid, gemv_max_m=0, grid=grid)
    run_swiglu(lib, 300, 640, 1000, seed=121 + grid, gemv_max_m=0, grid=grid)


def test_linear_swiglu_matches_unfused_pair(lib):
    """Same rows as spec_verify_linear on the split layout followed by spec_silu_mul, up to
    the bf16 rounding of gate and up that only the unfused pair does."""
    M, I, K = 9, 1024, 512
    X = bf16_dev(synth.normal_bf16_bits(11, (M, K), 1.0))
    Wg = bf16_dev(synth.normal_bf16_bits(12, (I, K), 0.05))
    Wu = bf16_dev(synth.normal_bf16_bits(13, (I, K), 0.05))
    import torch
    GU = lib.spec_verify_linear(X, torch.cat((Wg, Wu), 0))
    A0 = lib.spec_silu_mul(GU)
    A1 = lib.spec_verify_linear_swiglu(X, lib.interleave_gate_up(Wg, Wu))
    lib.spec_device_status()
    assert_close_rel(f64_of_bf16(A1), f64_of_bf16(A0), "fused vs unfused", rel=2e-2)


def test_linear_swiglu_strided_output_and_launches(lib):
    """Output into a column slice of a wider buffer; one launch (two when tiles are split)."""
    import torch
    M, I, K = 40, 1024, 512
    X = synth.normal_bf16_bits(21, (M, K), 1.0)
    Wg = synth.normal_bf16_bits(22, (I, K), 0.05)
    Wu = synth.normal_bf16_bits(23, (I, K), 0.05)
    buf = torch.zeros((M, I + 64), dtype=torch.bfloat16, device="cuda")
    lib.reset_launch_count()
    lib.spec_verify_linear_swiglu(bf16_dev(X), lib.interleave_gate_up(bf16_dev(Wg), bf16_dev(Wu)),
                                  A=buf[:, 64:])
    lib.spec_device_status()
    assert lib.launch_count() == (2 if lib.spec_swiglu_linear_workspace_bytes(M, I, K) > 0 else 1)
    x = obf.decode(X)
    ref = oops.silu_mul(oops.linear(x, obf.decode(Wg)), oops.linear(x, obf.decode(Wu)))
    assert_close_rel(f64_of_bf16(buf[:, 64:]), ref, "swiglu strided")
    assert torch.count_nonzero(buf[:, :64]).item() == 0


@pytest.mark.parametrize("M,I,K", [(1, 1024, 512), (3, 1024, 512), (4, 12288, 4096), (9, 1024, 512)])
def test_linear_swiglu_leaves_counter_region_zero(lib, M, I, K):
    """The first 64 KiB of a workspace are counters that every kernel finds zero and leaves
    zero; the fused call's scratch lives elsewhere."""
    import torch
    ws = lib.Workspace()
    ws.ensure(max(lib.spec_swiglu_linear_workspace_bytes(M, I, K), 1 << 17))
    ws.buf.zero_()
    X = bf16_dev(synth.normal_bf16_bits(31, (M, K), 1.0))
    Wgu = bf16_dev(synth.normal_bf16_bits(32, (2 * I, K), 0.05))
    lib.spec_verify_linear_swiglu(X, Wgu, ws=ws)
    lib.spec_device_status()
    assert torch.count_nonzero(ws.buf[:1 << 16]).item() == 0


@pytest.mark.parametrize("M,N,K,grid", [
    (368, 6144, 1024, 0),    # 48 weight tiles on the persistent kernel, stream-K remainder
    (300, 1152, 1000, 0),    # 9 weight tiles
    (513, 640, 256, 0),      # two token tiles, 5 weight tiles
    (100, 1000, 520, 7),     # ragged N, forced grid of 7 CTAs
    (368, 2048, 512, 3),     # 3 CTAs: every tile split between CTAs
    (64, 384, 264, 0),
])
def test_linear_persistent_stream_k(lib, M, N, K, grid):
    """Persistent GEMM with the cluster split-K plan switched off: whole tiles, stream-K pieces
    and the reduce kernel on every shape."""
    lib.spec_set_option("linear_cluster", 0)
    try:
        run_case(lib, M, N, K, True, seed=M + N + K, gemv_max_m=0, grid=grid)
    finally:
        lib.spec_set_option("linear_cluster", 1)


@pytest.mark.parametrize("grid", [0, 5])
def test_linear_swiglu_persistent(lib, grid):
    run_swiglu(lib, 368, 1216, 1024, seed=500 + grid, gemv_max_m=0, grid=grid)


@pytest.mark.parametrize("M,N,K", [(368, 24576, 4096), (200, 20480, 136), (300, 19584, 520)])
def test_linear_whole_tiles_then_cluster_remainder(lib, M, N, K):
    """More weight tiles than SMs (not a multiple), one-SM tiles (pairs off): whole tiles on the
    persistent kernel, the rest on the cluster split-K kernel (two launches, no workspace);
    stream-K as the control."""
    X = bf16_dev(synth.normal_bf16_bits(M + 1, (M, K), 1.0))
    W = bf16_dev(synth.normal_bf16_bits(M + 2, (N, K), 0.02))
    R = bf16_dev(synth.normal_bf16_bits(M + 3, (M, N), 1.0))
    lib.spec_set_option("linear_pair", 0)
    try:
        assert lib.spec_linear_workspace_bytes(M, N, K) == 0
        lib.reset_launch_count()
        Y = lib.spec_verify_linear(X, W, residual=R)
        assert lib.launch_count() == 2
        lib.spec_set_option("linear_cluster", 0)
        Y2 = lib.spec_verify_linear(X, W, residual=R)
    finally:
        lib.spec_set_option("linear_cluster", 1)
        lib.spec_set_option("linear_pair", 1)
    lib.spec_device_status()
    rows = np.r_[0:4, M - 4:M]
    ref = oops.linear(obf.decode(bits_of(X))[rows], obf.decode(bits_of(W)), obf.decode(bits_of(R))[rows])
    assert_close_rel(f64_of_bf16(Y)[rows], ref, "dp + cluster remainder")
    assert_close_rel(f64_of_bf16(Y2)[rows], ref, "stream-K control")
