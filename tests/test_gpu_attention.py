"""GPU parity of spec_verify_attention against the oracle (outputs and cache append)."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import bf16 as obf, ops as oops

from gpu_util import assert_close_attn, bf16_dev, bits_of, dev, f64_of_bf16

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(params=[1, 0], ids=["tcgen05", "mma_sync"])
def impl(request, lib):
    """Run each case on both attention kernels (tcgen05 is the default)."""
    lib.spec_set_option("attention_impl", request.param)
    yield request.param
    lib.spec_set_option("attention_impl", 1)


def run_case(lib, gammas, ctx, Hq, Hkv, seed, cap=None, fused_qkv=True):
    batch = synth.RaggedBatch(gammas, ctx, cap)
    M, B = batch.M, batch.B
    G = Hq // Hkv
    width = (Hq + 2 * Hkv) * D
    qkv = synth.normal_bf16_bits(seed, (M, width), 1.0)
    kc = synth.normal_bf16_bits(seed + 1, (B, Hkv, batch.cap, D), 1.0)
    vc = synth.normal_bf16_bits(seed + 2, (B, Hkv, batch.cap, D), 1.0)
    qkv_d = bf16_dev(qkv)
    hq, hk = Hq * D, Hkv * D
    if fused_qkv:
        Qd, Kd, Vd = qkv_d[:, :hq], qkv_d[:, hq:hq + hk], qkv_d[:, hq + hk:]
    else:
        Qd, Kd, Vd = (qkv_d[:, :hq].contiguous(), qkv_d[:, hq:hq + hk].contiguous(),
                      qkv_d[:, hq + hk:].contiguous())
    kcd, vcd = bf16_dev(kc), bf16_dev(vc)
    scale = 1.0 / math.sqrt(D)
    O = lib.spec_verify_attention(Qd, Kd, Vd, dev(batch.cu_rows), dev(batch.ctx_len), kcd, vcd,
                                  batch.max_rows, scale=scale)
    lib.spec_device_status()
    q = obf.decode(qkv[:, :hq]).reshape(M, Hq, D)
    k = obf.decode(qkv[:, hq:hq + hk]).reshape(M, Hkv, D)
    v = obf.decode(qkv[:, hq + hk:]).reshape(M, Hkv, D)
    Oref, Kref, Vref = oops.verify_attention(q, k, v, batch.cu_rows, obf.decode(kc), obf.decode(vc),
                                             batch.ctx_len, scale)
    # magnitude of the summed terms: the same weights applied to |v|
    Omag, _, _ = oops.verify_attention(q, k, np.abs(v), batch.cu_rows, obf.decode(kc),
                                       np.abs(obf.decode(vc)), batch.ctx_len, scale)
    assert_close_attn(f64_of_bf16(O).reshape(M, Hq, D), Oref, Omag, f"attention B={B} G={G}")
    # the cache append is a byte copy: bit-exact
    assert np.array_equal(obf.decode(bits_of(kcd)), Kref)
    assert np.array_equal(obf.decode(bits_of(vcd)), Vref)
    return batch


@pytest.mark.parametrize("gammas,ctx,Hq,Hkv", [
    ([0], [0], 4, 1),                         # a single key: output = its value
    ([4], [37], 32, 8),                       # config-1-like row count, GQA 4
    ([2, 0, 5], [7, 70, 0], 8, 2),            # ragged, one empty context
    ([10, 3, 7, 1], [130, 64, 511, 1000], 32, 8),   # 11 rows x 4 heads = 44 rows (4 m-tiles)
    ([3, 3], [300, 2], 16, 4),                # 16 rows: one m-tile
    ([6, 1], [90, 63], 16, 8),                # G = 2
    ([15], [5], 4, 1),                        # G*rows = 64 exactly
])
def test_attention_small(lib, impl, gammas, ctx, Hq, Hkv):
    run_case(lib, gammas, ctx, Hq, Hkv, seed=sum(ctx) + len(gammas))


def test_attention_split_kv_long_context(lib, impl):
    # long contexts with few sequences: several key chunks per (sequence, kv head)
    run_case(lib, [4, 2], [3000, 4096], 32, 8, seed=77)


def test_attention_separate_qkv_buffers(lib, impl):
    run_case(lib, [4, 1], [200, 17], 32, 8, seed=5, fused_qkv=False)


def test_attention_cap_with_slack(lib, impl):
    run_case(lib, [3, 9], [100, 500], 32, 8, seed=6, cap=700)


def test_attention_row_equals_single_decode(lib, impl):
    """Row j of a verify block equals a one-row call at context ctx + j (caches after j steps)."""
    gam, ctx, Hq, Hkv = 5, 150, 32, 8
    width = (Hq + 2 * Hkv) * D
    M = gam + 1
    qkv = bf16_dev(synth.normal_bf16_bits(31, (M, width), 1.0))
    kc0 = bf16_dev(synth.normal_bf16_bits(32, (1, Hkv, 200, D), 1.0))
    vc0 = bf16_dev(synth.normal_bf16_bits(33, (1, Hkv, 200, D), 1.0))
    hq, hk = Hq * D, Hkv * D
    kc, vc = kc0.clone(), vc0.clone()
    Ov = lib.spec_verify_attention(qkv[:, :hq], qkv[:, hq:hq + hk], qkv[:, hq + hk:],
                                   dev(np.array([0, M], np.int32)), dev(np.array([ctx], np.int32)),
                                   kc, vc, M)
    kd, vd = kc0.clone(), vc0.clone()
    rows = []
    for j in range(M):
        r = qkv[j:j + 1]
        rows.append(lib.spec_verify_attention(r[:, :hq], r[:, hq:hq + hk], r[:, hq + hk:],
                                              dev(np.array([0, 1], np.int32)),
                                              dev(np.array([ctx + j], np.int32)), kd, vd, 1))
    lib.spec_device_status()
    Od = torch.cat(rows)
    assert torch.equal(kc, kd) and torch.equal(vc, vd)
    # both sides round probabilities to bf16 at different running maxima: twice the one-side bar
    qkv_h = f64_of_bf16(qkv)
    q = qkv_h[:, :hq].reshape(M, Hq, D)
    k = qkv_h[:, hq:hq + hk].reshape(M, Hkv, D)
    v = qkv_h[:, hq + hk:].reshape(M, Hkv, D)
    Omag, _, _ = oops.verify_attention(q, k, np.abs(v), np.array([0, M]), f64_of_bf16(kc0),
                                       np.abs(f64_of_bf16(vc0)), np.array([ctx]), 1.0 / math.sqrt(D))
    assert_close_attn(f64_of_bf16(Ov).reshape(M, Hq, D), f64_of_bf16(Od).reshape(M, Hq, D), Omag,
                      "verify vs sequential decode", abs_frac=4.0 * 2.0 ** -9)


def test_attention_config3_shapes(lib, impl):
    """B=8, gamma=4, GQA 32/8, contexts U[512, 4096] (the verify-attention workload's shapes)."""
    batch = synth.ragged_batch(3, 8, 4, 4, 512, 4096)
    run_case(lib, batch.gammas, batch.ctx_len, 32, 8, seed=123)


@pytest.mark.parametrize("grid", [1, 5, 37, 300])
def test_attention_persistent_grids(lib, grid):
    """Different persistent grids cut the (sequence, kv head) pairs into different pieces."""
    lib.spec_set_option("persistent_grid", grid)
    try:
        run_case(lib, [10, 3, 7, 1, 0], [130, 64, 511, 1000, 2], 32, 8, seed=40 + grid)
        run_case(lib, [4, 2], [3000, 260], 16, 4, seed=41 + grid)
    finally:
        lib.spec_set_option("persistent_grid", 0)


def test_attention_very_long_context_many_pieces(lib, impl):
    """A context past 16k keys; with 300 CTAs each pair is cut into ~150 pieces to merge."""
    lib.spec_set_option("persistent_grid", 300)
    try:
        run_case(lib, [3], [20000], 8, 2, seed=9)
    finally:
        lib.spec_set_option("persistent_grid", 0)


@pytest.mark.parametrize("pair_cost", [0, 8, 64])
@pytest.mark.parametrize("grid", [7, 0, 300])
def test_attention_pair_cost_partitions(lib, pair_cost, grid):
    """Cost-balanced splits (pair starts charged 0, 2 or 16 tiles) over several grids, including
    grids with more CTAs than tiles (empty ranges between the pieces of one pair)."""
    lib.spec_set_option("attention_pair_cost", pair_cost)
    lib.spec_set_option("persistent_grid", grid)
    try:
        run_case(lib, [10, 3, 7, 1, 0, 5], [130, 64, 511, 1000, 2, 2900], 32, 8, seed=60 + grid + pair_cost)
        run_case(lib, [0, 2], [126, 3], 8, 8, seed=61 + grid)
        run_case(lib, [4], [130], 4, 2, seed=62 + grid)          # 4 tiles: most CTAs get nothing
    finally:
        lib.spec_set_option("attention_pair_cost", 12)
        lib.spec_set_option("persistent_grid", 0)


@pytest.mark.parametrize("grid,B", [(0, 48), (5, 48), (37, 48), (300, 96)])
def test_attention_many_short_pairs(lib, grid, B):
    """48 or 96 sequences x 8 kv heads of short contexts (0-700 keys, 1-6 rows): many pairs per
    CTA, on several grids including more CTAs than fit on the GPU at once."""
    rng = np.random.default_rng(grid + B)
    gammas, ctx = list(rng.integers(0, 6, size=B)), list(rng.integers(0, 700, size=B))
    lib.spec_set_option("persistent_grid", grid)
    try:
        run_case(lib, gammas, ctx, 32, 8, seed=90 + grid)
    finally:
        lib.spec_set_option("persistent_grid", 0)


def test_attention_at_the_batch_limit(lib):
    """1024 sequences, the most the tcgen05 kernel takes, of short contexts (0-199 keys, 1-4 rows):
    the per-sequence metadata its set-up stages in the V ring (3 x 1024 + 2 ints) and each CTA's
    1025-entry prefix slice in the workspace are at their largest, and most CTAs start many pairs."""
    rng = np.random.default_rng(7)
    B = 1024
    gammas, ctx = list(rng.integers(0, 4, size=B)), list(rng.integers(0, 200, size=B))
    run_case(lib, gammas, ctx, 8, 2, seed=1024)


def test_attention_full_ragged_round_sampled(lib):
    """The benchmark's attention launch at full size: B = 64, gamma_b ~ U{1..10}, ctx_b ~ U[128, 8192],
    GQA 32/8, D = 128, the default persistent grid and pair cost.  Outputs and the cache append are
    checked against the oracle on a sample of sequences (the shortest and longest contexts, the
    longest block and four seeded picks); the oracle sees host copies taken before the launch."""
    batch = synth.ragged_batch(0, 64, 1, 10, 128, 8192)
    Hq, Hkv, B, M = 32, 8, batch.B, batch.M
    cap = int((batch.ctx_len + batch.gammas + 1).max() + 15) // 16 * 16
    g = torch.Generator(device="cuda")
    g.manual_seed(2024)
    kc = torch.empty((B, Hkv, cap, D), dtype=torch.bfloat16, device="cuda").normal_(0, 1, generator=g)
    vc = torch.empty_like(kc).normal_(0, 1, generator=g)
    qkv = torch.empty((M, (Hq + 2 * Hkv) * D), dtype=torch.bfloat16, device="cuda").normal_(0, 1, generator=g)
    rng = np.random.default_rng(5)
    picks = {int(np.argmin(batch.ctx_len)), int(np.argmax(batch.ctx_len)), int(np.argmax(batch.gammas))}
    picks |= {int(b) for b in rng.choice(B, 4, replace=False)}
    picks = sorted(picks)
    qkv_h = bits_of(qkv)
    kc_h = {b: bits_of(kc[b]) for b in picks}
    vc_h = {b: bits_of(vc[b]) for b in picks}
    hq, hk = Hq * D, Hkv * D
    scale = 1.0 / math.sqrt(D)
    O = lib.spec_verify_attention(qkv[:, :hq], qkv[:, hq:hq + hk], qkv[:, hq + hk:], dev(batch.cu_rows),
                                  dev(batch.ctx_len), kc, vc, batch.max_rows, scale=scale)
    lib.spec_device_status()
    for b in picks:
        r0, r1 = int(batch.cu_rows[b]), int(batch.cu_rows[b + 1])
        mb = r1 - r0
        rows = qkv_h[r0:r1]
        q = obf.decode(rows[:, :hq]).reshape(mb, Hq, D)
        k = obf.decode(rows[:, hq:hq + hk]).reshape(mb, Hkv, D)
        v = obf.decode(rows[:, hq + hk:]).reshape(mb, Hkv, D)
        cu1, ctx1 = np.array([0, mb]), np.array([int(batch.ctx_len[b])])
        kc1, vc1 = obf.decode(kc_h[b])[None], obf.decode(vc_h[b])[None]
        Oref, Kref, Vref = oops.verify_attention(q, k, v, cu1, kc1, vc1, ctx1, scale)
        Omag, _, _ = oops.verify_attention(q, k, np.abs(v), cu1, kc1, np.abs(vc1), ctx1, scale)
        assert_close_attn(f64_of_bf16(O[r0:r1]).reshape(mb, Hq, D), Oref, Omag,
                          f"full round: sequence {b} (ctx {ctx1[0]}, {mb} rows)")
        assert np.array_equal(obf.decode(bits_of(kc[b])), Kref[0])
        assert np.array_equal(obf.decode(bits_of(vc[b])), Vref[0])
