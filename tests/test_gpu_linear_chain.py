"""GPU parity of spec_verify_linear_chain (the small-M weight-streaming chain of verify linears).

Each product of a chain is checked against the fp64 oracle applied to the inputs that product
actually read (so the single-linear bar applies), on chains built to exercise every dependency the
library derives from address ranges: tokens produced by an earlier product (column-aligned, per
tile; and not aligned, whole product), an in-place residual stream, a buffer overwritten after an
earlier product read it (write-after-read), ragged shapes, SwiGLU products, more products than one
launch holds.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import bf16 as obf, ops as oops

from gpu_util import assert_close_chain, assert_close_rel, bf16_dev, bits_of, f64_of_bf16

pytestmark = pytest.mark.gpu


def w_dev(seed, n, k, std=0.03):
    return bf16_dev(synth.normal_bf16_bits(seed, (n, k), std))


def x_dev(seed, m, k, std=1.0):
    return bf16_dev(synth.normal_bf16_bits(seed, (m, k), std))


def ref_linear(X, W, R=None):
    return oops.linear(f64_of_bf16(X), f64_of_bf16(W), f64_of_bf16(R) if R is not None else None)


def ref_swiglu(X, Wgu, lib):
    """Oracle SwiGLU on interleaved gate|up rows (blocks of 16)."""
    w = f64_of_bf16(Wgu)
    N, K = w.shape
    b = lib.GATE_UP_BLOCK
    blocks = w.reshape(N // (2 * b), 2, b, K)
    g = oops.linear(f64_of_bf16(X), blocks[:, 0].reshape(-1, K))
    u = oops.linear(f64_of_bf16(X), blocks[:, 1].reshape(-1, K))
    return oops.silu_mul(g, u)


@pytest.mark.parametrize("M", [1, 3, 5, 16, 17, 32, 33, 40, 64])
def test_independent_products(lib, M):
    """Products with no shared buffers: ragged N, K not a multiple of 64, a SwiGLU product."""
    shapes = [(4096, 4096), (1000, 520), (6144, 4096), (136, 72), (384, 1000)]
    ops, refs = [], []
    for i, (N, K) in enumerate(shapes):
        X, W = x_dev(10 * i + M, M, K), w_dev(10 * i + M + 1, N, K)
        R = x_dev(10 * i + M + 2, M, N) if i % 2 else None
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        ops.append(lib.linear_op(X, W, Y, residual=R))
        refs.append((Y, ref_linear(X, W, R), f"product {i} N={N} K={K}"))
    X = x_dev(99 + M, M, 1024)
    Wgu = w_dev(98 + M, 2 * 1024, 1024)
    A = torch.full((M, 1024), float("nan"), dtype=torch.bfloat16, device="cuda")
    ops.append(lib.linear_op(X, Wgu, A, swiglu=True))
    refs.append((A, ref_swiglu(X, Wgu, lib), "swiglu product"))
    lib.spec_verify_linear_chain(ops, M)
    lib.spec_device_status()
    for Y, ref, what in refs:
        assert_close_rel(f64_of_bf16(Y), ref, f"chain M={M}: {what}")


def _layer_buffers(M, d, I, L, seed):
    dev = dict(dtype=torch.bfloat16, device="cuda")
    Wq = [w_dev(seed + 10 * l + 1, 3 * 256, d) for l in range(L)]
    Wo = [w_dev(seed + 10 * l + 2, d, 512) for l in range(L)]
    Wgu = [w_dev(seed + 10 * l + 3, 2 * I, d) for l in range(L)]
    Wd = [w_dev(seed + 10 * l + 4, d, I) for l in range(L)]
    h = x_dev(seed + 5, M, d)
    o = x_dev(seed + 6, M, 512)
    x0 = x_dev(seed + 7, M, d)
    return dev, Wq, Wo, Wgu, Wd, h, o, x0


@pytest.mark.parametrize("M", [1, 5, 16, 40])
@pytest.mark.parametrize("interleaved", [False, True])
def test_layer_chain_with_distinct_buffers(lib, M, interleaved):
    """QKV, O (+ residual), gate|up (SwiGLU), down (+ residual) per layer, every output in its own
    buffer: each product reads the previous products' outputs (down reads a as tokens per tile and x
    as residual), and each is checked against the oracle on what it read."""
    d, I, L = 1024, 1536, 3
    dev, Wq, Wo, Wgu, Wd, h, o, x0 = _layer_buffers(M, d, I, L, 300 + M)
    qkv = [torch.empty((M, 3 * 256), **dev) for _ in range(L)]
    xo = [torch.empty((M, d), **dev) for _ in range(L)]
    a = [torch.empty((M, I), **dev) for _ in range(L)]
    xd = [torch.empty((M, d), **dev) for _ in range(L)]
    per_layer = []
    for l in range(L):
        xin = x0 if l == 0 else xd[l - 1]
        per_layer.append([lib.linear_op(h, Wq[l], qkv[l]), lib.linear_op(o, Wo[l], xo[l], residual=xin),
                          lib.linear_op(h, Wgu[l], a[l], swiglu=True),
                          lib.linear_op(a[l], Wd[l], xd[l], residual=xo[l])])
    ops = []
    if interleaved:          # the next layer's QKV between gate|up and down
        for l in range(L):
            q, ob, gu, dn = per_layer[l]
            if l == 0:
                ops += [q]
            ops += [ob, gu] + ([per_layer[l + 1][0]] if l + 1 < L else []) + [dn]
    else:
        for l in range(L):
            ops += per_layer[l]
    lib.spec_verify_linear_chain(ops, M)
    lib.spec_device_status()
    for l in range(L):
        xin = x0 if l == 0 else xd[l - 1]
        assert_close_rel(f64_of_bf16(qkv[l]), ref_linear(h, Wq[l]), f"qkv {l}")
        assert_close_rel(f64_of_bf16(xo[l]), ref_linear(o, Wo[l], xin), f"o-proj {l}")
        assert_close_rel(f64_of_bf16(a[l]), ref_swiglu(h, Wgu[l], lib), f"swiglu {l}")
        assert_close_rel(f64_of_bf16(xd[l]), ref_linear(a[l], Wd[l], xo[l]), f"down {l}")


@pytest.mark.parametrize("M", [1, 5, 16, 64])
def test_layer_chain_in_place_matches_product_by_product(lib, M):
    """The residual stream updated in place (x = x + ...) and one activation buffer reused by every
    layer (gate|up of layer l+1 overwrites what down of layer l read): the chain equals the same
    products issued one call at a time, within the chain bar of L layers."""
    d, I, L = 1024, 1536, 4
    dev, Wq, Wo, Wgu, Wd, h, o, x0 = _layer_buffers(M, d, I, L, 700 + M)
    results = []
    for mode in ("chain", "calls"):
        x = x0.clone()
        qkv = torch.empty((M, 3 * 256), **dev)
        a = torch.empty((M, I), **dev)
        ops = []
        for l in range(L):
            ops += [lib.linear_op(h, Wq[l], qkv), lib.linear_op(o, Wo[l], x, residual=x),
                    lib.linear_op(h, Wgu[l], a, swiglu=True), lib.linear_op(a, Wd[l], x, residual=x)]
        if mode == "chain":
            lib.spec_verify_linear_chain(ops, M)
        else:
            for op in ops:
                lib.spec_verify_linear_chain([op], M)
        lib.spec_device_status()
        results.append((f64_of_bf16(x), f64_of_bf16(qkv), f64_of_bf16(a)))
    (xc, qc, ac), (xs, qs, as_) = results
    assert_close_chain(xc, xs, L, f"residual stream after {L} layers M={M}")
    assert_close_rel(qc, qs, "last qkv")
    assert_close_rel(ac, as_, "last activation")
    # and the product-by-product run against the oracle on the same chain
    x = f64_of_bf16(x0)
    for l in range(L):
        x = obf.round_to_bf16(ref_linear(o, Wo[l]) + x)
        a_ref = obf.round_to_bf16(ref_swiglu(h, Wgu[l], lib))
        x = obf.round_to_bf16(oops.linear(a_ref, f64_of_bf16(Wd[l])) + x)
    assert_close_chain(xs, x, L, "product by product vs oracle")


def test_write_after_read_waits(lib):
    """A big product reads buffer A; the next, small one overwrites A.  The first must see A's old
    contents on every CTA."""
    M = 8
    A = x_dev(1, M, 4096)
    A0 = A.clone()
    W1, Y1 = w_dev(2, 24576, 4096), torch.empty((M, 24576), dtype=torch.bfloat16, device="cuda")
    B, W2 = x_dev(3, M, 512), w_dev(4, 4096, 512)
    lib.spec_verify_linear_chain([lib.linear_op(A, W1, Y1), lib.linear_op(B, W2, A)], M)
    lib.spec_device_status()
    assert_close_rel(f64_of_bf16(Y1), ref_linear(A0, W1), "reader of the old A")
    assert_close_rel(f64_of_bf16(A), ref_linear(B, W2), "new A")


def test_tokens_from_a_column_slice_and_a_strided_view(lib):
    """Product 2 reads columns 128..1151 of product 1's output (aligned: per-tile waits); product 3
    reads product 1's output through a view with another leading dimension (whole-product wait)."""
    M = 6
    X1, W1 = x_dev(5, M, 2048), w_dev(6, 2048, 2048)
    Y1 = torch.empty((M, 2048), dtype=torch.bfloat16, device="cuda")
    W2, Y2 = w_dev(7, 640, 1024), torch.empty((M, 640), dtype=torch.bfloat16, device="cuda")
    view = Y1.view(-1)[: (M // 2) * 4096].view(M // 2, 4096)     # rows of 4096: two rows of Y1 each
    W3, Y3 = w_dev(8, 256, 4096), torch.empty((M // 2, 256), dtype=torch.bfloat16, device="cuda")
    lib.spec_verify_linear_chain([lib.linear_op(X1, W1, Y1), lib.linear_op(Y1[:, 128:1152], W2, Y2)], M)
    lib.spec_verify_linear_chain([lib.linear_op(X1, W1, Y1), lib.linear_op(view, W3, Y3)], M // 2)
    lib.spec_device_status()
    assert_close_rel(f64_of_bf16(Y2), ref_linear(Y1[:, 128:1152], W2), "aligned column slice")
    assert_close_rel(f64_of_bf16(Y3), ref_linear(view, W3), "strided view")


def test_more_products_than_one_launch(lib):
    """110 dependent products (three launches): a running sum y_{i+1} = x W_i^T + y_i."""
    M, K, N = 4, 256, 256
    X = x_dev(11, M, K)
    Ws = [w_dev(100 + i, N, K, std=0.01) for i in range(110)]
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    lib.reset_launch_count()
    lib.spec_verify_linear_chain([lib.linear_op(X, W, y, residual=y) for W in Ws], M)
    assert lib.launch_count() == 3
    lib.spec_device_status()
    ref = np.zeros((M, N))
    for W in Ws:
        ref = obf.round_to_bf16(ref_linear(X, W) + ref)
    assert_close_chain(f64_of_bf16(y), ref, len(Ws), "110-product running sum")


def test_bit_identical_on_repeat(lib):
    """The on-chip sums run in CTA order: two runs give the same bits."""
    M = 5
    X, W = x_dev(20, M, 4096), w_dev(21, 6144, 4096)
    outs = []
    for _ in range(2):
        Y = torch.empty((M, 6144), dtype=torch.bfloat16, device="cuda")
        lib.spec_verify_linear_chain([lib.linear_op(X, W, Y)], M)
        outs.append(bits_of(Y))
    lib.spec_device_status()
    assert np.array_equal(outs[0], outs[1])
