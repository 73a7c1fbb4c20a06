"""GPU parity of spec_verify_attention_paged (paged KV cache, 128-key pages).

The paged pass visits the same key tiles in the same order as the contiguous one, so with the
cache's contents scattered into randomly permuted pages it must return bit-identical outputs
and write bit-identical cache rows; the oracle checks the result too.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import bf16 as obf, ops as oops

from gpu_util import assert_close_attn, bf16_dev, bits_of, dev

pytestmark = pytest.mark.gpu
PAGE = 128


def paged_case(seed, gammas, ctx, Hq=32, Hkv=8, extra_pages=5):
    rng = np.random.default_rng(seed)
    batch = synth.RaggedBatch(gammas, ctx)
    D = 128
    need = [(c + g + 1 + PAGE - 1) // PAGE for c, g in zip(batch.ctx_len, batch.gammas)]
    max_pages = max(need)
    cap = max_pages * PAGE
    kc = synth.normal_bf16_bits(seed + 1, (batch.B, Hkv, cap, D), 1.0)
    vc = synth.normal_bf16_bits(seed + 2, (batch.B, Hkv, cap, D), 1.0)
    qkv = synth.normal_bf16_bits(seed + 3, (batch.M, (Hq + 2 * Hkv) * D), 1.0)
    num_pages = batch.B * max_pages + extra_pages
    perm = rng.permutation(num_pages)
    table = perm[:batch.B * max_pages].reshape(batch.B, max_pages).astype(np.int32)
    kpool = synth.normal_bf16_bits(seed + 4, (Hkv, num_pages, PAGE, D), 1.0)   # unused pages: noise
    vpool = synth.normal_bf16_bits(seed + 5, (Hkv, num_pages, PAGE, D), 1.0)
    for b in range(batch.B):
        for t in range(max_pages):
            kpool[:, table[b, t]] = kc[b, :, t * PAGE:(t + 1) * PAGE]
            vpool[:, table[b, t]] = vc[b, :, t * PAGE:(t + 1) * PAGE]
    return batch, Hq, Hkv, D, kc, vc, qkv, table, kpool, vpool


def gather(pool, table):
    B, max_pages = table.shape
    return np.stack([np.concatenate([pool[:, table[b, t]] for t in range(max_pages)], axis=1) for b in range(B)])


@pytest.mark.parametrize("gammas,ctx", [
    ([3, 0, 7, 2, 10, 1, 5, 4], [100, 127, 128, 255, 700, 1, 0, 383]),
    ([4] * 16, list(range(120, 120 + 16 * 61, 61))),
])
def test_paged_equals_contiguous_and_oracle(lib, gammas, ctx):
    batch, Hq, Hkv, D, kc, vc, qkv, table, kpool, vpool = paged_case(7, gammas, ctx)
    hq, hk = Hq * D, Hkv * D
    Qd = bf16_dev(qkv)
    cu, cx = dev(batch.cu_rows), dev(batch.ctx_len)
    Kc, Vc = bf16_dev(kc).clone(), bf16_dev(vc).clone()
    O1 = lib.spec_verify_attention(Qd[:, :hq], Qd[:, hq:hq + hk], Qd[:, hq + hk:], cu, cx, Kc, Vc, batch.max_rows)
    Kp, Vp = bf16_dev(kpool).clone(), bf16_dev(vpool).clone()
    O2 = lib.spec_verify_attention_paged(Qd[:, :hq], Qd[:, hq:hq + hk], Qd[:, hq + hk:], cu, cx, Kp, Vp,
                                         dev(table), batch.max_rows)
    lib.spec_device_status()
    assert torch.equal(O1, O2)
    kp_after, vp_after = bits_of(Kp), bits_of(Vp)
    assert np.array_equal(gather(kp_after, table), bits_of(Kc))
    assert np.array_equal(gather(vp_after, table), bits_of(Vc))
    unused = np.setdiff1d(np.arange(kpool.shape[1]), table.reshape(-1))
    assert np.array_equal(kp_after[:, unused], kpool[:, unused]) and np.array_equal(vp_after[:, unused], vpool[:, unused])
    # and the oracle on the gathered cache
    q = obf.decode(qkv[:, :hq]).reshape(batch.M, Hq, D)
    k = obf.decode(qkv[:, hq:hq + hk]).reshape(batch.M, Hkv, D)
    v = obf.decode(qkv[:, hq + hk:]).reshape(batch.M, Hkv, D)
    ref, _, _ = oops.verify_attention(q, k, v, batch.cu_rows, obf.decode(kc), obf.decode(vc), batch.ctx_len,
                                      1.0 / np.sqrt(D))
    # magnitude of the summed terms: the same weights applied to |v| (the attention bar)
    mag, _, _ = oops.verify_attention(q, k, np.abs(v), batch.cu_rows, obf.decode(kc), np.abs(obf.decode(vc)),
                                      batch.ctx_len, 1.0 / np.sqrt(D))
    got = obf.decode(bits_of(O2)).reshape(batch.M, Hq, D)
    assert_close_attn(got, ref, mag, "paged attention")


def test_paged_bad_page_id_is_flagged(lib):
    batch, Hq, Hkv, D, kc, vc, qkv, table, kpool, vpool = paged_case(9, [2, 1], [200, 50])
    hq, hk = Hq * D, Hkv * D
    table[0, 0] = kpool.shape[1] + 3               # read by sequence 0's first tile
    Qd = bf16_dev(qkv)
    lib.spec_verify_attention_paged(Qd[:, :hq], Qd[:, hq:hq + hk], Qd[:, hq + hk:], dev(batch.cu_rows),
                                    dev(batch.ctx_len), bf16_dev(kpool), bf16_dev(vpool), dev(table),
                                    batch.max_rows)
    with pytest.raises(lib.SpecError):
        lib.spec_device_status()
    lib.spec_device_status()
