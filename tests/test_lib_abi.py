"""CPU checks of the C ABI library: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch
(no device is touched by these calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def built():
    from speculative_decoding_verify_05_gb300.build import build
    return build()


def header_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^SPEC_API\s+[\w\s\*]+?\b(spec_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    syms = header_symbols()
    for name in ("spec_verify_linear", "spec_verify_attention", "spec_lmhead_softmax",
                 "spec_reject_sample"):
        assert name in syms
    assert len(syms) >= 14


def test_library_exports_every_declared_symbol(built):
    lib = ctypes.CDLL(built)
    for name in header_symbols():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {built}").read()
    exported = set(re.findall(r" T (spec_\w+)", out))
    assert exported == set(header_symbols())


def test_binding_covers_the_header(built):
    from speculative_decoding_verify_05_gb300 import binding
    assert sorted(binding.EXPORTS) == header_symbols()
    assert binding.spec_version() == 1


def test_host_side_validation(built):
    from speculative_decoding_verify_05_gb300 import binding as S
    L = S._lib
    E = S.SPEC_EINVAL
    # null tensors, bad K, bad leading dimension
    assert L.spec_verify_linear(None, 4, 64, 64, None, 128, 64, None, 128, None, 0, None, 0, None) == E
    fake = ctypes.c_void_p(1 << 20)
    assert L.spec_verify_linear(fake, 4, 60, 64, fake, 128, 64, fake, 128, None, 0, None, 0, None) == E
    assert b"multiple of 8" in L.spec_last_error()
    assert L.spec_verify_linear(fake, 4, 64, 32, fake, 128, 64, fake, 128, None, 0, None, 0, None) == E
    # misaligned pointer
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert L.spec_verify_linear(odd, 4, 64, 64, fake, 128, 64, fake, 128, None, 0, None, 0, None) == E
    # M = 0 is a no-op that succeeds without touching anything
    assert L.spec_verify_linear(None, 0, 64, 64, None, 128, 64, None, 128, None, 0, None, 0, None) == 0
    # fused SwiGLU linear: I must be a multiple of 64, A's leading dimension at least I
    assert L.spec_verify_linear_swiglu(fake, 4, 64, 64, fake, 64, 96, fake, 96, None, 0, None) == E
    assert b"multiple of 64" in L.spec_last_error()
    assert L.spec_verify_linear_swiglu(fake, 4, 64, 64, fake, 64, 128, fake, 64, None, 0, None) == E
    assert L.spec_verify_linear_swiglu(odd, 4, 64, 64, fake, 64, 128, fake, 128, None, 0, None) == E
    assert L.spec_verify_linear_swiglu(None, 0, 64, 64, None, 64, 128, None, 128, None, 0, None) == 0
    # attention: unsupported head dim, too many rows per kv head
    args = [fake, 32 * 64, fake, fake, 8 * 64, fake, fake, 2, 5, fake, fake, 64, 32, 8, 64, 0.1, fake,
            32 * 64, None, 0, None]
    assert L.spec_verify_attention(*args) == S.SPEC_EUNSUPPORTED
    args = [fake, 32 * 128, fake, fake, 8 * 128, fake, fake, 2, 17, fake, fake, 64, 32, 8, 128, 0.1, fake,
            32 * 128, None, 0, None]
    assert L.spec_verify_attention(*args) == S.SPEC_EUNSUPPORTED
    # workspace too small
    args[-3] = fake
    args[-2] = 16
    args[8] = 4
    assert L.spec_verify_attention(*args) == E
    assert b"workspace" in L.spec_last_error()
    # LM head: negative temperature, V not a multiple of 4
    assert L.spec_lmhead_softmax(fake, 2, 64, fake, 128, -1.0, fake, fake, 1 << 30, None) == E
    assert L.spec_lmhead_softmax(fake, 2, 64, fake, 126, 1.0, fake, fake, 1 << 30, None) == E
    # sampler: null outputs
    assert L.spec_reject_sample(fake, fake, fake, fake, fake, 3, 8, 1e-5, None, fake, fake, None) == E
    # paged attention: no block table, no pages
    assert L.spec_verify_attention_paged(fake, 32 * 128, fake, fake, 8 * 128, fake, fake, 2, 5, fake, fake, 4,
                                         None, 2, 32, 8, 128, 0.1, fake, 32 * 128, fake, 1 << 30, None) == E
    assert L.spec_verify_attention_paged(fake, 32 * 128, fake, fake, 8 * 128, fake, fake, 2, 5, fake, fake, 0,
                                         fake, 2, 32, 8, 128, 0.1, fake, 32 * 128, fake, 1 << 30, None) == E
    # draft side: embedding with d not a multiple of 8, sampling rows with ldp < V, LM head ldp < V
    assert L.spec_embed(fake, 4, fake, 100, 12, 12, fake, 12, None) == E
    assert L.spec_sample_rows(fake, 10, 4, 16, fake, fake, None) == E
    assert L.spec_lmhead_softmax_ld(fake, 2, 64, fake, 128, 1.0, fake, 64, fake, 1 << 30, None) == E
    # n-gram drafter: empty window, window past the limit, k = 0
    assert L.spec_ngram_propose(fake, fake, 2, 4, 3, 2, fake, fake, None) == E
    assert L.spec_ngram_propose(fake, fake, 2, 4, 1, 65, fake, fake, None) == E
    assert L.spec_ngram_propose(fake, fake, 2, 0, 1, 4, fake, fake, None) == E
    assert L.spec_ngram_propose(None, None, 0, 4, 1, 4, None, None, None) == 0
    # typical acceptance: negative floor, infinite slope
    assert L.spec_typical_sample(fake, fake, fake, fake, 3, 8, -0.1, 0.3, 1e-5, fake, fake, fake, None) == E
    assert L.spec_typical_sample(fake, fake, fake, fake, 3, 8, 0.1, float("inf"), 1e-5, fake, fake, fake, None) == E
    # fused LM head -> sampler: fewer rows than sequences, null outputs, small workspace
    assert L.spec_lmhead_reject_sample(fake, 2, 64, fake, 128, 1.0, fake, fake, fake, fake, 3, 1e-5,
                                       fake, fake, fake, fake, 1 << 30, None) == E
    assert L.spec_lmhead_reject_sample(fake, 4, 64, fake, 128, 1.0, fake, fake, fake, fake, 3, 1e-5,
                                       None, fake, fake, fake, 1 << 30, None) == E
    assert L.spec_lmhead_reject_sample(fake, 4, 64, fake, 128, 1.0, fake, fake, fake, fake, 3, 1e-5,
                                       fake, fake, fake, fake, 16, None) == E
    assert b"workspace" in L.spec_last_error()
    assert L.spec_lmhead_reject_sample(fake, 4, 64, fake, 128, 1.0, fake, fake, fake, fake, 0, 1e-5,
                                       None, None, None, None, 0, None) == 0
    # options
    assert L.spec_set_option(b"no_such_knob", 1) == E
    assert L.spec_set_option(b"gemv_max_m", 9) == E
    assert L.spec_set_option(b"gemv_max_m", 4) == 0
    assert L.spec_set_option(b"gemv_max_m", 0) == 0
    assert L.spec_set_option(b"attention_pair_cost", 65) == E
    assert L.spec_set_option(b"attention_pair_cost", -1) == E
    assert L.spec_set_option(b"attention_pair_cost", 8) == 0
    assert L.spec_set_option(b"linear_multicast", 1) == E      # removed knob
    assert L.spec_set_option(b"linear_pair_persistent", 3) == E
    assert L.spec_set_option(b"linear_split_rows", 2) == E
    assert L.spec_set_option(b"linear_split_rows", 0) == 0
    assert L.spec_set_option(b"linear_split_rows", 1) == 0
    assert L.spec_set_option(b"weight_prefetch", 2) == E
    assert L.spec_set_option(b"weight_prefetch", 0) == 0
    assert L.spec_set_option(b"weight_prefetch", 1) == 0
    assert L.spec_set_option(b"linear_pair_persistent", 0) == 0
    assert L.spec_set_option(b"lmhead_pair", 2) == E
    assert L.spec_set_option(b"lmhead_pair", 1) == 0
    assert L.spec_set_option(b"kv_l2_promotion", 4) == E
    assert L.spec_set_option(b"kv_l2_promotion", 3) == 0
    # the bounded-wait probe checks its limit before touching the device
    assert L.spec_probe_bounded_wait(0, 0, None) == E
    assert L.spec_probe_bounded_wait(2000001, 0, None) == E
    assert L.spec_probe_bounded_wait(100, 2, None) == E
    # the allocation-free linear rejects bad arguments before any CUDA call
    assert L.spec_verify_linear_noalloc(None, 4, 64, 64, fake, 128, 64, fake, 128, None, 0, None) == E
    assert L.spec_verify_linear_noalloc(fake, 4, 64, 64, fake, 128, 64, fake, 128, odd, 128, None) == E
    assert L.spec_launches() == 0


def test_workspace_queries_are_host_only(built):
    from speculative_decoding_verify_05_gb300 import binding as S
    # split-K needs counters + partials; the counter region is a fixed 64 KiB
    n = S.spec_linear_workspace_bytes(5, 4096, 4096)
    assert n == 0 or n > 64 * 1024
    assert S.spec_attention_workspace_bytes(8, 5, 32, 8, 128, 4101) > 64 * 1024
    assert S.spec_lmhead_workspace_bytes(40, 4096, 151936) >= 64 * 1024 + 40 * 1187 * 8
    assert S.spec_linear_workspace_bytes(0, 4096, 4096) == 0
    # the fused LM head keeps the logits (fp32) unless it is greedy
    full = S.spec_lmhead_sample_workspace_bytes(40, 4096, 151936, 1.0)
    greedy = S.spec_lmhead_sample_workspace_bytes(40, 4096, 151936, 0.0)
    assert full >= greedy + 40 * 151936 * 4 and greedy == S.spec_lmhead_workspace_bytes(40, 4096, 151936)


def test_gate_up_interleave_layout(built):
    """Rows 32 j .. 32 j + 15 are gate rows 16 j .., the next 16 the matching up rows; the
    engine's in-place relayout goes there and back."""
    import torch
    from speculative_decoding_verify_05_gb300 import binding as S, engine as E
    I, K = 192, 8
    Wg = torch.arange(I * K, dtype=torch.float32).reshape(I, K).to(torch.bfloat16)
    Wu = -torch.arange(I * K, dtype=torch.float32).reshape(I, K).to(torch.bfloat16) - 1
    Wgu = S.interleave_gate_up(Wg, Wu)
    assert Wgu.shape == (2 * I, K)
    for j in range(I // 16):
        assert torch.equal(Wgu[32 * j:32 * j + 16], Wg[16 * j:16 * j + 16])
        assert torch.equal(Wgu[32 * j + 16:32 * j + 32], Wu[16 * j:16 * j + 16])
    split = torch.cat((Wg, Wu), 0)
    lw = E.LayerW(None, None, split.clone(), None, None, None)
    E.set_gu_layout(lw, "interleaved")
    assert torch.equal(lw.w_gu, Wgu) and lw.gu_layout == "interleaved"
    E.set_gu_layout(lw, "interleaved")            # idempotent
    assert torch.equal(lw.w_gu, Wgu)
    E.set_gu_layout(lw, "split")
    assert torch.equal(lw.w_gu, split) and lw.gu_layout == "split"
    with pytest.raises(ValueError):
        S.interleave_gate_up(Wg[:100], Wu[:100])
