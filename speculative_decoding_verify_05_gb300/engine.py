"""Verify-round driver for a Qwen3-8B-shaped decoder stack, built on the C ABI.

This is the caller's side of the library boundary: it owns device buffers
(torch allocations), walks the layers and issues one library call per step
of the verify pass, all on the current stream so that a whole round can be
captured in one CUDA graph.  It computes nothing itself.

Layer reading (the pages give only the shape: 36 layers, 32 query / 8 kv
heads of 128, grouped-query attention, a 151936-token vocabulary): pre-RMSNorm
(eps 1e-6), fused QKV projection, RoPE (theta 1e6, rotate-half) on q and k,
causal verify attention over the cache, O projection + residual, RMSNorm,
fused gate/up projection, SwiGLU, down projection + residual; final RMSNorm
and LM head.  By default the SwiGLU activation runs in the gate/up GEMM's
epilogue (spec_verify_linear_swiglu), which wants the gate and up weight rows
interleaved in blocks of 16: the engine relays each layer's ``w_gu`` out once,
in place, when it is built.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import binding as S


@dataclass
class Dims:
    d: int = 4096
    Hq: int = 32
    Hkv: int = 8
    D: int = 128
    I: int = 12288
    V: int = 151936
    layers: int = 36
    eps: float = 1e-6
    theta: float = 1e6

    @property
    def qkv(self) -> int:
        return (self.Hq + 2 * self.Hkv) * self.D


def draft_dims() -> Dims:
    """A Qwen3-0.6B-shaped draft stack: 28 layers, d 1024, 16 query / 8 kv heads of 128, I 3072,
    vocabulary 151936 shared with the target (LM head tied to the embedding table)."""
    return Dims(d=1024, Hq=16, Hkv=8, D=128, I=3072, V=151936, layers=28)


@dataclass
class LayerW:
    w_qkv: torch.Tensor      # [(Hq + 2 Hkv) D, d]
    w_o: torch.Tensor        # [d, Hq D]
    w_gu: torch.Tensor       # [2 I, d]  gate rows then up rows (see gu_layout)
    w_down: torch.Tensor     # [d, I]
    attn_norm: torch.Tensor  # [d]
    mlp_norm: torch.Tensor   # [d]
    gu_layout: str = "split"  # "split": gate rows then up rows; "interleaved": blocks of 16


@dataclass
class StackW:
    layers: list = field(default_factory=list)
    final_norm: torch.Tensor | None = None
    w_lm: torch.Tensor | None = None
    norms_folded: bool = False   # RMSNorm weights multiplied into the products that consume them


def fold_norm_weights(sw: StackW) -> None:
    """Folds each RMSNorm weight into the product that reads the normed rows, once, in place:
    W_qkv <- W_qkv diag(attn_norm), W_gu <- W_gu diag(mlp_norm), W_lm <- W_lm diag(final_norm)
    (one bf16 rounding of W w; exact for unit weights), and sets the norm weights to 1, so a
    product can take the raw rows and scale them by 1 / rms in its epilogue."""
    if sw.norms_folded:
        return
    for lw in sw.layers:
        lw.w_qkv.mul_(lw.attn_norm[None, :])
        lw.w_gu.mul_(lw.mlp_norm[None, :])
    if sw.w_lm is not None and sw.final_norm is not None:
        sw.w_lm.mul_(sw.final_norm[None, :])
    for lw in sw.layers:
        lw.attn_norm.fill_(1.0)
        lw.mlp_norm.fill_(1.0)
    if sw.final_norm is not None:
        sw.final_norm.fill_(1.0)
    sw.norms_folded = True


def random_stack(dims: Dims, seed: int, device, std: float = 0.02, with_head: bool = True) -> StackW:
    """Random-init bf16 weights N(0, std^2) of the stack's shapes (norm weights = 1)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def w(rows, cols):
        t = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
        t.normal_(0.0, std, generator=g)
        return t

    ones = torch.ones(dims.d, dtype=torch.bfloat16, device=device)
    sw = StackW()
    for _ in range(dims.layers):
        sw.layers.append(LayerW(w(dims.qkv, dims.d), w(dims.d, dims.Hq * dims.D), w(2 * dims.I, dims.d),
                                w(dims.d, dims.I), ones, ones))
    sw.final_norm = ones
    if with_head:
        sw.w_lm = w(dims.V, dims.d)
    return sw


def set_gu_layout(lw: LayerW, layout: str) -> None:
    """Reorders ``lw.w_gu``'s rows in place to ``layout`` (a one-time weight relayout)."""
    if lw.gu_layout == layout:
        return
    w = lw.w_gu
    I2, K = w.shape
    I = I2 // 2
    if layout == "interleaved":
        w.copy_(S.interleave_gate_up(w[:I], w[I:]))
    elif layout == "split":
        b = S.GATE_UP_BLOCK
        blocks = w.reshape(I // b, 2, b, K)
        w.copy_(torch.cat((blocks[:, 0].reshape(I, K), blocks[:, 1].reshape(I, K)), dim=0))
    else:
        raise ValueError(f"unknown gate/up layout {layout!r}")
    lw.gu_layout = layout


class VerifyEngine:
    """Buffers + call sequence of one verify pass / round for up to ``max_M`` rows."""

    def __init__(self, dims: Dims, weights: StackW, kcaches, vcaches, max_M: int, max_rows: int,
                 device=None, fused_swiglu: bool = True, fused_sampler: bool = True, fused_rope: bool = True,
                 fold_norms: bool = True):
        self.dims = dims
        self.w = weights
        # verify_round: LM head and sampler in one call that never materialises p
        self.fused_sampler = fused_sampler
        # RoPE applied by the QKV projection from a per-pass (cos, sin) table (head size 128 only)
        self.fused_rope = fused_rope and dims.D == 128
        self.fused_swiglu = fused_swiglu and dims.I % 64 == 0
        want = "interleaved" if self.fused_swiglu else "split"
        for lw in weights.layers:
            set_gu_layout(lw, want)
        # RMSNorm folded into the products: the products that store the residual stream leave its
        # per-tile sums of squares, the products that read it scale their rows (no norm launches)
        self.fold_norms = fold_norms
        if fold_norms:
            fold_norm_weights(weights)
        self.kc = kcaches
        self.vc = vcaches
        self.max_M = max_M
        self.max_rows = max_rows
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.device = dev
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.x = torch.empty((max_M, dims.d), **bf)
        self.h = torch.empty((max_M, dims.d), **bf)
        self.qkv = torch.empty((max_M, dims.qkv), **bf)
        self.o = torch.empty((max_M, dims.Hq * dims.D), **bf)
        self.gu = None if self.fused_swiglu else torch.empty((max_M, 2 * dims.I), **bf)
        self.a = torch.empty((max_M, dims.I), **bf)
        self.cs = torch.empty((max_M, dims.D // 2, 2), dtype=torch.float32, device=dev)
        self.ssq = torch.empty((max_M, (dims.d + 127) // 128), dtype=torch.float32, device=dev)
        self.norm_in = S.row_norm(in_ssq=self.ssq, eps=dims.eps) if fold_norms else None
        self.norm_out = S.row_norm(out_ssq=self.ssq) if fold_norms else None
        self.P = torch.empty((max_M, dims.V), dtype=torch.float32, device=dev) if weights.w_lm is not None else None
        B, cap = (kcaches[0].shape[0], kcaches[0].shape[2]) if kcaches else (1, 1)
        need = 0
        for M in range(1, max_M + 1):
            for (n, k) in ((dims.qkv, dims.d), (dims.d, dims.Hq * dims.D), (2 * dims.I, dims.d),
                           (dims.d, dims.I)):
                need = max(need, S.spec_linear_workspace_bytes(M, n, k))
            if self.fused_swiglu:
                need = max(need, S.spec_swiglu_linear_workspace_bytes(M, dims.I, dims.d))
            if fold_norms:
                need = max(need, S.spec_linear_norm_workspace_bytes(M, dims.qkv, dims.d),
                           S.spec_linear_norm_workspace_bytes(M, 2 * dims.I, dims.d),
                           S.spec_linear_norm_workspace_bytes(M, dims.I, dims.d, swiglu=True))
        if kcaches:
            need = max(need, S.spec_attention_workspace_bytes(B, max_rows, dims.Hq, dims.Hkv, dims.D, cap))
        if weights.w_lm is not None:
            need = max(need, S.spec_lmhead_workspace_bytes(max_M, dims.d, dims.V))
            if fused_sampler:
                need = max(need, S.spec_lmhead_sample_workspace_bytes(max_M, dims.d, dims.V, 1.0))
        self.ws = S.Workspace(dev, need)
        self._graphs = []          # captured rounds (kept alive with the engine)

    # ------------------------------------------------------------------ one layer
    def layer(self, li: int, M: int, cu_rows, ctx_len, B: int, max_rows: int):
        dm, lw = self.dims, self.w.layers[li]
        x, h, qkv, o, a = (self.x[:M], self.h[:M], self.qkv[:M], self.o[:M], self.a[:M])
        hq = dm.Hq * dm.D
        hk = dm.Hkv * dm.D
        # the pre-norm input of the QKV and gate|up products: x itself when the norms are folded
        # (its sums of squares in self.ssq), else the RMSNorm kernel's output h
        nin, nout = self.norm_in, self.norm_out
        if not self.fold_norms:
            S.spec_rmsnorm(x, lw.attn_norm, dm.eps, Y=h)
        hin = x if self.fold_norms else h
        if self.fused_rope:
            S.spec_verify_linear_rope(hin, lw.w_qkv, self.cs[:M], dm.Hq + dm.Hkv, Y=qkv, ws=self.ws, norm=nin)
        else:
            S.spec_verify_linear(hin, lw.w_qkv, Y=qkv, ws=self.ws, norm=nin)
        q, k, v = qkv[:, :hq], qkv[:, hq:hq + hk], qkv[:, hq + hk:]
        if not self.fused_rope:
            S.spec_rope(q, k, cu_rows, ctx_len, dm.D, dm.theta)
        S.spec_verify_attention(q, k, v, cu_rows, ctx_len, self.kc[li], self.vc[li], max_rows, O=o,
                                ws=self.ws)
        S.spec_verify_linear(o, lw.w_o, Y=x, residual=x, ws=self.ws, norm=nout)
        if not self.fold_norms:
            S.spec_rmsnorm(x, lw.mlp_norm, dm.eps, Y=h)
        if self.fused_swiglu:
            S.spec_verify_linear_swiglu(hin, lw.w_gu, A=a, ws=self.ws, norm=nin)
        else:
            S.spec_verify_linear(hin, lw.w_gu, Y=self.gu[:M], ws=self.ws, norm=nin)
            S.spec_silu_mul(self.gu[:M], A=a)
        S.spec_verify_linear(a, lw.w_down, Y=x, residual=x, ws=self.ws, norm=nout)

    def _stack(self, x0, cu_rows, ctx_len, max_rows, n_layers, final_norm: bool = True):
        """All layers and (with final_norm) the final RMSNorm over the packed rows into self.h.  With
        folded norms and final_norm False, the LM head reads self.x with the sums of squares."""
        M = x0.shape[0]
        B = cu_rows.numel() - 1
        max_rows = self.max_rows if max_rows is None else max_rows
        if M > self.max_M:
            raise ValueError("more rows than the engine was sized for")
        if x0.data_ptr() != self.x.data_ptr():
            self.x[:M].copy_(x0)
        L = len(self.w.layers) if n_layers is None else n_layers
        if self.fused_rope and L > 0:
            S.spec_rope_table(cu_rows, ctx_len, M, self.dims.D, self.dims.theta, cs=self.cs[:M])
        if self.fold_norms and L > 0:
            S.spec_row_ssq(self.x[:M], out=self.ssq[:M])     # the first layer's input has no producer
        for li in range(L):
            self.layer(li, M, cu_rows, ctx_len, B, max_rows)
        if self.w.w_lm is not None and (final_norm or not self.fold_norms):
            S.spec_rmsnorm(self.x[:M], self.w.final_norm, self.dims.eps, Y=self.h[:M])
        return M

    def verify_pass(self, x0, cu_rows, ctx_len, temperature: float, max_rows: int | None = None,
                    n_layers: int | None = None):
        """All layers + LM head over the packed rows; returns P [M, V] (fp32 view)."""
        M = self._stack(x0, cu_rows, ctx_len, max_rows, n_layers)
        if self.w.w_lm is None:
            return None
        return S.spec_lmhead_softmax(self.h[:M], self.w.w_lm, temperature, P=self.P[:M], ws=self.ws)

    def verify_round(self, x0, cu_rows, ctx_len, q, drafts, U, temperature: float,
                     tie_eps: float = 1e-5, max_rows: int | None = None, out=None):
        """Verify pass + rejection sampler; returns (n_acc, out_tok, near_tie)."""
        if not self.fused_sampler:
            P = self.verify_pass(x0, cu_rows, ctx_len, temperature, max_rows)
            return S.spec_reject_sample(P, q, drafts, U, cu_rows, tie_eps, out=out)
        M = self._stack(x0, cu_rows, ctx_len, max_rows, None, final_norm=False)
        if self.fold_norms:
            if self.dims.layers == 0:
                S.spec_row_ssq(self.x[:M], out=self.ssq[:M])
            return S.spec_lmhead_reject_sample(self.x[:M], self.w.w_lm, temperature, q, drafts, U, cu_rows, tie_eps,
                                               out=out, ws=self.ws, norm=self.norm_in)
        return S.spec_lmhead_reject_sample(self.h[:M], self.w.w_lm, temperature, q, drafts, U, cu_rows, tie_eps,
                                           out=out, ws=self.ws)

    def capture_round(self, x0, cu_rows, ctx_len, q, drafts, U, temperature: float, out,
                      tie_eps: float = 1e-5, max_rows: int | None = None):
        """verify_round on these device buffers, captured once in a CUDA graph; returns the replay
        function.  A serving loop writes each round's inputs into the same buffers and replays:
        every launch of the round is re-issued with no per-launch host work.  M and B stay those
        of the capture; cu_rows, ctx_len, the tokens, q and U may change between rounds (the
        kernels read them from device memory).  The buffers must hold a valid round when this is
        called: the capture runs it twice.  The graph keeps the engine's workspace pointer, so that
        workspace must not be regrown afterwards (it is sized for every call the engine makes; give
        other calls their own)."""
        dev = self.device
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self.verify_round(x0, cu_rows, ctx_len, q, drafts, U, temperature, tie_eps, max_rows, out)
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            self.verify_round(x0, cu_rows, ctx_len, q, drafts, U, temperature, tie_eps, max_rows, out)
        torch.cuda.current_stream(dev).wait_stream(side)
        self._graphs.append(graph)
        return graph.replay


class DraftEngine:
    """The step before the verify pass: gamma autoregressive decode steps of a draft-shaped stack
    for B sequences at M = B rows ("Speculative Decoding Spends Arithmetic You May Not Have",
    Algorithm 1: the draft proposes x_1 .. x_gamma one at a time and keeps q_1 .. q_gamma).

    Step i: embedding rows of the current tokens (spec_embed; the LM head is tied to the
    embedding table), the stack at positions ctx_b + i (verify attention with one row per
    sequence writes that row's K/V into the draft cache), the LM head writing q_i straight into
    row b * gamma + i of the packed q that the verify sampler reads (spec_lmhead_softmax_ld),
    and the next token drawn from q_i (spec_sample_rows, uniform U[i, b]).  All arithmetic in
    the library's kernels; the engine only sequences the calls and advances positions.
    """

    def __init__(self, dims: Dims, weights: StackW, kcaches, vcaches, B: int, gamma: int, device=None):
        self.dims = dims
        self.B = B
        self.gamma = gamma
        # (the LM head is the embedding table here: its rows must stay unscaled, so no folded norms)
        self.eng = VerifyEngine(dims, weights, kcaches, vcaches, max_M=B, max_rows=1, device=device,
                                fused_sampler=False, fold_norms=False)
        dev = self.eng.device
        self.table = weights.w_lm
        self.cu = torch.arange(B + 1, dtype=torch.int32, device=dev)
        self.ctx = torch.empty((gamma, B), dtype=torch.int32, device=dev)
        self.step_tok = torch.empty((gamma + 1, B), dtype=torch.int32, device=dev)
        self.steps = torch.arange(gamma, dtype=torch.int32, device=dev)[:, None]

    def draft(self, tok0, ctx_len, U, temperature: float, Q, drafts):
        """tok0 [B] int32 (each sequence's last committed token), ctx_len [B] int32 (tokens in the
        draft cache), U [gamma, B] fp32; writes Q [B * gamma, V] fp32 (q rows, sequence-major) and
        drafts [B * gamma] int32 (sequence b's drafts at b * gamma ..)."""
        B, g, V = self.B, self.gamma, self.dims.V
        e = self.eng
        self.step_tok[0].copy_(tok0)
        torch.add(ctx_len[None, :], self.steps, out=self.ctx)     # positions ctx_b + i
        Qv = Q.view(B, g, V)
        for i in range(g):
            S.spec_embed(self.step_tok[i], self.table, X=e.x[:B])
            e._stack(e.x[:B], self.cu, self.ctx[i], 1, None)
            S.spec_lmhead_softmax(e.h[:B], self.table, temperature, P=Qv[:, i, :], ws=e.ws)
            S.spec_sample_rows(Qv[:, i, :], U[i], out=self.step_tok[i + 1])
        drafts.view(B, g).copy_(self.step_tok[1:].t())

