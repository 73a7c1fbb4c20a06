"""Python binding of ``libspecverify.so`` — argument marshalling only.

Every function here has the name of the C entry point it wraps.  It reads
shapes, strides and device pointers off torch tensors, passes them through
ctypes and raises :class:`SpecError` on a non-zero status.  All arithmetic
of the verify round runs in the library's CUDA kernels; torch only provides
device memory and the current stream.  If the library is missing the import
fails loudly: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SPEC_OK, SPEC_EINVAL, SPEC_EUNSUPPORTED, SPEC_ECUDA, SPEC_ETIMEOUT = range(5)

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "spec_last_error": (ctypes.c_char_p, []),
    "spec_version": (_i, []),
    "spec_launches": (_i, []),
    "spec_set_option": (_i, [ctypes.c_char_p, _i]),
    "spec_device_status": (_i, [_vp, ctypes.POINTER(_i)]),
    "spec_probe_bounded_wait": (_i, [_i, _i, _vp]),
    "spec_linear_workspace_bytes": (_sz, [_i, _i, _i]),
    "spec_verify_linear": (_i, [_vp, _i, _i, _i, _vp, _i, _i, _vp, _i, _vp, _i, _vp, _sz, _vp]),
    "spec_verify_linear_noalloc": (_i, [_vp, _i, _i, _i, _vp, _i, _i, _vp, _i, _vp, _i, _vp]),
    "spec_verify_linear_rope": (_i, [_vp, _i, _i, _i, _vp, _i, _i, _vp, _i, _vp, _i, _vp, _sz, _vp]),
    "spec_row_ssq": (_i, [_vp, _i, _i, _i, _vp, _vp]),
    "spec_linear_norm_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "spec_verify_linear_norm": (_i, [_vp, _i, _i, _i, _vp, _i, _i, _vp, _i, _vp, _i, _vp, _vp, _sz, _vp]),
    "spec_verify_linear_swiglu_norm": (_i, [_vp, _i, _i, _i, _vp, _i, _i, _vp, _i, _vp, _vp, _sz, _vp]),
    "spec_verify_linear_rope_norm": (_i, [_vp, _i, _i, _i, _vp, _i, _i, _vp, _i, _vp, _i, _vp, _vp, _sz, _vp]),
    "spec_lmhead_reject_sample_norm": (_i, [_vp, _i, _i, _vp, _i, _f, _vp, _vp, _vp, _vp, _i, _f, _vp, _vp, _vp,
                                            _vp, _vp, _sz, _vp]),
    "spec_linear_chain_workspace_bytes": (_sz, [_vp, _i, _i]),
    "spec_verify_linear_chain": (_i, [_vp, _i, _i, _vp, _sz, _vp]),
    "spec_rope_table": (_i, [_vp, _vp, _i, _i, _i, _f, _vp, _vp]),
    "spec_swiglu_linear_workspace_bytes": (_sz, [_i, _i, _i]),
    "spec_verify_linear_swiglu": (_i, [_vp, _i, _i, _i, _vp, _i, _i, _vp, _i, _vp, _sz, _vp]),
    "spec_attention_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "spec_verify_attention": (_i, [_vp, _i, _vp, _vp, _i, _vp, _vp, _i, _i, _vp, _vp, _i,
                                   _i, _i, _i, _f, _vp, _i, _vp, _sz, _vp]),
    "spec_attention_paged_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "spec_verify_attention_paged": (_i, [_vp, _i, _vp, _vp, _i, _vp, _vp, _i, _i, _vp, _vp, _i, _vp, _i,
                                         _i, _i, _i, _f, _vp, _i, _vp, _sz, _vp]),
    "spec_lmhead_workspace_bytes": (_sz, [_i, _i, _i]),
    "spec_lmhead_softmax": (_i, [_vp, _i, _i, _vp, _i, _f, _vp, _vp, _sz, _vp]),
    "spec_lmhead_softmax_ld": (_i, [_vp, _i, _i, _vp, _i, _f, _vp, ctypes.c_longlong, _vp, _sz, _vp]),
    "spec_embed": (_i, [_vp, _i, _vp, _i, _i, _i, _vp, _i, _vp]),
    "spec_reject_sample": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _f, _vp, _vp, _vp, _vp]),
    "spec_ngram_propose": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp]),
    "spec_sample_rows": (_i, [_vp, ctypes.c_longlong, _i, _i, _vp, _vp, _vp]),
    "spec_typical_sample": (_i, [_vp, _vp, _vp, _vp, _i, _i, _f, _f, _f, _vp, _vp, _vp, _vp]),
    "spec_lmhead_sample_workspace_bytes": (_sz, [_i, _i, _i, _f]),
    "spec_lmhead_reject_sample": (_i, [_vp, _i, _i, _vp, _i, _f, _vp, _vp, _vp, _vp, _i, _f, _vp, _vp, _vp,
                                       _vp, _sz, _vp]),
    "spec_rmsnorm": (_i, [_vp, _i, _i, _i, _vp, _f, _vp, _i, _vp]),
    "spec_rope": (_i, [_vp, _i, _i, _vp, _i, _i, _i, _vp, _vp, _i, _i, _f, _vp]),
    "spec_silu_mul": (_i, [_vp, _i, _i, _i, _vp, _i, _vp]),
}
EXPORTS = tuple(_SIGS)


class SpecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[spec code {code}] {msg}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library and declare every exported signature (no device work)."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(the verify path has no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = load()


def _check(rc: int, compute: bool = False) -> None:
    """Raise on an error code; after a compute call, add the kernels it enqueued."""
    global _launches
    if rc != SPEC_OK:
        raise SpecError(rc, _lib.spec_last_error().decode())
    if compute:
        _launches += _lib.spec_launches()


# Number of library kernels launched through this binding (for launch accounting).
_launches = 0


def reset_launch_count() -> None:
    global _launches
    _launches = 0


def launch_count() -> int:
    return _launches


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _rowmajor(t: torch.Tensor, name: str) -> int:
    """Leading dimension of a 2-D tensor whose rows are contiguous."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with contiguous rows")
    return t.stride(0)


def _need(t, dtype, name):
    if t.dtype != dtype or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA {dtype} tensor")


# --------------------------------------------------------------------------- misc
def spec_version() -> int:
    return _lib.spec_version()


def spec_set_option(name: str, value: int) -> None:
    _check(_lib.spec_set_option(name.encode(), int(value)))


def spec_device_status(stream=None) -> int:
    """Synchronize and read/clear the device status word (raises on a timeout)."""
    detail = ctypes.c_int(0)
    _check(_lib.spec_device_status(_stream(stream), ctypes.byref(detail)))
    return detail.value


def spec_device_status_code(stream=None) -> tuple[int, int]:
    """Like spec_device_status, but returns (status code, site detail) instead of raising on a
    device-side status (SPEC_ETIMEOUT / SPEC_EINVAL)."""
    detail = ctypes.c_int(0)
    rc = _lib.spec_device_status(_stream(stream), ctypes.byref(detail))
    if rc not in (SPEC_OK, SPEC_ETIMEOUT, SPEC_EINVAL):
        _check(rc)
    return rc, detail.value


PROBE_WAIT_SITE = 0x1E1


def spec_probe_bounded_wait(limit_us: int, arrive: bool = False, stream=None) -> None:
    """One bounded device wait that runs out after limit_us (arrive False) or completes."""
    _check(_lib.spec_probe_bounded_wait(int(limit_us), 1 if arrive else 0, _stream(stream)), compute=True)


class Workspace:
    """A zero-filled device buffer that grows on demand (plumbing for the kernels' scratch).

    One Workspace can serve every call issued on one stream: the library keeps
    its counters at zero between calls.
    """

    def __init__(self, device=None, nbytes: int = 0):
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.buf = None
        if nbytes:
            self.ensure(nbytes)

    def ensure(self, nbytes: int) -> "Workspace":
        if nbytes and (self.buf is None or self.buf.numel() < nbytes):
            self.buf = torch.zeros(int(nbytes), dtype=torch.uint8, device=self.device)
        return self

    def args(self):
        if self.buf is None:
            return None, 0
        return ctypes.c_void_p(self.buf.data_ptr()), self.buf.numel()


def _ws_args(ws: Workspace | None, need: int, device):
    if need == 0:
        return (ws.args() if ws is not None else (None, 0))
    if ws is None:
        ws = Workspace(device)
    ws.ensure(need)
    return ws.args()


# --------------------------------------------------------------------------- verify linear
def spec_linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return _lib.spec_linear_workspace_bytes(M, N, K)


class RowNorm(ctypes.Structure):
    """A folded RMSNorm (the C struct spec_rownorm): in_ssq [M, in_tiles] fp32 partial sums of
    squares of X's rows (X's rows are scaled by 1 / sqrt(sum / K + eps)), out_ssq [M, ceil(N/128)]
    fp32 filled with the sums of squares of the output as stored."""
    _fields_ = [("in_ssq", _vp), ("in_tiles", _i), ("eps", _f), ("out_ssq", _vp)]


def row_norm(in_ssq=None, eps: float = 1e-6, out_ssq=None) -> "RowNorm":
    for t, name in ((in_ssq, "in_ssq"), (out_ssq, "out_ssq")):
        if t is not None:
            _need(t, torch.float32, name)
            if not t.is_contiguous() or t.dim() != 2:
                raise ValueError(f"{name} must be a contiguous [M, tiles] tensor")
    nm = RowNorm(in_ssq.data_ptr() if in_ssq is not None else None,
                 in_ssq.shape[1] if in_ssq is not None else 0, float(eps),
                 out_ssq.data_ptr() if out_ssq is not None else None)
    nm.tensors = (in_ssq, out_ssq)
    return nm


def spec_row_ssq(X, out=None, stream=None):
    """out[M, ceil(N/128)] = per row and 128-column tile, the sum of squares of X's bf16 values."""
    _need(X, torch.bfloat16, "X")
    M, N = X.shape
    if out is None:
        out = torch.empty((M, (N + 127) // 128), dtype=torch.float32, device=X.device)
    _need(out, torch.float32, "out")
    _check(_lib.spec_row_ssq(_p(X), M, N, _rowmajor(X, "X"), _p(out), _stream(stream)), True)
    return out


def spec_linear_norm_workspace_bytes(M, N, K, swiglu: bool = False) -> int:
    return _lib.spec_linear_norm_workspace_bytes(M, N, K, 1 if swiglu else 0)


def spec_verify_linear(X, W, Y=None, residual=None, ws: Workspace | None = None, stream=None, norm=None):
    """Y[M, N] = X[M, K] @ W[N, K]^T (+ residual), bf16 in/out, fp32 accumulate (norm: a folded
    RMSNorm, see row_norm)."""
    _need(X, torch.bfloat16, "X"); _need(W, torch.bfloat16, "W")
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("W must be [N, K]")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    _need(Y, torch.bfloat16, "Y")
    if residual is not None:
        _need(residual, torch.bfloat16, "residual")
    if norm is not None:
        wp, wn = _ws_args(ws, spec_linear_norm_workspace_bytes(M, N, K), X.device)
        _check(_lib.spec_verify_linear_norm(
            _p(X), M, K, _rowmajor(X, "X"), _p(W), N, _rowmajor(W, "W"), _p(Y), _rowmajor(Y, "Y"),
            _p(residual), _rowmajor(residual, "residual") if residual is not None else 0,
            ctypes.byref(norm), wp, wn, _stream(stream)), True)
        return Y
    wp, wn = _ws_args(ws, spec_linear_workspace_bytes(M, N, K), X.device)
    _check(_lib.spec_verify_linear(
        _p(X), M, K, _rowmajor(X, "X"), _p(W), N, _rowmajor(W, "W"), _p(Y), _rowmajor(Y, "Y"),
        _p(residual), _rowmajor(residual, "residual") if residual is not None else 0,
        wp, wn, _stream(stream)), True)
    return Y


def spec_verify_linear_noalloc(X, W, Y, residual=None, stream=None):
    """Same product as spec_verify_linear, for callers that cannot allocate.

    Y must be given (nothing is allocated here either); split-K scratch comes
    from the library's static device array (see the header for the limit).
    """
    _need(X, torch.bfloat16, "X"); _need(W, torch.bfloat16, "W"); _need(Y, torch.bfloat16, "Y")
    M, K = X.shape
    N = W.shape[0]
    if residual is not None:
        _need(residual, torch.bfloat16, "residual")
    _check(_lib.spec_verify_linear_noalloc(
        _p(X), M, K, _rowmajor(X, "X"), _p(W), N, _rowmajor(W, "W"), _p(Y), _rowmajor(Y, "Y"),
        _p(residual), _rowmajor(residual, "residual") if residual is not None else 0,
        _stream(stream)), True)
    return Y


class LinearOp(ctypes.Structure):
    """One product of spec_verify_linear_chain (the C struct spec_linear_op)."""
    _fields_ = [("X", _vp), ("ldx", _i), ("W", _vp), ("ldw", _i), ("Y", _vp), ("ldy", _i),
                ("residual", _vp), ("ldr", _i), ("N", _i), ("K", _i), ("swiglu", _i)]


def linear_op(X, W, Y, residual=None, swiglu: bool = False) -> "LinearOp":
    """Describe Y = X W^T (+ residual), or the fused SwiGLU form (W gate|up interleaved, Y = A)."""
    for t, name in ((X, "X"), (W, "W"), (Y, "Y")):
        _need(t, torch.bfloat16, name)
    if residual is not None:
        _need(residual, torch.bfloat16, "residual")
    N, K = W.shape
    if X.shape[1] != K or Y.shape[0] != X.shape[0] or Y.shape[1] != (N // 2 if swiglu else N):
        raise ValueError("shapes of X, W and Y do not match")
    op = LinearOp(X.data_ptr(), _rowmajor(X, "X"), W.data_ptr(), _rowmajor(W, "W"), Y.data_ptr(),
                  _rowmajor(Y, "Y"), residual.data_ptr() if residual is not None else None,
                  _rowmajor(residual, "residual") if residual is not None else 0, N, K, 1 if swiglu else 0)
    op.tensors = (X, W, Y, residual)    # the struct holds raw pointers: keep their memory alive with it
    return op


def _op_array(ops):
    arr = (LinearOp * len(ops))()
    for i, o in enumerate(ops):
        arr[i] = o
    return arr


def spec_linear_chain_workspace_bytes(ops, M: int) -> int:
    return int(_lib.spec_linear_chain_workspace_bytes(_op_array(ops), len(ops), int(M)))


def spec_verify_linear_chain(ops, M: int, ws=None, stream=None, device=None) -> None:
    """Run the products `ops` (a list of linear_op(...)) over M rows in one weight stream."""
    arr = _op_array(ops)
    need = int(_lib.spec_linear_chain_workspace_bytes(arr, len(ops), int(M)))
    wp, wn = _ws_args(ws, need, device if device is not None else torch.cuda.current_device())
    _check(_lib.spec_verify_linear_chain(arr, len(ops), int(M), wp, wn, _stream(stream)), True)


def spec_rope_table(cu_rows, ctx_len, M: int, D: int, theta: float = 1e6, cs=None, stream=None):
    """(cos, sin) per verify row and frequency: cs [M, D/2, 2] fp32."""
    _need(cu_rows, torch.int32, "cu_rows"); _need(ctx_len, torch.int32, "ctx_len")
    B = cu_rows.numel() - 1
    if cs is None:
        cs = torch.empty((M, D // 2, 2), dtype=torch.float32, device=cu_rows.device)
    _need(cs, torch.float32, "cs")
    if not cs.is_contiguous():
        raise ValueError("cs must be contiguous")
    _check(_lib.spec_rope_table(_p(cu_rows), _p(ctx_len), B, M, D, float(theta), _p(cs), _stream(stream)), True)
    return cs


def spec_verify_linear_rope(X, W, cs, rope_heads: int, Y=None, ws: Workspace | None = None, stream=None,
                            norm=None):
    """Y = X W^T with the first rope_heads 128-column heads rotated by the table cs [M, 64, 2]."""
    _need(X, torch.bfloat16, "X"); _need(W, torch.bfloat16, "W"); _need(cs, torch.float32, "cs")
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("W must be [N, K]")
    if not cs.is_contiguous() or cs.shape[0] < M:
        raise ValueError("cs must be a contiguous table with a row per verify row")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    _need(Y, torch.bfloat16, "Y")
    if norm is not None:
        wp, wn = _ws_args(ws, spec_linear_norm_workspace_bytes(M, N, K), X.device)
        _check(_lib.spec_verify_linear_rope_norm(_p(X), M, K, _rowmajor(X, "X"), _p(W), N, _rowmajor(W, "W"), _p(Y),
                                                 _rowmajor(Y, "Y"), _p(cs), int(rope_heads), ctypes.byref(norm), wp,
                                                 wn, _stream(stream)), True)
        return Y
    wp, wn = _ws_args(ws, spec_linear_workspace_bytes(M, N, K), X.device)
    _check(_lib.spec_verify_linear_rope(_p(X), M, K, _rowmajor(X, "X"), _p(W), N, _rowmajor(W, "W"), _p(Y),
                                        _rowmajor(Y, "Y"), _p(cs), int(rope_heads), wp, wn, _stream(stream)), True)
    return Y


def spec_swiglu_linear_workspace_bytes(M, I, K) -> int:
    return _lib.spec_swiglu_linear_workspace_bytes(M, I, K)


GATE_UP_BLOCK = 16   # rows per gate / up block in the interleaved layout


def interleave_gate_up(Wg, Wu):
    """Weight layout of spec_verify_linear_swiglu: gate and up rows in alternating blocks of 16.

    A one-time relayout of the model's weights (a copy), not part of a verify pass.
    """
    I, K = Wg.shape
    b = GATE_UP_BLOCK
    if Wu.shape != (I, K) or I % 64:
        raise ValueError("Wg and Wu must both be [I, K] with I % 64 == 0")
    return torch.stack((Wg.reshape(I // b, b, K), Wu.reshape(I // b, b, K)), dim=1).reshape(2 * I, K).contiguous()


def spec_verify_linear_swiglu(X, Wgu, A=None, ws: Workspace | None = None, stream=None, norm=None):
    """A[M, I] = silu(X Wg^T) * (X Wu^T), Wgu = interleave_gate_up(Wg, Wu) of shape [2I, K]."""
    _need(X, torch.bfloat16, "X"); _need(Wgu, torch.bfloat16, "Wgu")
    M, K = X.shape
    N2 = Wgu.shape[0]
    if Wgu.shape[1] != K or N2 % 128:
        raise ValueError("Wgu must be [2I, K] with I % 64 == 0")
    inter = N2 // 2
    if A is None:
        A = torch.empty((M, inter), dtype=torch.bfloat16, device=X.device)
    _need(A, torch.bfloat16, "A")
    if norm is not None:
        wp, wn = _ws_args(ws, spec_linear_norm_workspace_bytes(M, inter, K, swiglu=True), X.device)
        _check(_lib.spec_verify_linear_swiglu_norm(
            _p(X), M, K, _rowmajor(X, "X"), _p(Wgu), _rowmajor(Wgu, "Wgu"), inter,
            _p(A), _rowmajor(A, "A"), ctypes.byref(norm), wp, wn, _stream(stream)), True)
        return A
    wp, wn = _ws_args(ws, spec_swiglu_linear_workspace_bytes(M, inter, K), X.device)
    _check(_lib.spec_verify_linear_swiglu(
        _p(X), M, K, _rowmajor(X, "X"), _p(Wgu), _rowmajor(Wgu, "Wgu"), inter,
        _p(A), _rowmajor(A, "A"), wp, wn, _stream(stream)), True)
    return A


# --------------------------------------------------------------------------- attention
def spec_attention_workspace_bytes(B, max_rows, Hq, Hkv, D, cap) -> int:
    return _lib.spec_attention_workspace_bytes(B, max_rows, Hq, Hkv, D, cap)


def spec_verify_attention(Q, Knew, Vnew, cu_rows, ctx_len, Kcache, Vcache, max_rows: int,
                          scale: float | None = None, O=None, ws: Workspace | None = None,
                          stream=None):
    """Causal GQA verify attention; appends Knew/Vnew to the cache at ctx_len.

    Q [M, Hq*D] and Knew/Vnew [M, Hkv*D] are 2-D (possibly strided column
    slices of a fused QKV output); Kcache/Vcache [B, Hkv, cap, D].
    """
    for t, n in ((Q, "Q"), (Knew, "Knew"), (Vnew, "Vnew"), (Kcache, "Kcache"), (Vcache, "Vcache")):
        _need(t, torch.bfloat16, n)
    _need(cu_rows, torch.int32, "cu_rows"); _need(ctx_len, torch.int32, "ctx_len")
    B, Hkv, cap, D = Kcache.shape
    if not (Kcache.is_contiguous() and Vcache.is_contiguous() and Vcache.shape == Kcache.shape):
        raise ValueError("Kcache/Vcache must be contiguous [B, Hkv, cap, D]")
    M = Q.shape[0]
    Hq = Q.shape[1] // D
    ldkv = _rowmajor(Knew, "Knew")
    if _rowmajor(Vnew, "Vnew") != ldkv:
        raise ValueError("Knew and Vnew must share a leading dimension")
    if O is None:
        O = torch.empty((M, Hq * D), dtype=torch.bfloat16, device=Q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    wp, wn = _ws_args(ws, spec_attention_workspace_bytes(B, max_rows, Hq, Hkv, D, cap), Q.device)
    _check(_lib.spec_verify_attention(
        _p(Q), _rowmajor(Q, "Q"), _p(Knew), _p(Vnew), ldkv, _p(cu_rows), _p(ctx_len), B,
        int(max_rows), _p(Kcache), _p(Vcache), cap, Hq, Hkv, D, float(scale), _p(O),
        _rowmajor(O, "O"), wp, wn, _stream(stream)), True)
    return O


def spec_attention_paged_workspace_bytes(B, max_rows, Hq, Hkv, D, max_pages) -> int:
    return _lib.spec_attention_paged_workspace_bytes(B, max_rows, Hq, Hkv, D, max_pages)


def spec_verify_attention_paged(Q, Knew, Vnew, cu_rows, ctx_len, Kpool, Vpool, block_table, max_rows: int,
                                scale: float | None = None, O=None, ws: Workspace | None = None, stream=None):
    """Verify attention over a paged cache: Kpool/Vpool [Hkv, num_pages, 128, D], block_table
    [B, max_pages] int32 (page of each 128-key block of each sequence)."""
    for t, n in ((Q, "Q"), (Knew, "Knew"), (Vnew, "Vnew"), (Kpool, "Kpool"), (Vpool, "Vpool")):
        _need(t, torch.bfloat16, n)
    _need(cu_rows, torch.int32, "cu_rows"); _need(ctx_len, torch.int32, "ctx_len")
    _need(block_table, torch.int32, "block_table")
    Hkv, num_pages, page, D = Kpool.shape
    if page != 128 or not (Kpool.is_contiguous() and Vpool.is_contiguous() and Vpool.shape == Kpool.shape):
        raise ValueError("Kpool/Vpool must be contiguous [Hkv, num_pages, 128, D]")
    if not block_table.is_contiguous() or block_table.dim() != 2:
        raise ValueError("block_table must be a contiguous [B, max_pages] tensor")
    B, max_pages = block_table.shape
    M = Q.shape[0]
    Hq = Q.shape[1] // D
    ldkv = _rowmajor(Knew, "Knew")
    if _rowmajor(Vnew, "Vnew") != ldkv:
        raise ValueError("Knew and Vnew must share a leading dimension")
    if O is None:
        O = torch.empty((M, Hq * D), dtype=torch.bfloat16, device=Q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    wp, wn = _ws_args(ws, spec_attention_paged_workspace_bytes(B, max_rows, Hq, Hkv, D, max_pages), Q.device)
    _check(_lib.spec_verify_attention_paged(
        _p(Q), _rowmajor(Q, "Q"), _p(Knew), _p(Vnew), ldkv, _p(cu_rows), _p(ctx_len), B, int(max_rows),
        _p(Kpool), _p(Vpool), num_pages, _p(block_table), max_pages, Hq, Hkv, D, float(scale), _p(O),
        _rowmajor(O, "O"), wp, wn, _stream(stream)), True)
    return O


# --------------------------------------------------------------------------- LM head
def spec_lmhead_workspace_bytes(M, K, V) -> int:
    return _lib.spec_lmhead_workspace_bytes(M, K, V)


def spec_lmhead_softmax(H, Wlm, temperature: float, P=None, ws: Workspace | None = None, stream=None):
    """P[M, V] = softmax(H @ Wlm^T / T) in fp32; T == 0 gives one-hot argmax rows."""
    _need(H, torch.bfloat16, "H"); _need(Wlm, torch.bfloat16, "Wlm")
    M, K = H.shape
    V = Wlm.shape[0]
    if not (H.is_contiguous() and Wlm.is_contiguous()):
        raise ValueError("H and Wlm must be contiguous")
    if P is None:
        P = torch.empty((M, V), dtype=torch.float32, device=H.device)
    _need(P, torch.float32, "P")
    if P.shape != (M, V) or P.stride(1) != 1:
        raise ValueError("P must be [M, V] with unit column stride")
    wp, wn = _ws_args(ws, spec_lmhead_workspace_bytes(M, K, V), H.device)
    if P.stride(0) == V:
        _check(_lib.spec_lmhead_softmax(_p(H), M, K, _p(Wlm), V, float(temperature), _p(P), wp, wn,
                                        _stream(stream)), True)
    else:   # rows of a larger array (e.g. one decode step's rows of a packed q)
        _check(_lib.spec_lmhead_softmax_ld(_p(H), M, K, _p(Wlm), V, float(temperature), _p(P), P.stride(0),
                                           wp, wn, _stream(stream)), True)
    return P


def spec_embed(ids, table, X=None, stream=None):
    """X[r] = table[ids[r]] (bf16 rows)."""
    _need(ids, torch.int32, "ids"); _need(table, torch.bfloat16, "table")
    M = ids.numel()
    V, d = table.shape
    if X is None:
        X = torch.empty((M, d), dtype=torch.bfloat16, device=table.device)
    _need(X, torch.bfloat16, "X")
    if not ids.is_contiguous():
        raise ValueError("ids must be contiguous")
    _check(_lib.spec_embed(_p(ids), M, _p(table), V, d, _rowmajor(table, "table"), _p(X), _rowmajor(X, "X"),
                           _stream(stream)), True)
    return X


# --------------------------------------------------------------------------- sampler
def spec_reject_sample(P, Q, draft_tok, U, cu_rows, tie_eps: float = 1e-5, out=None, stream=None):
    """Returns (n_acc [B], out_tok [M], near_tie [B]) int32 device tensors."""
    _need(P, torch.float32, "P"); _need(Q, torch.float32, "Q"); _need(U, torch.float32, "U")
    _need(draft_tok, torch.int32, "draft_tok"); _need(cu_rows, torch.int32, "cu_rows")
    M, V = P.shape
    B = cu_rows.numel() - 1
    if out is None:
        dev = P.device
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(M, dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev))
    n_acc, out_tok, near = out
    for t in (P, Q, U, draft_tok, cu_rows):
        if not t.is_contiguous():
            raise ValueError("sampler inputs must be contiguous")
    _check(_lib.spec_reject_sample(_p(P), _p(Q), _p(draft_tok), _p(U), _p(cu_rows), B, V,
                                   float(tie_eps), _p(n_acc), _p(out_tok), _p(near), _stream(stream)), True)
    return n_acc, out_tok, near


def spec_ngram_propose(tokens, cu_len, k: int, n_min: int, n_max: int, out=None, stream=None):
    """n-gram prompt lookup; returns (drafts [B, k] (-1 padded), n_drafts [B]) int32 device tensors."""
    _need(tokens, torch.int32, "tokens"); _need(cu_len, torch.int32, "cu_len")
    if not (tokens.is_contiguous() and cu_len.is_contiguous()):
        raise ValueError("tokens and cu_len must be contiguous")
    B = cu_len.numel() - 1
    if out is None:
        out = (torch.empty((B, k), dtype=torch.int32, device=tokens.device),
               torch.empty(B, dtype=torch.int32, device=tokens.device))
    drafts, n = out
    _check(_lib.spec_ngram_propose(_p(tokens), _p(cu_len), B, int(k), int(n_min), int(n_max), _p(drafts), _p(n),
                                   _stream(stream)), True)
    return drafts, n


def spec_sample_rows(P, U, out=None, stream=None):
    """One token per row of P [M, V] (rows may be strided) drawn with U [M]; returns out [M] int32."""
    _need(P, torch.float32, "P"); _need(U, torch.float32, "U")
    M, V = P.shape
    if out is None:
        out = torch.empty(M, dtype=torch.int32, device=P.device)
    _check(_lib.spec_sample_rows(_p(P), _rowmajor(P, "P"), M, V, _p(U), _p(out), _stream(stream)), True)
    return out


def spec_typical_sample(P, draft_tok, U, cu_rows, epsilon: float, delta: float, tie_eps: float = 1e-5, out=None,
                        stream=None):
    """Typical acceptance; returns (n_acc [B], out_tok [M], near_tie [B]) int32 device tensors."""
    _need(P, torch.float32, "P"); _need(U, torch.float32, "U")
    _need(draft_tok, torch.int32, "draft_tok"); _need(cu_rows, torch.int32, "cu_rows")
    M, V = P.shape
    B = cu_rows.numel() - 1
    if out is None:
        dev = P.device
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(M, dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev))
    n_acc, out_tok, near = out
    for t in (P, U, draft_tok, cu_rows):
        if not t.is_contiguous():
            raise ValueError("sampler inputs must be contiguous")
    _check(_lib.spec_typical_sample(_p(P), _p(draft_tok), _p(U), _p(cu_rows), B, V, float(epsilon), float(delta),
                                    float(tie_eps), _p(n_acc), _p(out_tok), _p(near), _stream(stream)), True)
    return n_acc, out_tok, near


def spec_lmhead_sample_workspace_bytes(M, K, V, temperature) -> int:
    return _lib.spec_lmhead_sample_workspace_bytes(M, K, V, float(temperature))


def spec_lmhead_reject_sample(H, W_lm, temperature: float, Q, draft_tok, U, cu_rows, tie_eps: float = 1e-5,
                              out=None, ws: Workspace | None = None, stream=None, norm=None):
    """Fused LM head -> sampler; returns (n_acc [B], out_tok [M], near_tie [B]) int32 device tensors."""
    _need(H, torch.bfloat16, "H"); _need(W_lm, torch.bfloat16, "W_lm")
    _need(Q, torch.float32, "Q"); _need(U, torch.float32, "U")
    _need(draft_tok, torch.int32, "draft_tok"); _need(cu_rows, torch.int32, "cu_rows")
    M, K = H.shape
    V = W_lm.shape[0]
    if W_lm.shape[1] != K:
        raise ValueError("W_lm must be [V, K]")
    for t in (H, W_lm, Q, U, draft_tok, cu_rows):
        if not t.is_contiguous():
            raise ValueError("fused sampler inputs must be contiguous")
    B = cu_rows.numel() - 1
    if out is None:
        dev = H.device
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(M, dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev))
    n_acc, out_tok, near = out
    wp, wn = _ws_args(ws, spec_lmhead_sample_workspace_bytes(M, K, V, temperature), H.device)
    if norm is not None:
        _check(_lib.spec_lmhead_reject_sample_norm(_p(H), M, K, _p(W_lm), V, float(temperature), _p(Q),
                                                   _p(draft_tok), _p(U), _p(cu_rows), B, float(tie_eps), _p(n_acc),
                                                   _p(out_tok), _p(near), ctypes.byref(norm), wp, wn,
                                                   _stream(stream)), True)
        return n_acc, out_tok, near
    _check(_lib.spec_lmhead_reject_sample(_p(H), M, K, _p(W_lm), V, float(temperature), _p(Q), _p(draft_tok),
                                          _p(U), _p(cu_rows), B, float(tie_eps), _p(n_acc), _p(out_tok),
                                          _p(near), wp, wn, _stream(stream)), True)
    return n_acc, out_tok, near


# --------------------------------------------------------------------------- glue
def spec_rmsnorm(X, w, eps: float = 1e-6, Y=None, stream=None):
    _need(X, torch.bfloat16, "X"); _need(w, torch.bfloat16, "w")
    M, N = X.shape
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    _check(_lib.spec_rmsnorm(_p(X), M, N, _rowmajor(X, "X"), _p(w), float(eps), _p(Y),
                             _rowmajor(Y, "Y"), _stream(stream)), True)
    return Y


def spec_rope(Q, K, cu_rows, ctx_len, D: int, theta: float = 1e6, stream=None):
    """In-place RoPE on Q [M, Hq*D] and K [M, Hkv*D] (2-D, contiguous rows)."""
    _need(Q, torch.bfloat16, "Q"); _need(K, torch.bfloat16, "K")
    M = Q.shape[0]
    B = cu_rows.numel() - 1
    _check(_lib.spec_rope(_p(Q), _rowmajor(Q, "Q"), Q.shape[1] // D, _p(K), _rowmajor(K, "K"),
                          K.shape[1] // D, D, _p(cu_rows), _p(ctx_len), B, M, float(theta),
                          _stream(stream)), True)


def spec_silu_mul(GU, A=None, stream=None):
    """A[M, I] = silu(GU[:, :I]) * GU[:, I:2I]."""
    _need(GU, torch.bfloat16, "GU")
    M, two_i = GU.shape
    inter = two_i // 2
    if A is None:
        A = torch.empty((M, inter), dtype=torch.bfloat16, device=GU.device)
    _check(_lib.spec_silu_mul(_p(GU), M, inter, _rowmajor(GU, "GU"), _p(A), _rowmajor(A, "A"),
                              _stream(stream)), True)
    return A
