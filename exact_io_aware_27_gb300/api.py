"""ctypes binding of the C-ABI in ``include/fa.h`` (argument marshalling only).

Every function here checks the Python-side arguments, allocates outputs with
torch when the caller passes none, and calls the library function of the same
name on the current torch CUDA stream. All attention arithmetic runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback: if the library
is missing, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import _build

LIBRARY = _build.LIBRARY

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED_HEAD_DIM = -2
FA_ERR_MISALIGNED = -3
FA_ERR_UNSUPPORTED_DEVICE = -4
FA_ERR_WORKSPACE_TOO_SMALL = -5
FA_ERR_CUDA = -6
FA_ERR_DEVICE_TIMEOUT = -7

# Every entry point of include/fa.h and include/fa_selftest.h with its ctypes
# signature: (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_S = ctypes.c_size_t
SIGNATURES = {
    "fa_forward": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "fa_backward_workspace_size": (_S, [_I, _I, _I, _I, _I]),
    "fa_backward": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P,
                         _S, _P]),
    "fa_backward_preprocess": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _S, _P]),
    "fa_backward_dkdv": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _S, _P]),
    "fa_backward_dq": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _S, _P]),
    "fa_backward_grads": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _S,
                               _P]),
    "fa_backward_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                                 _P, _P]),
    "fa_online_softmax_stats": (_I, [_P, ctypes.c_longlong, ctypes.c_longlong, _P, _P, _P]),
    "fa_standard_matrix_bytes": (_S, [_I, _I, _I, _I]),
    "fa_standard_forward": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P]),
    "fa_session_create": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_P)]),
    "fa_session_destroy": (None, [_P]),
    "fa_session_step": (_I, [_P, _P, _P, _P, _P, _I, _F, _P, _P, _P, _P, _P]),
    "fa_session_submit": (_I, [_P, _P, _P, _P, _P, _I, _F, _P, _P, _P, _P, _P]),
    "fa_session_sync": (_I, [_P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_get_device_status": (_I, [ctypes.POINTER(_I)]),
    "fa_version": (_I, []),
    "fa_selftest_mma": (_I, [_I, _P, _P, _P, _P]),
    "fa_selftest_wait_timeout": (_I, [ctypes.c_longlong, _P, _P]),
}

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    """A negative status returned by the library."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """The loaded library. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIBRARY):
                raise RuntimeError(
                    f"CUDA library {LIBRARY} is not built; run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            handle = ctypes.CDLL(LIBRARY)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def version() -> int:
    return int(lib().fa_version())


def _check(fn: str, rc: int) -> None:
    if rc != FA_OK:
        raise FAError(fn, rc)


def _stream(t: torch.Tensor, stream) -> int:
    if stream is None:
        return torch.cuda.current_stream(t.device).cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _bf16_4d(name, t):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 4-D bf16 CUDA tensor [B,H,seq,d]")


def _scale(scale, d):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def _same_device(*ts):
    dev = ts[0].device
    for t in ts[1:]:
        if t.device != dev:
            raise ValueError("all tensors of a call must be on the same device")


def _out(name, t, shape, dtype, device):
    """A tensor the library writes through its pointer (a caller-provided output):
    its shape, dtype, device and layout must match exactly, since the library only
    sees the address."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if (tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device
            or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape "
                         f"{tuple(shape)} on {device}")
    return t


def _lse(L, B, H, n, device):
    """The forward's L as an input: fp32 [B,H,n] on the inputs' device."""
    if (not isinstance(L, torch.Tensor) or L.dtype != torch.float32
            or tuple(L.shape) != (B, H, n) or not L.is_contiguous() or L.device != device):
        raise ValueError("L must be a contiguous fp32 [B,H,n] tensor on the inputs' device")


def _workspace_bytes(ws, device):
    if (not isinstance(ws, torch.Tensor) or not ws.is_contiguous() or ws.device != device):
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    return ws.numel() * ws.element_size()


def _attention_inputs(Q, K, V, *more):
    """Checks Q [B,H,n,d], K and V [B,H,m,d] and any further [B,H,n,d] tensors
    (O, dO); returns (B, H, n, m, d)."""
    for name, t in (("Q", Q), ("K", K), ("V", V)) + tuple(more):
        _bf16_4d(name, t)
    B, H, n, d = Q.shape
    m = K.shape[2]
    if tuple(K.shape) != (B, H, m, d) or tuple(V.shape) != (B, H, m, d):
        raise ValueError("K and V must be [B,H,m,d] with Q's B, H and d")
    for name, t in more:
        if tuple(t.shape) != (B, H, n, d):
            raise ValueError(f"{name} must have Q's shape [B,H,n,d]")
    _same_device(Q, K, V, *(t for _, t in more))
    return B, H, n, m, d


def fa_forward(Q, K, V, causal: bool = False, scale: float | None = None, O=None, L=None,
               stream=None):
    """O [B,H,n,d] bf16 and L [B,H,n] fp32 (natural-log logsumexp)."""
    B, H, n, m, d = _attention_inputs(Q, K, V)
    if O is None:
        O = torch.empty_like(Q)
    if L is None:
        L = torch.empty((B, H, n), dtype=torch.float32, device=Q.device)
    _out("O", O, (B, H, n, d), torch.bfloat16, Q.device)
    _out("L", L, (B, H, n), torch.float32, Q.device)
    rc = lib().fa_forward(Q.data_ptr(), K.data_ptr(), V.data_ptr(), B, H, n, m, d,
                          int(bool(causal)), _scale(scale, d), O.data_ptr(), L.data_ptr(),
                          _stream(Q, stream))
    _check("fa_forward", rc)
    return O, L


def fa_standard_matrix_bytes(B: int, H: int, n: int, m: int) -> int:
    """Bytes of one of the S, P matrices of fa_standard_forward (bf16 [B,H,n,m_pad])."""
    return int(lib().fa_standard_matrix_bytes(B, H, n, m))


def fa_standard_forward(Q, K, V, causal: bool = False, scale: float | None = None, S=None,
                        P=None, O=None, L=None, stream=None):
    """Materialised standard attention: (O, L, S, P) with S = scale Q K^T and
    P = softmax(S) as bf16 [B,H,n,m_pad] matrices in device memory (m_pad = m
    rounded up to 64; the columns past m are 0)."""
    B, H, n, m, d = _attention_inputs(Q, K, V)
    m_pad = (m + 63) // 64 * 64
    if S is None:
        S = torch.empty((B, H, n, m_pad), dtype=torch.bfloat16, device=Q.device)
    if P is None:
        P = torch.empty((B, H, n, m_pad), dtype=torch.bfloat16, device=Q.device)
    if O is None:
        O = torch.empty_like(Q)
    if L is None:
        L = torch.empty((B, H, n), dtype=torch.float32, device=Q.device)
    _out("S", S, (B, H, n, m_pad), torch.bfloat16, Q.device)
    _out("P", P, (B, H, n, m_pad), torch.bfloat16, Q.device)
    _out("O", O, (B, H, n, d), torch.bfloat16, Q.device)
    _out("L", L, (B, H, n), torch.float32, Q.device)
    rc = lib().fa_standard_forward(Q.data_ptr(), K.data_ptr(), V.data_ptr(), B, H, n, m, d,
                                   int(bool(causal)), _scale(scale, d), S.data_ptr(), P.data_ptr(),
                                   O.data_ptr(), L.data_ptr(), _stream(Q, stream))
    _check("fa_standard_forward", rc)
    return O, L, S, P


def fa_backward_workspace_size(B: int, H: int, n: int, m: int, d: int) -> int:
    return int(lib().fa_backward_workspace_size(B, H, n, m, d))


def alloc_workspace(B, H, n, m, d, device) -> torch.Tensor:
    size = fa_backward_workspace_size(B, H, n, m, d)
    if size == 0:
        raise ValueError("invalid sizes for the backward workspace")
    return torch.empty(size, dtype=torch.uint8, device=device)


def fa_backward(Q, K, V, O, L, dO, causal: bool = False, scale: float | None = None, dQ=None,
                dK=None, dV=None, workspace=None, stream=None):
    """dQ, dK, dV (bf16) for upstream gradient dO, given the forward's O and L."""
    B, H, n, m, d = _attention_inputs(Q, K, V, ("O", O), ("dO", dO))
    _lse(L, B, H, n, Q.device)
    dQ, dK, dV = _grad_outputs(Q, K, V, dQ, dK, dV)
    if workspace is None:
        workspace = alloc_workspace(B, H, n, m, d, Q.device)
    ws_bytes = _workspace_bytes(workspace, Q.device)
    rc = lib().fa_backward(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), L.data_ptr(),
                           dO.data_ptr(), B, H, n, m, d, int(bool(causal)), _scale(scale, d),
                           dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), workspace.data_ptr(),
                           ws_bytes, _stream(Q, stream))
    _check("fa_backward", rc)
    return dQ, dK, dV


def _grad_outputs(Q, K, V, dQ, dK, dV):
    """dQ, dK, dV: allocated like Q, K, V when not given, else checked against them."""
    dQ = torch.empty_like(Q) if dQ is None else _out("dQ", dQ, Q.shape, torch.bfloat16, Q.device)
    dK = torch.empty_like(K) if dK is None else _out("dK", dK, K.shape, torch.bfloat16, K.device)
    dV = torch.empty_like(V) if dV is None else _out("dV", dV, V.shape, torch.bfloat16, V.device)
    return dQ, dK, dV


NOALLOC_WORKSPACE_BYTES = 1024 * 1024


def fa_backward_noalloc(Q, K, V, O, L, dO, causal: bool = False, scale: float | None = None,
                        dQ=None, dK=None, dV=None, stream=None):
    """fa_backward using the library's static device workspace instead of a
    caller buffer (for callers that cannot allocate device memory; limited to
    problems whose workspace fits in NOALLOC_WORKSPACE_BYTES). Outputs are
    allocated here only when not given."""
    B, H, n, m, d = _attention_inputs(Q, K, V, ("O", O), ("dO", dO))
    _lse(L, B, H, n, Q.device)
    dQ, dK, dV = _grad_outputs(Q, K, V, dQ, dK, dV)
    rc = lib().fa_backward_noalloc(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                                   L.data_ptr(), dO.data_ptr(), B, H, n, m, d,
                                   int(bool(causal)), _scale(scale, d), dQ.data_ptr(),
                                   dK.data_ptr(), dV.data_ptr(), _stream(Q, stream))
    _check("fa_backward_noalloc", rc)
    return dQ, dK, dV


def fa_backward_preprocess(O, dO, L, workspace, stream=None):
    for name, t in (("O", O), ("dO", dO)):
        _bf16_4d(name, t)
    if tuple(dO.shape) != tuple(O.shape):
        raise ValueError("dO must have O's shape [B,H,n,d]")
    _same_device(O, dO)
    B, H, n, d = O.shape
    _lse(L, B, H, n, O.device)
    rc = lib().fa_backward_preprocess(O.data_ptr(), dO.data_ptr(), L.data_ptr(), B, H, n, d,
                                      workspace.data_ptr(), _workspace_bytes(workspace, O.device),
                                      _stream(O, stream))
    _check("fa_backward_preprocess", rc)


def fa_backward_dkdv(Q, K, V, dO, workspace, causal=False, scale=None, dK=None, dV=None,
                     stream=None):
    B, H, n, m, d = _attention_inputs(Q, K, V, ("dO", dO))
    dK = torch.empty_like(K) if dK is None else _out("dK", dK, K.shape, torch.bfloat16, K.device)
    dV = torch.empty_like(V) if dV is None else _out("dV", dV, V.shape, torch.bfloat16, V.device)
    rc = lib().fa_backward_dkdv(Q.data_ptr(), K.data_ptr(), V.data_ptr(), dO.data_ptr(), B, H, n,
                                m, d, int(bool(causal)), _scale(scale, d), dK.data_ptr(),
                                dV.data_ptr(), workspace.data_ptr(),
                                _workspace_bytes(workspace, Q.device), _stream(Q, stream))
    _check("fa_backward_dkdv", rc)
    return dK, dV


def fa_backward_dq(Q, K, V, dO, workspace, causal=False, scale=None, dQ=None, stream=None):
    B, H, n, m, d = _attention_inputs(Q, K, V, ("dO", dO))
    dQ = torch.empty_like(Q) if dQ is None else _out("dQ", dQ, Q.shape, torch.bfloat16, Q.device)
    rc = lib().fa_backward_dq(Q.data_ptr(), K.data_ptr(), V.data_ptr(), dO.data_ptr(), B, H, n,
                              m, d, int(bool(causal)), _scale(scale, d), dQ.data_ptr(),
                              workspace.data_ptr(), _workspace_bytes(workspace, Q.device),
                              _stream(Q, stream))
    _check("fa_backward_dq", rc)
    return dQ


def fa_backward_grads(Q, K, V, dO, workspace, causal=False, scale=None, dQ=None, dK=None,
                      dV=None, stream=None):
    """dQ, dK, dV in one launch from a workspace fa_backward_preprocess filled."""
    B, H, n, m, d = _attention_inputs(Q, K, V, ("dO", dO))
    dQ, dK, dV = _grad_outputs(Q, K, V, dQ, dK, dV)
    rc = lib().fa_backward_grads(Q.data_ptr(), K.data_ptr(), V.data_ptr(), dO.data_ptr(), B, H,
                                 n, m, d, int(bool(causal)), _scale(scale, d), dQ.data_ptr(),
                                 dK.data_ptr(), dV.data_ptr(), workspace.data_ptr(),
                                 _workspace_bytes(workspace, Q.device), _stream(Q, stream))
    _check("fa_backward_grads", rc)
    return dQ, dK, dV


def fa_online_softmax_stats(x: torch.Tensor, m=None, l=None, stream=None):
    """(m, l) per row of the fp32 CUDA matrix x [rows, cols]: m = row max,
    l = sum exp(x - m) ("05_flash_attention.py", online_softmax_stats)."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2 or x.dtype != torch.float32:
        raise ValueError("x must be a 2-D float32 tensor")
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    rows, cols = x.shape
    m = (torch.empty(rows, dtype=torch.float32, device=x.device) if m is None
         else _out("m", m, (rows,), torch.float32, x.device))
    l = (torch.empty(rows, dtype=torch.float32, device=x.device) if l is None
         else _out("l", l, (rows,), torch.float32, x.device))
    rc = lib().fa_online_softmax_stats(x.data_ptr(), rows, cols, m.data_ptr(), l.data_ptr(),
                                       _stream(x, stream))
    _check("fa_online_softmax_stats", rc)
    return m, l


class Session:
    """A host-buffer session (fa_session_create / fa_session_step, or
    fa_session_submit and fa_session_sync / destroy): one forward + backward step
    on CPU tensors, pipelined on the GPU over chunks of `chunk_heads` heads.
    Inputs and outputs are CPU tensors (page-locked ones let the copies run
    asynchronously); the device is the current CUDA device."""

    def __init__(self, B: int, H: int, n: int, m: int, d: int, chunk_heads: int):
        self.shape = (B, H, n, m, d)
        handle = ctypes.c_void_p()
        _check("fa_session_create",
               lib().fa_session_create(B, H, n, m, d, chunk_heads, ctypes.byref(handle)))
        self._handle = handle

    def step(self, Q, K, V, dO, causal: bool = False, scale: float | None = None, O=None,
             L=None, dQ=None, dK=None, dV=None):
        """O, L, dQ, dK, dV (CPU tensors, allocated here when not given), in host
        memory when the call returns."""
        return self._run("fa_session_step", Q, K, V, dO, causal, scale, O, L, dQ, dK, dV)

    def submit(self, Q, K, V, dO, causal: bool = False, scale: float | None = None, O=None,
               L=None, dQ=None, dK=None, dV=None):
        """Queues one step (fa_session_submit) and returns its O, L, dQ, dK, dV
        tensors, which hold the results once sync() has returned. Until then the
        inputs must stay unchanged and the outputs unread."""
        return self._run("fa_session_submit", Q, K, V, dO, causal, scale, O, L, dQ, dK, dV)

    def sync(self):
        """Waits until every submitted step's outputs are in host memory."""
        _check("fa_session_sync", lib().fa_session_sync(self._handle))

    def _run(self, fn, Q, K, V, dO, causal, scale, O, L, dQ, dK, dV):
        B, H, n, m, d = self.shape
        for name, t, rows in (("Q", Q, n), ("K", K, m), ("V", V, m), ("dO", dO, n)):
            if (t.is_cuda or t.dtype != torch.bfloat16 or tuple(t.shape) != (B, H, rows, d)
                    or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous bf16 CPU tensor {(B, H, rows, d)}")
        pin = Q.is_pinned()
        new = (lambda like: torch.empty_like(like, pin_memory=pin))
        cpu = torch.device("cpu")
        bf = torch.bfloat16
        O = new(Q) if O is None else _out("O", O, (B, H, n, d), bf, cpu)
        L = (torch.empty((B, H, n), dtype=torch.float32, pin_memory=pin) if L is None
             else _out("L", L, (B, H, n), torch.float32, cpu))
        dQ = new(Q) if dQ is None else _out("dQ", dQ, (B, H, n, d), bf, cpu)
        dK = new(K) if dK is None else _out("dK", dK, (B, H, m, d), bf, cpu)
        dV = new(V) if dV is None else _out("dV", dV, (B, H, m, d), bf, cpu)
        rc = getattr(lib(), fn)(self._handle, Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                                dO.data_ptr(), int(bool(causal)), _scale(scale, d),
                                O.data_ptr(), L.data_ptr(), dQ.data_ptr(), dK.data_ptr(),
                                dV.data_ptr())
        _check(fn, rc)
        return O, L, dQ, dK, dV

    def close(self):
        if self._handle:
            lib().fa_session_destroy(self._handle)
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fa_get_device_status() -> int:
    out = ctypes.c_int(0)
    _check("fa_get_device_status", lib().fa_get_device_status(ctypes.byref(out)))
    return int(out.value)


def fa_selftest_mma(mode: int, A: torch.Tensor, B: torch.Tensor) -> torch.Tensor:
    """One tcgen05 GEMM in the layout family ``mode`` (see include/fa_selftest.h)."""
    N = 64 if mode >= 3 else 128
    D = torch.empty((128, N), dtype=torch.float32, device=A.device)
    rc = lib().fa_selftest_mma(int(mode), A.data_ptr(), B.data_ptr(), D.data_ptr(),
                               torch.cuda.current_stream(A.device).cuda_stream)
    if rc != 0:
        raise RuntimeError(f"fa_selftest_mma failed ({rc})")
    return D


def fa_selftest_wait_timeout(limit_cycles: int, device=None) -> list:
    """Runs the bounded-wait failure test kernel (see include/fa_selftest.h) on
    the current stream and returns [ok of warp 0, ok of warp 1] (both 0 when
    both waits gave up, as they must)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    out = torch.full((2,), -1, dtype=torch.int32, device=dev)
    rc = lib().fa_selftest_wait_timeout(int(limit_cycles), out.data_ptr(),
                                        torch.cuda.current_stream(dev).cuda_stream)
    if rc != 0:
        raise RuntimeError(f"fa_selftest_wait_timeout failed ({rc})")
    return [int(x) for x in out.cpu()]


class FlashAttention(torch.autograd.Function):
    """Autograd wrapper: the forward saves Q, K, V, O and L (no n x m tensor),
    the backward returns dQ, dK, dV ("05_flash_attention.py", FlashAttention)."""

    @staticmethod
    def forward(ctx, Q, K, V, causal=False, scale=None):
        O, L = fa_forward(Q, K, V, causal, scale)
        ctx.save_for_backward(Q, K, V, O, L)
        ctx.causal = bool(causal)
        ctx.scale = scale
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, O, L = ctx.saved_tensors
        dQ, dK, dV = fa_backward(Q, K, V, O, L, dO.contiguous(), ctx.causal, ctx.scale)
        return dQ, dK, dV, None, None


def flash_attention(Q, K, V, causal: bool = False, scale: float | None = None):
    return FlashAttention.apply(Q, K, V, causal, scale)
