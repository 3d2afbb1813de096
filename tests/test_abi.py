"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every symbol the public headers declare, and rejects bad arguments before any
CUDA work (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import exact_io_aware_27_gb300 as fa
from exact_io_aware_27_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.lib()


def _declared_symbols():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"FA_(?:SELFTEST_)?API\s+[\w\s\*]*?\b(fa_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(names) == set(api.SIGNATURES), "binding and headers disagree"


def test_status_strings(lib):
    for code in range(0, -8, -1):
        s = fa.status_string(code)
        assert s and s != "unknown status"
    assert fa.status_string(-100) == "unknown status"
    assert fa.version() >= 100


def test_workspace_size(lib):
    # -D and -L * log2(e): n_pad floats each per head, n_pad = n rounded up to 128
    assert fa.fa_backward_workspace_size(2, 3, 100, 50, 64) == 2 * 3 * 128 * 2 * 4
    assert fa.fa_backward_workspace_size(1, 1, 128, 128, 128) == 128 * 2 * 4
    assert fa.fa_backward_workspace_size(1, 1, 129, 7, 128) == 256 * 2 * 4
    assert fa.fa_backward_workspace_size(1, 1, 0, 7, 128) == 0
    assert fa.fa_backward_workspace_size(1, 1, 8, 7, 96) == 128 * 2 * 4
    assert fa.fa_backward_workspace_size(1, 1, 8, 7, 100) == 0  # unsupported d


FAKE = 1 << 20  # an aligned non-null address; never dereferenced (validation fails first)


def _fwd(lib, Q=FAKE, K=FAKE + (1 << 24), V=FAKE + (2 << 24), B=1, H=1, n=8, m=8, d=64,
         causal=0, scale=0.125, O=FAKE + (3 << 24), L=FAKE + (4 << 24)):
    return lib.fa_forward(Q, K, V, B, H, n, m, d, causal, scale, O, L, None)


def test_forward_argument_errors(lib):
    assert _fwd(lib, Q=None) == api.FA_ERR_INVALID_ARG
    assert _fwd(lib, L=None) == api.FA_ERR_INVALID_ARG
    assert _fwd(lib, n=0) == api.FA_ERR_INVALID_ARG
    assert _fwd(lib, m=-3) == api.FA_ERR_INVALID_ARG
    assert _fwd(lib, B=0) == api.FA_ERR_INVALID_ARG
    assert _fwd(lib, B=256, H=256) == api.FA_ERR_INVALID_ARG
    for d in (0, 4, 12, 100, 136, 256):  # not a multiple of 8 in [8, 128]
        assert _fwd(lib, d=d) == api.FA_ERR_UNSUPPORTED_HEAD_DIM
    assert _fwd(lib, scale=0.0) == api.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=-1.0) == api.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == api.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("inf")) == api.FA_ERR_INVALID_ARG
    assert _fwd(lib, Q=FAKE + 2) == api.FA_ERR_MISALIGNED
    assert _fwd(lib, O=FAKE + (3 << 24) + 8) == api.FA_ERR_MISALIGNED
    assert _fwd(lib, L=FAKE + (4 << 24) + 2) == api.FA_ERR_MISALIGNED
    assert _fwd(lib, O=FAKE) == api.FA_ERR_INVALID_ARG        # O overlaps Q
    assert _fwd(lib, L=FAKE + (2 << 24) + 64) == api.FA_ERR_INVALID_ARG  # L overlaps V


def test_forward_valid_arguments_reach_the_device_check(lib):
    # Every argument is acceptable, so the call goes on to ask CUDA for the
    # device: without a GPU that fails (FA_ERR_CUDA / unsupported device).
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for d in (8, 16, 32, 64, 96, 128):
        assert _fwd(lib, d=d) in (api.FA_ERR_CUDA, api.FA_ERR_UNSUPPORTED_DEVICE)


def test_backward_argument_errors(lib):
    ws = fa.fa_backward_workspace_size(1, 1, 8, 8, 64)
    base = [FAKE + (i << 24) for i in range(10)]

    def bwd(**kw):
        a = dict(Q=base[0], K=base[1], V=base[2], O=base[3], L=base[4], dO=base[5], B=1, H=1,
                 n=8, m=8, d=64, causal=0, scale=0.125, dQ=base[6], dK=base[7], dV=base[8],
                 ws=base[9], wsb=ws)
        a.update(kw)
        return lib.fa_backward(a["Q"], a["K"], a["V"], a["O"], a["L"], a["dO"], a["B"], a["H"],
                               a["n"], a["m"], a["d"], a["causal"], a["scale"], a["dQ"], a["dK"],
                               a["dV"], a["ws"], a["wsb"], None)

    assert bwd(dO=None) == api.FA_ERR_INVALID_ARG
    assert bwd(ws=None) == api.FA_ERR_INVALID_ARG
    assert bwd(d=20) == api.FA_ERR_UNSUPPORTED_HEAD_DIM
    assert bwd(d=144) == api.FA_ERR_UNSUPPORTED_HEAD_DIM
    assert bwd(wsb=ws - 4) == api.FA_ERR_WORKSPACE_TOO_SMALL
    assert bwd(dK=base[7] + 2) == api.FA_ERR_MISALIGNED
    assert bwd(ws=base[9] + 4) == api.FA_ERR_MISALIGNED
    assert bwd(dQ=base[0]) == api.FA_ERR_INVALID_ARG           # dQ overlaps Q
    assert bwd(dV=base[7]) == api.FA_ERR_INVALID_ARG           # dV overlaps dK
    assert bwd(ws=base[6]) == api.FA_ERR_INVALID_ARG           # workspace overlaps dQ
    assert bwd(scale=0.0) == api.FA_ERR_INVALID_ARG


def test_backward_stage_argument_errors(lib):
    """The stage entry points share fa_backward's checks: missing pointers, head
    dims, alignment, overlaps and the workspace size, all before any CUDA call."""
    ws = fa.fa_backward_workspace_size(1, 1, 8, 8, 64)
    Q, K, V, O, L, dO, dQ, dK, dV, W = [FAKE + (i << 24) for i in range(10)]
    pre = lambda o=O, do=dO, l=L, d=64, w=W, wb=ws: lib.fa_backward_preprocess(
        o, do, l, 1, 1, 8, d, w, wb, None)
    assert pre(o=None) == api.FA_ERR_INVALID_ARG
    assert pre(l=None) == api.FA_ERR_INVALID_ARG
    assert pre(d=12) == api.FA_ERR_UNSUPPORTED_HEAD_DIM
    assert pre(l=L + 2) == api.FA_ERR_MISALIGNED
    assert pre(wb=ws - 4) == api.FA_ERR_WORKSPACE_TOO_SMALL
    assert pre(w=O) == api.FA_ERR_INVALID_ARG                  # workspace overlaps O
    dkdv = lambda k=K, dk=dK, dv=dV, w=W, wb=ws, scale=0.125: lib.fa_backward_dkdv(
        Q, k, V, dO, 1, 1, 8, 8, 64, 0, scale, dk, dv, w, wb, None)
    assert dkdv(k=None) == api.FA_ERR_INVALID_ARG
    assert dkdv(dv=None) == api.FA_ERR_INVALID_ARG
    assert dkdv(dk=dK + 8) == api.FA_ERR_MISALIGNED
    assert dkdv(dv=dK) == api.FA_ERR_INVALID_ARG               # dV overlaps dK
    assert dkdv(dk=K) == api.FA_ERR_INVALID_ARG                # dK overlaps K
    assert dkdv(wb=0) == api.FA_ERR_WORKSPACE_TOO_SMALL
    assert dkdv(scale=float("nan")) == api.FA_ERR_INVALID_ARG
    dq = lambda q=Q, dq_=dQ, w=W, wb=ws: lib.fa_backward_dq(
        q, K, V, dO, 1, 1, 8, 8, 64, 1, 0.125, dq_, w, wb, None)
    assert dq(dq_=None) == api.FA_ERR_INVALID_ARG
    assert dq(dq_=V) == api.FA_ERR_INVALID_ARG                 # dQ overlaps V
    assert dq(w=dQ) == api.FA_ERR_INVALID_ARG                  # workspace overlaps dQ
    assert dq(q=Q + 4) == api.FA_ERR_MISALIGNED
    grads = lambda dq_=dQ, dk=dK, dv=dV, w=W: lib.fa_backward_grads(
        Q, K, V, dO, 1, 1, 8, 8, 64, 0, 0.125, dq_, dk, dv, w, ws, None)
    assert grads(dk=None) == api.FA_ERR_INVALID_ARG
    assert grads(dq_=dV) == api.FA_ERR_INVALID_ARG             # dQ overlaps dV
    assert grads(w=None) == api.FA_ERR_INVALID_ARG


def test_noalloc_argument_errors(lib):
    Q, K, V, O, L, dO, dQ, dK, dV = [FAKE + (i << 24) for i in range(9)]
    f = lambda l=L, n=8, dk=dK: lib.fa_backward_noalloc(
        Q, K, V, O, l, dO, 1, 1, n, 8, 64, 0, 0.125, dQ, dk, dV, None)
    assert f(l=None) == api.FA_ERR_INVALID_ARG
    assert f(dk=dK + 2) == api.FA_ERR_MISALIGNED
    assert f(n=1 << 20) == api.FA_ERR_WORKSPACE_TOO_SMALL     # more than the static buffer
    assert f(n=0) == api.FA_ERR_INVALID_ARG


def test_device_status_needs_pointer(lib):
    assert lib.fa_get_device_status(None) == api.FA_ERR_INVALID_ARG


def test_python_binding_rejects_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_forward(x, x, x)


def test_python_binding_checks_buffers_it_writes_through():
    """The library sees only addresses, so the binding checks every tensor it hands
    over for writing (and the forward's L and the workspace) before any call."""
    import torch
    from exact_io_aware_27_gb300 import api as A
    cpu = torch.device("cpu")
    ok = torch.zeros(2, 3, 5, 8, dtype=torch.bfloat16)
    assert A._out("O", ok, (2, 3, 5, 8), torch.bfloat16, cpu) is ok
    bad = [
        torch.zeros(2, 3, 5, 16, dtype=torch.bfloat16),                  # shape
        torch.zeros(2, 3, 5, 8, dtype=torch.float32),                     # dtype
        torch.zeros(2, 3, 8, 5, dtype=torch.bfloat16).transpose(2, 3),    # layout
        torch.zeros(2, 3, 5, 8, dtype=torch.bfloat16, device="meta"),     # device
    ]
    for t in bad:
        with pytest.raises(ValueError):
            A._out("O", t, (2, 3, 5, 8), torch.bfloat16, cpu)
    with pytest.raises(TypeError):
        A._out("O", None, (2, 3, 5, 8), torch.bfloat16, cpu)
    A._lse(torch.zeros(2, 3, 5), 2, 3, 5, cpu)
    for L in (torch.zeros(2, 3, 6), torch.zeros(2, 3, 5, dtype=torch.float64),
              torch.zeros(2, 3, 5, device="meta")):
        with pytest.raises(ValueError):
            A._lse(L, 2, 3, 5, cpu)
    assert A._workspace_bytes(torch.zeros(10, dtype=torch.float32), cpu) == 40
    with pytest.raises(ValueError):
        A._workspace_bytes(torch.zeros(10, device="meta"), cpu)
    with pytest.raises(ValueError):
        A._same_device(ok, ok.to("meta"))


def test_selftest_argument_errors(lib):
    assert lib.fa_selftest_mma(7, FAKE, FAKE, FAKE, None) == -1
    assert lib.fa_selftest_mma(0, None, FAKE, FAKE, None) == -1
    assert lib.fa_selftest_mma(0, FAKE + 2, FAKE, FAKE, None) == -3
    assert lib.fa_selftest_wait_timeout(10**6, None, None) == -1
    assert lib.fa_selftest_wait_timeout(999, FAKE, None) == -1
    assert lib.fa_selftest_wait_timeout(2 * 10**9, FAKE, None) == -1
    assert lib.fa_selftest_wait_timeout(10**6, FAKE + 2, None) == -3


def test_online_softmax_argument_errors(lib):
    f = lib.fa_online_softmax_stats
    x, m, l = FAKE, FAKE + (1 << 24), FAKE + (2 << 24)
    assert f(None, 4, 8, m, l, None) == api.FA_ERR_INVALID_ARG
    assert f(x, 4, 8, None, l, None) == api.FA_ERR_INVALID_ARG
    assert f(x, 0, 8, m, l, None) == api.FA_ERR_INVALID_ARG
    assert f(x, 4, 0, m, l, None) == api.FA_ERR_INVALID_ARG
    assert f(x + 2, 4, 8, m, l, None) == api.FA_ERR_MISALIGNED
    assert f(x, 4, 8, x + 16, l, None) == api.FA_ERR_INVALID_ARG  # m inside x
    assert f(x, 4, 8, m, m + 8, None) == api.FA_ERR_INVALID_ARG   # l overlaps m


def test_session_argument_errors(lib):
    import ctypes
    h = ctypes.c_void_p()
    assert lib.fa_session_create(1, 1, 8, 8, 64, 1, None) == api.FA_ERR_INVALID_ARG
    assert lib.fa_session_create(0, 1, 8, 8, 64, 1, ctypes.byref(h)) == api.FA_ERR_INVALID_ARG
    assert lib.fa_session_create(1, 1, 8, 8, 20, 1, ctypes.byref(h)) == api.FA_ERR_UNSUPPORTED_HEAD_DIM
    assert lib.fa_session_create(1, 2, 8, 8, 64, 0, ctypes.byref(h)) == api.FA_ERR_INVALID_ARG
    assert lib.fa_session_create(1, 2, 8, 8, 64, 3, ctypes.byref(h)) == api.FA_ERR_INVALID_ARG
    assert not h.value  # nothing handed out on failure
    lib.fa_session_destroy(None)  # a no-op
    assert lib.fa_session_step(None, FAKE, FAKE, FAKE, FAKE, 0, 0.125, FAKE, FAKE, FAKE, FAKE,
                               FAKE) == api.FA_ERR_INVALID_ARG
    assert lib.fa_session_submit(None, FAKE, FAKE, FAKE, FAKE, 0, 0.125, FAKE, FAKE, FAKE, FAKE,
                                 FAKE) == api.FA_ERR_INVALID_ARG
    assert lib.fa_session_sync(None) == api.FA_ERR_INVALID_ARG


def test_standard_forward_argument_errors(lib):
    f = lib.fa_standard_forward
    Q, K, V = FAKE, FAKE + (1 << 24), FAKE + (2 << 24)
    S, P, O, L = FAKE + (3 << 24), FAKE + (4 << 24), FAKE + (5 << 24), FAKE + (6 << 24)

    def call(**kw):
        a = dict(Q=Q, K=K, V=V, B=1, H=1, n=8, m=8, d=64, causal=0, scale=0.125, S=S, P=P, O=O,
                 L=L)
        a.update(kw)
        return f(a["Q"], a["K"], a["V"], a["B"], a["H"], a["n"], a["m"], a["d"], a["causal"],
                 a["scale"], a["S"], a["P"], a["O"], a["L"], None)

    assert call(Q=None) == api.FA_ERR_INVALID_ARG
    assert call(S=None) == api.FA_ERR_INVALID_ARG
    assert call(P=None) == api.FA_ERR_INVALID_ARG
    assert call(n=0) == api.FA_ERR_INVALID_ARG
    assert call(d=20) == api.FA_ERR_UNSUPPORTED_HEAD_DIM
    assert call(scale=0.0) == api.FA_ERR_INVALID_ARG
    assert call(S=S + 8) == api.FA_ERR_MISALIGNED
    assert call(L=L + 2) == api.FA_ERR_MISALIGNED
    assert call(P=S) == api.FA_ERR_INVALID_ARG          # S and P overlap
    assert call(S=Q) == api.FA_ERR_INVALID_ARG          # an output over an input
    assert call(n=65535 * 128 + 1) == api.FA_ERR_INVALID_ARG  # more query tiles than grid rows


def test_standard_matrix_bytes(lib):
    assert fa.fa_standard_matrix_bytes(1, 1, 8, 8) == 8 * 64 * 2      # m_pad = 64
    assert fa.fa_standard_matrix_bytes(2, 3, 5, 64) == 2 * 3 * 5 * 64 * 2
    assert fa.fa_standard_matrix_bytes(2, 3, 5, 65) == 2 * 3 * 5 * 128 * 2
    assert fa.fa_standard_matrix_bytes(1, 1, 0, 8) == 0
    assert fa.fa_standard_matrix_bytes(1, 1, 8, 0) == 0
