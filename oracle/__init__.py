"""fp64 CPU oracle for exact attention (forward, logsumexp and gradients).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The CUDA
library never calls it and it never calls the CUDA library: the two share no
code, only the seeded input generator in ``exact_io_aware_27_gb300.inputs``
(which holds no attention arithmetic).

The arithmetic lives in ``attention_fp64.cpp`` (plain C++17 + OpenMP, double
precision). This module compiles it with the system ``g++`` and calls it
through ctypes, one head at a time.

Definitions followed (see the C++ header comment for the full list):
  * standard attention and its causal mask -- "05_flash_attention.py",
    ``standard_attention``;
  * L = m + log l -- same page, ``flash_attention_forward`` docstring;
  * dV, dP, D, dS, dQ, dK -- same page, ``flash_attention_backward``
    docstring, and "Flash Attention" notes, section 1.5;
  * the online max / rescaled-sum recurrence -- same page,
    ``online_softmax_stats``; notes, section 1.1.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(closed forms, library special cases, finite differences, invariants and
hand-derived golden values) and by ``tests/test_oracle_mutants.py`` (planted
mistakes must fail a pin).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attention_fp64.cpp")
LIBRARY = os.path.join(_HERE, "liboracle_attention.so")

_lock = threading.Lock()
_default = None

_CXXFLAGS = ["-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off"]


def build(force: bool = False, src: str = SOURCE, out: str = LIBRARY) -> str:
    """Compile the oracle into a shared library (idempotent unless ``force``)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["g++", *_CXXFLAGS, src, "-o", tmp], check=True)
    os.replace(tmp, out)
    return out


_dptr = ctypes.POINTER(ctypes.c_double)


def _as_ptr(a: np.ndarray):
    return a.ctypes.data_as(_dptr)


class Oracle:
    """ctypes handle on one compiled copy of the oracle."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_online_softmax_stats.argtypes = [
            _dptr, ctypes.c_long, ctypes.c_long, _dptr, _dptr]
        lib.oracle_online_softmax_stats.restype = ctypes.c_int
        lib.oracle_attention_forward.argtypes = [
            _dptr, _dptr, _dptr, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.c_int, ctypes.c_double, _dptr, _dptr]
        lib.oracle_attention_forward.restype = ctypes.c_int
        lib.oracle_attention_backward.argtypes = [
            _dptr, _dptr, _dptr, _dptr, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.c_int, ctypes.c_double, _dptr, _dptr, _dptr, _dptr]
        lib.oracle_attention_backward.restype = ctypes.c_int
        _lp = ctypes.POINTER(ctypes.c_long)
        lib.oracle_attention_forward_rows.argtypes = [
            _dptr, _dptr, _dptr, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_int,
            ctypes.c_double, _lp, ctypes.c_long, _dptr, _dptr]
        lib.oracle_attention_forward_rows.restype = ctypes.c_int
        lib.oracle_attention_backward_rows.argtypes = [
            _dptr, _dptr, _dptr, _dptr, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.c_int, ctypes.c_double, _lp, ctypes.c_long, _lp, ctypes.c_long, _dptr,
            _dptr, _dptr, _dptr]
        lib.oracle_attention_backward_rows.restype = ctypes.c_int
        lib.oracle_attention_probabilities.argtypes = [
            _dptr, _dptr, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_int,
            ctypes.c_double, _dptr, _dptr]
        lib.oracle_attention_probabilities.restype = ctypes.c_int
        self._lib = lib
        self.path = path

    # -- threads -----------------------------------------------------------
    def num_threads(self) -> int:
        return int(self._lib.oracle_num_threads())

    def set_num_threads(self, t: int) -> None:
        self._lib.oracle_set_num_threads(int(t))

    # -- online statistics -------------------------------------------------
    def online_softmax_stats(self, x, block: int):
        """(m, l) of the one-pass recurrence over the 1-D array ``x``."""
        x = np.ascontiguousarray(x, dtype=np.float64).ravel()
        m = np.zeros(1)
        l = np.zeros(1)
        rc = self._lib.oracle_online_softmax_stats(_as_ptr(x), x.size, int(block),
                                                   _as_ptr(m), _as_ptr(l))
        if rc != 0:
            raise ValueError("oracle_online_softmax_stats: bad arguments")
        return float(m[0]), float(l[0])

    # -- attention ---------------------------------------------------------
    @staticmethod
    def _heads(x):
        x = np.ascontiguousarray(x, dtype=np.float64)
        lead = x.shape[:-2]
        return x.reshape(-1, x.shape[-2], x.shape[-1]), lead

    def forward(self, Q, K, V, causal: bool = False, scale: float | None = None):
        """O [..., n, d] and natural-log L [..., n] for every head of Q, K, V."""
        q, lead = self._heads(Q)
        k, _ = self._heads(K)
        v, _ = self._heads(V)
        nh, n, d = q.shape
        m = k.shape[1]
        if scale is None:
            scale = 1.0 / np.sqrt(d)
        O = np.empty((nh, n, d))
        L = np.empty((nh, n))
        for h in range(nh):
            rc = self._lib.oracle_attention_forward(
                _as_ptr(q[h]), _as_ptr(k[h]), _as_ptr(v[h]), n, m, d, int(bool(causal)),
                float(scale), _as_ptr(O[h]), _as_ptr(L[h]))
            if rc != 0:
                raise ValueError("oracle_attention_forward: bad arguments")
        return O.reshape(*lead, n, d), L.reshape(*lead, n)

    def probabilities(self, Q, K, causal: bool = False, scale: float | None = None):
        """S [..., n, m] (-inf where masked) and P = softmax(S) [..., n, m] per head."""
        q, lead = self._heads(Q)
        k, _ = self._heads(K)
        nh, n, d = q.shape
        m = k.shape[1]
        if scale is None:
            scale = 1.0 / np.sqrt(d)
        S = np.empty((nh, n, m))
        P = np.empty((nh, n, m))
        for h in range(nh):
            rc = self._lib.oracle_attention_probabilities(
                _as_ptr(q[h]), _as_ptr(k[h]), n, m, d, int(bool(causal)), float(scale),
                _as_ptr(S[h]), _as_ptr(P[h]))
            if rc != 0:
                raise ValueError("oracle_attention_probabilities: bad arguments")
        return S.reshape(*lead, n, m), P.reshape(*lead, n, m)

    def backward(self, Q, K, V, dO, causal: bool = False, scale: float | None = None):
        """dQ, dK, dV and D (= sum_j P_ij dP_ij) for the loss sum(O * dO)."""
        q, lead = self._heads(Q)
        k, _ = self._heads(K)
        v, _ = self._heads(V)
        do, _ = self._heads(dO)
        nh, n, d = q.shape
        m = k.shape[1]
        if scale is None:
            scale = 1.0 / np.sqrt(d)
        dQ = np.empty((nh, n, d))
        dK = np.empty((nh, m, d))
        dV = np.empty((nh, m, d))
        D = np.empty((nh, n))
        for h in range(nh):
            rc = self._lib.oracle_attention_backward(
                _as_ptr(q[h]), _as_ptr(k[h]), _as_ptr(v[h]), _as_ptr(do[h]), n, m, d,
                int(bool(causal)), float(scale), _as_ptr(dQ[h]), _as_ptr(dK[h]),
                _as_ptr(dV[h]), _as_ptr(D[h]))
            if rc != 0:
                raise ValueError("oracle_attention_backward: bad arguments")
        return (dQ.reshape(*lead, n, d), dK.reshape(*lead, m, d),
                dV.reshape(*lead, m, d), D.reshape(*lead, n))


    # -- sampled rows of one head -------------------------------------------
    def forward_rows(self, Q, K, V, rows, causal=False, scale=None):
        """O[rows] and L[rows] of one head (Q [n,d], K and V [m,d])."""
        q, k, v = (np.ascontiguousarray(x, dtype=np.float64) for x in (Q, K, V))
        n, d = q.shape
        m = k.shape[0]
        idx = np.ascontiguousarray(rows, dtype=np.int64)
        scale = 1.0 / np.sqrt(d) if scale is None else scale
        O = np.empty((idx.size, d))
        L = np.empty(idx.size)
        rc = self._lib.oracle_attention_forward_rows(
            _as_ptr(q), _as_ptr(k), _as_ptr(v), n, m, d, int(bool(causal)), float(scale),
            idx.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), idx.size, _as_ptr(O), _as_ptr(L))
        if rc != 0:
            raise ValueError("oracle_attention_forward_rows: bad arguments")
        return O, L

    def backward_rows(self, Q, K, V, dO, q_rows, k_rows, causal=False, scale=None):
        """dQ[q_rows], dK[k_rows], dV[k_rows] and D (all rows) of one head."""
        q, k, v, do = (np.ascontiguousarray(x, dtype=np.float64) for x in (Q, K, V, dO))
        n, d = q.shape
        m = k.shape[0]
        qi = np.ascontiguousarray(q_rows, dtype=np.int64)
        ki = np.ascontiguousarray(k_rows, dtype=np.int64)
        scale = 1.0 / np.sqrt(d) if scale is None else scale
        dQ = np.empty((max(qi.size, 1), d))
        dK = np.empty((max(ki.size, 1), d))
        dV = np.empty((max(ki.size, 1), d))
        D = np.empty(n)
        lp = ctypes.POINTER(ctypes.c_long)
        rc = self._lib.oracle_attention_backward_rows(
            _as_ptr(q), _as_ptr(k), _as_ptr(v), _as_ptr(do), n, m, d, int(bool(causal)),
            float(scale), qi.ctypes.data_as(lp), qi.size, ki.ctypes.data_as(lp), ki.size,
            _as_ptr(dQ), _as_ptr(dK), _as_ptr(dV), _as_ptr(D))
        if rc != 0:
            raise ValueError("oracle_attention_backward_rows: bad arguments")
        return dQ[:qi.size], dK[:ki.size], dV[:ki.size], D


def default() -> Oracle:
    """The oracle compiled from this package's source (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def online_softmax_stats(x, block):
    return default().online_softmax_stats(x, block)


def forward(Q, K, V, causal=False, scale=None):
    return default().forward(Q, K, V, causal, scale)


def backward(Q, K, V, dO, causal=False, scale=None):
    return default().backward(Q, K, V, dO, causal, scale)


def probabilities(Q, K, causal=False, scale=None):
    return default().probabilities(Q, K, causal, scale)
