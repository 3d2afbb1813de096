"""Helpers for comparing the CUDA path with the fp64 oracle.

Tolerances (fp32 accumulation, bf16 inputs and outputs):
  O   max-abs error <= 1e-2 beyond O's inherent bf16 rounding, on every element:
        |O_gpu - O_ref| <= 1e-2 + half_ulp_bf16(O_ref) + 2^-8 (P |V|)_ic
      Any kernel that feeds P to the tensor cores as bf16 and returns O in
      bf16 pays those two roundings: up to 2^-8 of each weight P_ij (an error
      up to 2^-8 sum_j P_ij |V_jc| in O, which passes 0.01 when a row's weight
      sits on a few keys with |V| > 2.5: the first rows under causal masking,
      a peaked softmax) and half a bf16 ulp of O (0.0156 for |O| in [4, 8)).
      P |V| comes from the oracle run on |V|. Checks with raw_o=True (the
      named workloads with N(0,1) inputs, the closed forms) also assert the
      raw bound |O_gpu - O_ref| <= 1e-2 on every element. The raw figure is
      recorded for every check.
  L   max-abs error  <= 2e-3   (natural log)
  dQ, dK, dV  relative Frobenius error ||g - r||_F / ||r||_F <= 1e-2

Every check records its figures in REPORTS, which tests/conftest.py writes out
as JSON when FA_PARITY_REPORT names a file.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import exact_io_aware_27_gb300 as fa
import oracle

O_MAXABS = 1e-2
L_MAXABS = 2e-3
GRAD_REL = 1e-2


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def half_ulp_bf16(x) -> np.ndarray:
    """Half the bf16 spacing at |x| (8 significant bits): 2^(floor(log2|x|) - 8)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 8)


REPORTS = []  # one dict per check: label and figures


def o_errors(g, r, pv_abs=None) -> dict:
    """Raw max-abs error of O, and the error beyond O's inherent bf16 rounding:
    half a bf16 ulp of r, plus 2^-8 (P |V|) when pv_abs (the oracle's output for
    |V|) is given."""
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    diff = np.abs(g - r)
    allow = half_ulp_bf16(r)
    if pv_abs is not None:
        allow = allow + np.ldexp(np.asarray(pv_abs, dtype=np.float64), -8)
    return {
        "O_raw": float(diff.max()) if diff.size else 0.0,
        "O_beyond_rounding": float((diff - allow).max()) if diff.size else 0.0,
    }


def o_error(g, r) -> float:
    """Raw max-abs error of O."""
    return o_errors(g, r)["O_raw"]


def _merge(report, errs):
    for key, val in errs.items():
        report[key] = max(report.get(key, 0.0), val)


def _record(report, label, raw_o):
    if label is None:
        label = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    REPORTS.append({"label": label, "raw_o": raw_o, **report})


def rel_fro(g, r) -> float:
    den = float(np.linalg.norm(r))
    num = float(np.linalg.norm(np.asarray(g, dtype=np.float64) - r))
    return num / den if den > 0 else num


def run_gpu(Q, K, V, dO, causal, scale=None, device="cuda"):
    """Forward + backward through the C-ABI; returns fp64 numpy arrays."""
    q, k, v, do = (t.to(device).contiguous() for t in (Q, K, V, dO))
    O, L = fa.fa_forward(q, k, v, causal, scale)
    dQ, dK, dV = fa.fa_backward(q, k, v, O, L, do, causal, scale)
    torch.cuda.synchronize()
    return {"O": f64(O), "L": f64(L), "dQ": f64(dQ), "dK": f64(dK), "dV": f64(dV)}


def check_heads(Q, K, V, dO, causal, got, heads=None, scale=None, label=None, raw_o=False):
    """Full-row comparison on every head (or the listed flat head indices).
    raw_o=True also asserts the raw O bound on every element."""
    B, H, n, d = Q.shape
    m = K.shape[2]
    flat = [t.reshape(B * H, -1, d) for t in (Q, K, V, dO)]
    g = {k: v.reshape(B * H, *v.shape[2:]) for k, v in got.items()}
    heads = range(B * H) if heads is None else heads
    report = {}
    for h in heads:
        q, k, v, do = (f64(t[h]) for t in flat)
        O_r, L_r = oracle.forward(q, k, v, causal, scale)
        dQ_r, dK_r, dV_r, _ = oracle.backward(q, k, v, do, causal, scale)
        pv_abs = oracle.forward(q, k, np.abs(v), causal, scale)[0]
        errs = {
            **o_errors(g["O"][h], O_r, pv_abs),
            "L": float(np.max(np.abs(g["L"][h] - L_r))),
            "dQ": rel_fro(g["dQ"][h], dQ_r),
            "dK": rel_fro(g["dK"][h], dK_r),
            "dV": rel_fro(g["dV"][h], dV_r),
        }
        _merge(report, errs)
    _record(report, label, raw_o)
    assert_within(report, raw_o)
    return report


def check_sampled(Q, K, V, dO, causal, got, heads, q_rows, k_rows, scale=None, label=None,
                  raw_o=False):
    """Sampled rows of sampled heads (for workloads the full oracle is too slow on)."""
    B, H, n, d = Q.shape
    flat = [t.reshape(B * H, -1, d) for t in (Q, K, V, dO)]
    g = {k: v.reshape(B * H, *v.shape[2:]) for k, v in got.items()}
    orc = oracle.default()
    report = {}
    for h in heads:
        q, k, v, do = (f64(t[h]) for t in flat)
        O_r, L_r = orc.forward_rows(q, k, v, q_rows, causal, scale)
        dQ_r, dK_r, dV_r, _ = orc.backward_rows(q, k, v, do, q_rows, k_rows, causal, scale)
        errs = {
            **o_errors(g["O"][h][q_rows], O_r,
                       orc.forward_rows(q, k, np.abs(v), q_rows, causal, scale)[0]),
            "L": float(np.max(np.abs(g["L"][h][q_rows] - L_r))),
            "dQ": rel_fro(g["dQ"][h][q_rows], dQ_r),
            "dK": rel_fro(g["dK"][h][k_rows], dK_r),
            "dV": rel_fro(g["dV"][h][k_rows], dV_r),
        }
        _merge(report, errs)
    _record(report, label, raw_o)
    assert_within(report, raw_o)
    return report


def assert_within(report, raw_o=False):
    bad = []
    if raw_o and not report["O_raw"] <= O_MAXABS:
        bad.append(f"O max-abs {report['O_raw']:.3e} > {O_MAXABS}")
    if not report["O_beyond_rounding"] <= O_MAXABS:
        bad.append(f"O max-abs beyond its inherent bf16 rounding "
                   f"{report['O_beyond_rounding']:.3e} > {O_MAXABS}")
    if not report["L"] <= L_MAXABS:
        bad.append(f"L max-abs {report['L']:.3e} > {L_MAXABS}")
    for k in ("dQ", "dK", "dV"):
        if not report[k] <= GRAD_REL:
            bad.append(f"{k} rel-Frobenius {report[k]:.3e} > {GRAD_REL}")
    assert not bad, "; ".join(bad) + f" (all: {report})"
