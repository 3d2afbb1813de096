"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` function takes a compiled oracle (``oracle.Oracle``) and raises
``AssertionError`` if the oracle disagrees with a value fixed independently of
it: hand-derived closed forms (``tests/golden``), special cases that reduce to
a library routine (scipy softmax / logsumexp, torch autograd in fp64), finite
differences, algebraic invariants, and tiling independence: the online-softmax
merge of per-block statistics and the per-block gradient terms, over shuffled
even and uneven block partitions, must reproduce the untiled oracle.

The same pins run against mutated copies of the oracle in
``test_oracle_mutants.py``; every planted mistake must trip at least one.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "closed_form_tiny.json")


def _close(a, b, rtol, atol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    if not np.allclose(a, b, rtol=rtol, atol=atol):
        err = np.max(np.abs(a - b))
        raise AssertionError(f"{what}: max abs diff {err:.3e}")


def _eval(expr):
    return float(eval(expr, {"__builtins__": {}}, {"log": math.log, "sqrt": math.sqrt}))


def _arr(x):
    if isinstance(x, str):
        return _eval(x)
    return np.array([_arr(v) for v in x], dtype=np.float64)


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# Hand-derived closed forms (tests/golden/closed_form_tiny.json)
# --------------------------------------------------------------------------
def pin_golden(orc):
    data = json.load(open(GOLDEN))
    for case in data["cases"]:
        Q, K, V, dO = (_arr(case[k]) for k in ("Q", "K", "V", "dO"))
        scale = _eval(case["scale"])
        O, L = orc.forward(Q, K, V, case["causal"], scale)
        _close(O, _arr(case["O"]), 1e-13, 1e-13, case["name"] + " O")
        _close(L, _arr(case["L"]), 1e-13, 1e-13, case["name"] + " L")
        dQ, dK, dV, D = orc.backward(Q, K, V, dO, case["causal"], scale)
        for name, got in (("D", D), ("dQ", dQ), ("dK", dK), ("dV", dV)):
            _close(got, _arr(case[name]), 1e-13, 1e-13, f"{case['name']} {name}")
    for case in data["online_stats"]:
        m, l = orc.online_softmax_stats(_arr(case["x"]), case["block"])
        _close(m, _eval(case["m"]), 1e-14, 1e-14, case["name"] + " m")
        _close(l, _eval(case["l"]), 1e-14, 1e-14, case["name"] + " l")


# --------------------------------------------------------------------------
# O1: online statistics equal the direct max / logsumexp
# --------------------------------------------------------------------------
def pin_online_stats(orc):
    rng = _rng(1)
    for length in (1, 10, 37, 200):
        x = rng.standard_normal(length) * 5.0  # the pages' demo draws randn(10) * 5
        for block in sorted({1, 2, 3, 4, 16, 24, length}):
            m, l = orc.online_softmax_stats(x, block)
            _close(m, np.max(x), 0, 0, f"online max len={length} block={block}")
            _close(m + math.log(l), scipy.special.logsumexp(x), 1e-12, 1e-12,
                   f"online logsumexp len={length} block={block}")
            _close(np.exp(x - m) / l, scipy.special.softmax(x), 1e-12, 1e-15,
                   f"online softmax len={length} block={block}")


# --------------------------------------------------------------------------
# O2: with V = identity the output is P itself (library softmax); rows sum to 1
# --------------------------------------------------------------------------
def pin_softmax_identity_v(orc):
    rng = _rng(2)
    n, m = 6, 5
    for causal in (False, True):
        Q = rng.standard_normal((n, m))
        K = rng.standard_normal((m, m))
        V = np.eye(m)
        scale = 0.7
        O, L = orc.forward(Q, K, V, causal, scale)
        S = (Q @ K.T) * scale
        if causal:
            S = np.where(np.arange(m)[None, :] > np.arange(n)[:, None], -np.inf, S)
        _close(O, scipy.special.softmax(S, axis=1), 1e-12, 1e-15, f"P causal={causal}")
        _close(L, scipy.special.logsumexp(S, axis=1), 1e-12, 1e-12, f"L causal={causal}")
        ones = np.ones((m, m))
        O1, _ = orc.forward(Q, K, ones, causal, scale)
        _close(O1, np.ones((n, m)), 1e-13, 1e-13, f"row sums causal={causal}")


# --------------------------------------------------------------------------
# O3: causal row 0 sees only key 0
# --------------------------------------------------------------------------
def pin_causal_row0(orc):
    rng = _rng(3)
    n, m, d = 9, 9, 4
    Q, K, V = rng.standard_normal((n, d)), rng.standard_normal((m, d)), rng.standard_normal((m, d))
    O, L = orc.forward(Q, K, V, True, 0.5)
    _close(O[0], V[0], 1e-14, 1e-14, "causal O_0 = V_0")
    _close(L[0], 0.5 * float(Q[0] @ K[0]), 1e-14, 1e-14, "causal L_0 = s Q_0.K_0")


# --------------------------------------------------------------------------
# O4: Q = 0 gives uniform attention
# --------------------------------------------------------------------------
def pin_zero_query(orc):
    rng = _rng(4)
    n, m, d = 7, 7, 3
    Q = np.zeros((n, d))
    K, V = rng.standard_normal((m, d)), rng.standard_normal((m, d))
    O, L = orc.forward(Q, K, V, False, 0.3)
    _close(O, np.repeat(V.mean(axis=0, keepdims=True), n, axis=0), 1e-13, 1e-14, "Q=0 O")
    _close(L, np.full(n, math.log(m)), 1e-14, 1e-14, "Q=0 L")
    O, L = orc.forward(Q, K, V, True, 0.3)
    cummean = np.cumsum(V, axis=0) / np.arange(1, m + 1)[:, None]
    _close(O, cummean, 1e-13, 1e-14, "Q=0 causal O")
    _close(L, np.log(np.arange(1, n + 1)), 1e-14, 1e-14, "Q=0 causal L")


# --------------------------------------------------------------------------
# O5: a single key
# --------------------------------------------------------------------------
def pin_single_key(orc):
    rng = _rng(5)
    n, d = 6, 4
    Q, K, V, dO = (rng.standard_normal(s) for s in ((n, d), (1, d), (1, d), (n, d)))
    for causal in (False, True):
        O, L = orc.forward(Q, K, V, causal, 0.4)
        _close(O, np.repeat(V, n, axis=0), 1e-14, 1e-14, "m=1 O")
        _close(L, 0.4 * (Q @ K[0]), 1e-14, 1e-14, "m=1 L")
        dQ, dK, dV, _ = orc.backward(Q, K, V, dO, causal, 0.4)
        _close(dQ, np.zeros_like(dQ), 0, 1e-14, "m=1 dQ")
        _close(dK, np.zeros_like(dK), 0, 1e-14, "m=1 dK")
        _close(dV, dO.sum(axis=0, keepdims=True), 1e-14, 1e-14, "m=1 dV")


# --------------------------------------------------------------------------
# O6: central finite differences of f = sum(O * dO)
# --------------------------------------------------------------------------
def pin_finite_differences(orc):
    rng = _rng(6)
    h = 1e-6
    for (n, m, d, causal) in ((5, 6, 3, False), (4, 4, 4, True), (6, 4, 2, True)):
        Q, K, V, dO = (rng.standard_normal(s) for s in ((n, d), (m, d), (m, d), (n, d)))
        scale = 0.6

        def f(Q_, K_, V_):
            O, _ = orc.forward(Q_, K_, V_, causal, scale)
            return float(np.sum(O * dO))

        dQ, dK, dV, _ = orc.backward(Q, K, V, dO, causal, scale)
        for name, X, G in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
            num = np.zeros_like(X)
            for idx in np.ndindex(X.shape):
                Xp, Xm = X.copy(), X.copy()
                Xp[idx] += h
                Xm[idx] -= h
                args_p = {"Q": (Xp, K, V), "K": (Q, Xp, V), "V": (Q, K, Xp)}[name]
                args_m = {"Q": (Xm, K, V), "K": (Q, Xm, V), "V": (Q, K, Xm)}[name]
                num[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
            scale_ref = max(1.0, float(np.max(np.abs(num))))
            err = float(np.max(np.abs(num - G))) / scale_ref
            assert err <= 1e-7, f"finite differences d{name} n={n} m={m} causal={causal}: {err:.2e}"


# --------------------------------------------------------------------------
# O7: invariants of the gradients
# --------------------------------------------------------------------------
def pin_invariants(orc):
    rng = _rng(7)
    for (n, m, d, causal) in ((7, 9, 4, False), (8, 8, 5, True), (9, 7, 3, True)):
        Q, K, V, dO = (rng.standard_normal(s) for s in ((n, d), (m, d), (m, d), (n, d)))
        scale = 0.45
        O, _ = orc.forward(Q, K, V, causal, scale)
        dQ, dK, dV, D = orc.backward(Q, K, V, dO, causal, scale)
        tag = f"n={n} m={m} causal={causal}"
        _close(D, np.sum(dO * O, axis=1), 1e-12, 1e-13, "D = rowsum(dO*O) " + tag)
        _close(dK.sum(axis=0), np.zeros(d), 0, 1e-12, "sum_j dK_j = 0 " + tag)
        _close(dV.sum(axis=0), dO.sum(axis=0), 1e-12, 1e-12, "sum dV = sum dO " + tag)
        _close(np.sum(Q * dQ), np.sum(K * dK), 1e-12, 1e-12, "<Q,dQ> = <K,dK> " + tag)


# --------------------------------------------------------------------------
# Library special case: torch autograd through standard attention in fp64
# --------------------------------------------------------------------------
def pin_torch_autograd(orc):
    import torch
    rng = _rng(8)
    for (n, m, d, causal) in ((6, 7, 5, False), (7, 7, 5, True), (8, 5, 3, True)):
        Q, K, V, dO = (rng.standard_normal(s) for s in ((n, d), (m, d), (m, d), (n, d)))
        scale = 1.0 / math.sqrt(d)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
        S = (tq @ tk.T) * scale
        if causal:
            S = S.masked_fill(torch.ones(n, m, dtype=torch.bool).triu(1), float("-inf"))
        O_t = torch.softmax(S, dim=-1) @ tv
        L_t = torch.logsumexp(S, dim=-1)
        (O_t * torch.tensor(dO)).sum().backward()
        O, L = orc.forward(Q, K, V, causal, scale)
        dQ, dK, dV, _ = orc.backward(Q, K, V, dO, causal, scale)
        tag = f"n={n} m={m} causal={causal}"
        _close(O, O_t.detach().numpy(), 1e-12, 1e-13, "O vs torch " + tag)
        _close(L, L_t.detach().numpy(), 1e-12, 1e-13, "L vs torch " + tag)
        _close(dQ, tq.grad.numpy(), 1e-11, 1e-12, "dQ vs torch " + tag)
        _close(dK, tk.grad.numpy(), 1e-11, 1e-12, "dK vs torch " + tag)
        _close(dV, tv.grad.numpy(), 1e-11, 1e-12, "dV vs torch " + tag)


# --------------------------------------------------------------------------
# O8: tiling independence. The forward is the online-softmax recurrence
# ("Flash Attention" notes, section 1.1) in its merge form: for two disjoint
# sets of keys with statistics (m1, l1), (m2, l2) and unnormalised outputs U1, U2,
#   M = max(m1, m2),  l = l1 e^(m1 - M) + l2 e^(m2 - M),  U = U1 e^(m1 - M) + U2 e^(m2 - M),
# so any partition of the score matrix into blocks, merged in any order, must
# reproduce the oracle. The backward sums the per-block terms of the FA-2
# gradient formulas ("05_flash_attention.py", flash_attention_backward
# docstring: P = exp(S - L), dV += P^T dO, dS = P o (dO V^T - D), dQ += s dS K,
# dK += s dS^T Q), which any visiting order must also reproduce. Blocks are
# visited in a shuffled order, over even and uneven partitions.
# --------------------------------------------------------------------------
def _even_cuts(total, size):
    """Boundaries of consecutive blocks of `size` rows (the last one ragged)."""
    return list(range(0, total, size)) + [total]


def _uneven_cuts(total, rng, lo, hi):
    """Boundaries of consecutive blocks of random sizes in [lo, hi]."""
    cuts = [0]
    while cuts[-1] < total:
        cuts.append(min(total, cuts[-1] + int(rng.integers(lo, hi + 1))))
    return cuts


def _block_grid(row_cuts, col_cuts, causal):
    """(query range, key range) pairs holding at least one visible score."""
    grid = []
    for r0, r1 in zip(row_cuts, row_cuts[1:]):
        for c0, c1 in zip(col_cuts, col_cuts[1:]):
            if causal and c0 > r1 - 1:  # top-left causal: key c visible from query q iff c <= q
                continue
            grid.append(((r0, r1), (c0, c1)))
    return grid


def _block_scores(Q, K, rows, cols, causal, scale):
    S = scale * (Q[rows[0]:rows[1]] @ K[cols[0]:cols[1]].T)
    if causal:
        hidden = np.arange(*cols)[None, :] > np.arange(*rows)[:, None]
        S = np.where(hidden, -np.inf, S)
    return S


def _merge_weights(m_a, m_b):
    """e^(m_a - M), e^(m_b - M) for M = max(m_a, m_b); 0 for a side still at -inf."""
    M = np.maximum(m_a, m_b)
    finite = np.isfinite(M)
    safe = np.where(finite, M, 0.0)
    w_a = np.where(np.isfinite(m_a), np.exp(np.where(np.isfinite(m_a), m_a, 0.0) - safe), 0.0)
    w_b = np.where(np.isfinite(m_b), np.exp(np.where(np.isfinite(m_b), m_b, 0.0) - safe), 0.0)
    return M, w_a, w_b


def _tiled_forward(Q, K, V, causal, row_cuts, col_cuts, rng):
    n, d = Q.shape
    scale = 1.0 / math.sqrt(d)
    run_m = np.full(n, -np.inf)      # running maximum per query
    run_l = np.zeros(n)              # exp-sum relative to run_m
    run_u = np.zeros((n, d))         # unnormalised output relative to run_m
    grid = _block_grid(row_cuts, col_cuts, causal)
    for g in rng.permutation(len(grid)):
        rows, cols = grid[g]
        S = _block_scores(Q, K, rows, cols, causal, scale)
        blk_m = S.max(axis=1)        # -inf for a row with no visible key in the block
        E = np.exp(S - np.where(np.isfinite(blk_m), blk_m, 0.0)[:, None])
        blk_l, blk_u = E.sum(axis=1), E @ V[cols[0]:cols[1]]
        sl = slice(*rows)
        M, w_run, w_blk = _merge_weights(run_m[sl], blk_m)
        run_l[sl] = run_l[sl] * w_run + blk_l * w_blk
        run_u[sl] = run_u[sl] * w_run[:, None] + blk_u * w_blk[:, None]
        run_m[sl] = M
    return run_u / run_l[:, None], run_m + np.log(run_l)


def _tiled_backward(Q, K, V, O, L, dO, causal, row_cuts, col_cuts, rng):
    d = Q.shape[1]
    scale = 1.0 / math.sqrt(d)
    Drow = np.einsum("ij,ij->i", dO, O)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    grid = _block_grid(row_cuts, col_cuts, causal)
    for g in rng.permutation(len(grid)):
        rows, cols = grid[g]
        qs, ks = slice(*rows), slice(*cols)
        P = np.exp(_block_scores(Q, K, rows, cols, causal, scale) - L[qs, None])
        dS = P * (dO[qs] @ V[ks].T - Drow[qs, None])
        dQ[qs] += scale * (dS @ K[ks])
        dK[ks] += scale * (dS.T @ Q[qs])
        dV[ks] += P.T @ dO[qs]
    return dQ, dK, dV


def pin_tiled_page1(orc):
    rng = _rng(9)
    # the pages' forward demo shape: n = 100, d = 32, 16-query x 24-key blocks
    n, d = 100, 32
    Q, K, V = (rng.standard_normal((n, d)) for _ in range(3))
    parts = [("16x24", _even_cuts(n, 16), _even_cuts(n, 24)),
             ("uneven", _uneven_cuts(n, rng, 3, 29), _uneven_cuts(n, rng, 2, 31))]
    for causal in (False, True):
        O, L = orc.forward(Q, K, V, causal)
        for tag, rc, cc in parts:
            O_t, L_t = _tiled_forward(Q, K, V, causal, rc, cc, rng)
            _close(O, O_t, 1e-12, 1e-12, f"tiled forward O {tag} causal={causal}")
            _close(L, L_t, 1e-12, 1e-12, f"tiled forward L {tag} causal={causal}")
    # the pages' backward demo: n = 70, d = 16, loss sum(O**2) so dO = 2 O
    n, d = 70, 16
    Q, K, V = (rng.standard_normal((n, d)) for _ in range(3))
    parts = [("16x16", _even_cuts(n, 16), _even_cuts(n, 16)),
             ("uneven", _uneven_cuts(n, rng, 2, 23), _uneven_cuts(n, rng, 4, 19))]
    for causal in (False, True):
        O, L = orc.forward(Q, K, V, causal)
        dO = 2.0 * O
        dQ, dK, dV, _ = orc.backward(Q, K, V, dO, causal)
        for tag, rc, cc in parts:
            dQ_t, dK_t, dV_t = _tiled_backward(Q, K, V, O, L, dO, causal, rc, cc, rng)
            _close(dQ, dQ_t, 1e-11, 1e-12, f"tiled backward dQ {tag} causal={causal}")
            _close(dK, dK_t, 1e-11, 1e-12, f"tiled backward dK {tag} causal={causal}")
            _close(dV, dV_t, 1e-11, 1e-12, f"tiled backward dV {tag} causal={causal}")


# --------------------------------------------------------------------------
# Top-left causal alignment when n != m
# --------------------------------------------------------------------------
def pin_causal_nonsquare(orc):
    rng = _rng(10)
    d = 3
    # more queries than keys: rows i >= m-1 see every key
    n, m = 6, 3
    Q, K, V = rng.standard_normal((n, d)), rng.standard_normal((m, d)), rng.standard_normal((m, d))
    Oc, Lc = orc.forward(Q, K, V, True, 0.5)
    On, Ln = orc.forward(Q, K, V, False, 0.5)
    _close(Oc[m - 1:], On[m - 1:], 1e-14, 1e-14, "n>m causal rows past m")
    # more keys than queries: row i sees exactly keys 0..i
    n, m = 3, 6
    Q, K, V = rng.standard_normal((n, d)), rng.standard_normal((m, d)), rng.standard_normal((m, d))
    Oc, Lc = orc.forward(Q, K, V, True, 0.5)
    for i in range(n):
        Oi, Li = orc.forward(Q[i:i + 1], K[:i + 1], V[:i + 1], False, 0.5)
        _close(Oc[i], Oi[0], 1e-14, 1e-14, f"n<m causal row {i} O")
        _close(Lc[i], Li[0], 1e-14, 1e-14, f"n<m causal row {i} L")


# --------------------------------------------------------------------------
# Sampled-row evaluation equals the same rows of the full evaluation
# --------------------------------------------------------------------------
def pin_sampled_rows(orc):
    rng = _rng(11)
    for (n, m, d, causal) in ((13, 11, 4, True), (9, 14, 3, False)):
        Q, K, V, dO = (rng.standard_normal(s) for s in ((n, d), (m, d), (m, d), (n, d)))
        O, L = orc.forward(Q, K, V, causal, 0.5)
        dQ, dK, dV, D = orc.backward(Q, K, V, dO, causal, 0.5)
        qr = np.array([n - 1, 0, 5, 2])
        kr = np.array([3, m - 1, 0])
        Os, Ls = orc.forward_rows(Q, K, V, qr, causal, 0.5)
        _close(Os, O[qr], 1e-15, 1e-15, "sampled O")
        _close(Ls, L[qr], 1e-15, 1e-15, "sampled L")
        dQs, dKs, dVs, Ds = orc.backward_rows(Q, K, V, dO, qr, kr, causal, 0.5)
        _close(dQs, dQ[qr], 1e-15, 1e-15, "sampled dQ")
        _close(dKs, dK[kr], 1e-15, 1e-15, "sampled dK")
        _close(dVs, dV[kr], 1e-15, 1e-15, "sampled dV")
        _close(Ds, D, 1e-15, 1e-15, "sampled D")


# --------------------------------------------------------------------------
# S and P of standard attention: S against a library matrix product, P against
# scipy's softmax with the causal entries removed; P V reproduces O.
# --------------------------------------------------------------------------
def pin_probabilities(orc):
    rng = _rng(12)
    for (n, m, d, causal, scale) in ((6, 9, 4, False, 0.4), (9, 9, 3, True, 0.7),
                                     (8, 5, 5, True, 0.3)):
        Q, K, V = rng.standard_normal((n, d)), rng.standard_normal((m, d)), rng.standard_normal((m, d))
        S, P = orc.probabilities(Q, K, causal, scale)
        ref = scale * (Q @ K.T)
        hidden = np.arange(m)[None, :] > np.arange(n)[:, None] if causal else np.zeros((n, m), bool)
        assert np.all(np.isneginf(S[hidden])), "masked scores must be -inf"
        _close(S[~hidden], ref[~hidden], 1e-14, 1e-14, f"scores causal={causal}")
        soft = scipy.special.softmax(np.where(hidden, -np.inf, ref), axis=1)
        _close(P, soft, 1e-13, 1e-15, f"probabilities causal={causal}")
        assert np.all(P[hidden] == 0.0)
        O, _ = orc.forward(Q, K, V, causal, scale)
        _close(P @ V, O, 1e-13, 1e-14, f"P V = O causal={causal}")


ALL_PINS = [pin_golden, pin_online_stats, pin_softmax_identity_v, pin_causal_row0,
            pin_zero_query, pin_single_key, pin_finite_differences, pin_invariants,
            pin_torch_autograd, pin_tiled_page1, pin_causal_nonsquare, pin_sampled_rows,
            pin_probabilities]
