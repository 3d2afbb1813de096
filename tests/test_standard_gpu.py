"""The materialised standard-attention path (fa_standard_forward: S and P
written to memory as bf16, then O = P V) against the fp64 oracle.

The oracle gives the exact S, P, O and L. The path rounds S and P to bf16 on
purpose (they are the n x m matrices the pages' standard implementation stores),
so each output is checked against a bound derived from those roundings, per
row i (Delta_i bounds the stored scores' error):
  S    |S_gpu - S| <= 2^-8 |S| + 1e-4           (bf16 rounding of the fp32 score)
  L    |L_gpu - L| <= Delta_i = 2^-8 max_j |S_ij| + 1e-4 (logsumexp is 1-Lipschitz)
  P    |P_gpu - P| <= P (e^(2 Delta_i) (1 + 2^-8) - 1) + 1e-6
                                                (softmax of perturbed scores, then
                                                 bf16 rounding of each weight)
  O    |O_gpu - O| <= E (1 + 2^-8) + 2^-8 |O| + 1e-5,
       E = (e^(2 Delta_i) (1 + 2^-8) - 1) sum_j P_ij |V_jc|
Masked entries of P and the padding columns (past m) must be exactly 0."""
import numpy as np
import pytest
import torch

import exact_io_aware_27_gb300 as fa
import oracle
from exact_io_aware_27_gb300 import inputs as wl

pytestmark = pytest.mark.gpu

U = 2.0 ** -8  # half a bf16 ulp, relative


@pytest.fixture(scope="module", autouse=True)
def _built():
    fa.build()
    oracle.build()


def check_standard(Q, K, V, causal, scale=None):
    B, H, n, d = Q.shape
    m = K.shape[2]
    q, k, v = (t.cuda() for t in (Q, K, V))
    O, L, S, P = fa.fa_standard_forward(q, k, v, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.api.FA_OK
    Sg, Pg = S.double().cpu().numpy(), P.double().cpu().numpy()
    Og, Lg = O.double().cpu().numpy(), L.double().cpu().numpy()
    worst = {"S": 0.0, "P": 0.0, "O": 0.0, "L": 0.0}
    for b in range(B):
        for h in range(H):
            qh, kh, vh = (t[b, h].double().numpy() for t in (Q, K, V))
            S_r, P_r = oracle.probabilities(qh, kh, causal, scale)
            O_r, L_r = oracle.forward(qh, kh, vh, causal, scale)
            PV_abs, _ = oracle.forward(qh, kh, np.abs(vh), causal, scale)
            vis = np.isfinite(S_r)
            s_abs = np.where(vis, np.abs(S_r), 0.0)
            delta = U * s_abs.max(axis=1) + 1e-4                    # per row
            grow = np.exp(2 * delta) * (1 + U) - 1
            # padding columns are 0 in both matrices, masked weights are exactly 0
            assert np.all(Pg[b, h, :, m:] == 0) and np.all(Sg[b, h, :, m:] == 0)
            assert np.all(Pg[b, h, :, :m][~vis] == 0)
            # the stored S holds every score, masked or not (the mask is the softmax's)
            S_all = S_r if not causal else oracle.probabilities(qh, kh, False, scale)[0]
            err_s = np.abs(Sg[b, h, :, :m] - S_all)
            assert np.all(err_s <= U * np.abs(S_all) + 1e-4), f"S error {err_s.max():.3e}"
            err_p = np.abs(Pg[b, h, :, :m] - P_r)
            assert np.all(err_p <= P_r * grow[:, None] + 1e-6), f"P error {err_p.max():.3e}"
            err_l = np.abs(Lg[b, h] - L_r)
            assert np.all(err_l <= delta + 1e-5), f"L error {err_l.max():.3e}"
            E = grow[:, None] * PV_abs
            err_o = np.abs(Og[b, h] - O_r)
            assert np.all(err_o <= E * (1 + U) + U * np.abs(O_r) + 1e-5), f"O error {err_o.max():.3e}"
            for key, e in (("S", err_s.max()), ("P", err_p.max()), ("O", err_o.max()),
                           ("L", err_l.max())):
                worst[key] = max(worst[key], float(e))
    return worst


STANDARD = [
    # (B, H, n, m, d, causal)
    (1, 1, 128, 128, 64, False),
    (1, 1, 128, 128, 64, True),
    (1, 2, 1024, 1024, 64, True),
    (2, 3, 127, 129, 128, False),
    (2, 3, 129, 127, 128, True),
    (1, 1, 1000, 3000, 64, False),
    (1, 1, 77, 300, 128, True),
    (1, 1, 200, 77, 64, True),
    (1, 1, 1, 1, 64, False),
    (1, 2, 300, 200, 96, True),
    (2, 2, 70, 70, 16, True),
    (1, 1, 4096, 4096, 128, True),
]


@pytest.mark.parametrize("B,H,n,m,d,causal", STANDARD)
def test_standard_matches_oracle(B, H, n, m, d, causal):
    Q, K, V, _ = wl.attention_inputs(B, H, n, m, d, seed=8100 + n + 3 * m + d, qk_std=1.0)
    check_standard(Q, K, V, causal)


def test_standard_peaked_scores_custom_scale():
    # Q, K ~ 3 N(0,1) with scale 0.05: scores spread over many units, where the
    # bf16 score matrix costs the most accuracy (the bounds grow with max |S|)
    Q, K, V, _ = wl.attention_inputs(1, 2, 300, 500, 128, seed=8200, qk_std=3.0)
    for causal in (False, True):
        check_standard(Q, K, V, causal, scale=0.05)


def test_standard_and_flash_agree_within_the_standard_bound():
    # the same inputs through both paths: O of the tiled path (fp32 scores never
    # rounded) is the more accurate one; both are within the standard bound
    Q, K, V, _ = wl.attention_inputs(1, 4, 512, 512, 128, seed=8300, qk_std=1.0)
    q, k, v = (t.cuda() for t in (Q, K, V))
    O_s, L_s, _, _ = fa.fa_standard_forward(q, k, v, True)
    O_f, L_f = fa.fa_forward(q, k, v, True)
    torch.cuda.synchronize()
    O_r, L_r = oracle.forward(*(t.double().numpy() for t in (Q, K, V)), True)
    e_std = float(np.abs(O_s.double().cpu().numpy() - O_r).max())
    e_fl = float(np.abs(O_f.double().cpu().numpy() - O_r).max())
    assert e_fl <= 1e-2 and e_fl <= e_std + 2e-3, (e_fl, e_std)


def test_standard_argument_errors():
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_standard_forward(q, q, q, S=torch.empty(1, 1, 8, 8, dtype=torch.bfloat16, device="cuda"))
    assert fa.fa_standard_matrix_bytes(1, 1, 8, 8) == 8 * 64 * 2
    assert fa.fa_standard_matrix_bytes(2, 3, 5, 65) == 2 * 3 * 5 * 128 * 2
    assert fa.fa_standard_matrix_bytes(0, 1, 8, 8) == 0
