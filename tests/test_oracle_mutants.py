"""Planted mistakes in copies of the oracle must fail at least one pin.

Each mutant is a textual edit of ``oracle/attention_fp64.cpp`` (a dropped
term, a wrong sign, a wrong index or operand, an off-by-one mask) compiled into
a temporary library. The original source is never modified. This shows that
the pins in ``oracle_pins`` are sharp enough to catch the plausible mistakes a
restatement of the method could contain.
"""
import os

import pytest

import oracle
from tests import oracle_pins

MUTANTS = {
    "dS_sign": ("const double dS = p * (dp - Drow[i]);",
                "const double dS = p * (dp + Drow[i]);"),
    "causal_off_by_one": ("if (causal && j > i) return kNegInf;",
                          "if (causal && j > i + 1) return kNegInf;"),
    "lse_drops_max": ("return mx + std::log(sum);", "return std::log(sum);"),
    "online_drops_rescale": ("l = l * std::exp(m - m_new) + csum;", "l = l + csum;"),
    "dV_wrong_operand": ("dVj[c] += p * dO[i * d + c];", "dVj[c] += p * V[j * d + c];"),
    "dK_drops_scale": ("dKj[c] += scale * dS * Q[i * d + c];", "dKj[c] += dS * Q[i * d + c];"),
    "score_index_reversed": ("acc += Q[i * d + c] * K[j * d + c];",
                             "acc += Q[i * d + c] * K[j * d + (d - 1 - c)];"),
    "D_drops_P": ("Di += p * dp;", "Di += dp;"),
    "dQ_wrong_operand": ("dQi[c] += scale * dS * K[j * d + c];",
                         "dQi[c] += scale * dS * Q[i * d + c];"),
    "O_wrong_weight": ("Oi[c] += p * V[j * d + c];", "Oi[c] += std::exp(s[j]) * V[j * d + c];"),
    "P_unnormalised": ("std::exp(si[j] - Li);", "std::exp(si[j]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(before) >= 1, f"mutation site for {name} not found"
    mutated = tmp_path / f"mutant_{name}.cpp"
    mutated.write_text(src.replace(before, after))  # every occurrence
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / f"lib_{name}.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
    os.remove(lib)
