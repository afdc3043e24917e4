"""Pins of the oracle's quantised probability path against a hand-derived case.

The forward's E4M3 probability operand (integer running row maximum, the 2^8
factor, RNE to E4M3), the backward's dV operand RNE_E4M3(2^8 P) and D taken
from the forward's BF16 output are checked against values worked out by hand
in ``golden/probability_path.txt`` (review page, sec. 1.2, 3.1 and 3.3).

Each plausible mistake in those steps is then planted in a copy of the oracle
(its source with one line changed, loaded as a separate module on the CPU),
and the pin must fail on it: dropping the E4M3 rounding of P^ or of P^b, a
floor instead of a ceiling for the row maximum, 2^7 instead of 2^8, and the
exact O instead of its BF16 rounding in D.
"""
import math
import os
import types

import numpy as np
import pytest

from oracle import flamia_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "probability_path.txt")
ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle",
                          "flamia_oracle.py")

Q = [[448, 0], [448, 0], [448, 0]]
K = [[448, 0], [224, 0], [-416, 0]]
V = [[448, -64], [96, 320], [-288, 176]]
DO = [[448, 32], [-160, 208], [80, -112]]
SM_SCALE = 6.825 * math.log(2.0) / 448.0 ** 2


def load_golden():
    rows = {}
    with open(GOLDEN) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, i, *vals = line.split()
            rows.setdefault(name, {})[int(i)] = [float(v) for v in vals]
    return {n: np.array([r[i] for i in sorted(r)]) for n, r in rows.items()}


def run(mod):
    t = lambda a: np.asarray(a, dtype=np.float64)[:, None, :]
    return mod.attention(t(Q), t(K), t(V), t(DO), [0, 3], SM_SCALE, quant=True)


def check_pins(mod):
    """Raises AssertionError (or the oracle's own error) unless every pinned
    quantity matches the hand derivation."""
    g = load_golden()
    r = run(mod)
    np.testing.assert_allclose(r["O"][:, 0], g["O"], rtol=1e-12)
    np.testing.assert_array_equal(r["O_bf16"][:, 0], g["O_bf16"])
    np.testing.assert_allclose(r["lse"][0], g["LSE"][:, 0], rtol=1e-12)
    np.testing.assert_allclose(r["D"][0], g["D"][:, 0], rtol=1e-12)
    np.testing.assert_allclose(r["dV"][:, 0], g["dV"], rtol=1e-12)


def test_inputs_quantise_to_themselves():
    """The hand derivation assumes exponent 0 and codes equal to the values."""
    for x in (Q, K, V, DO):
        codes, sbytes = O.quantize_tokenblock(np.asarray(x, float)[:, None, :], [0, 3])
        assert (sbytes == 127).all()
        np.testing.assert_array_equal(O.e4m3_decode(codes)[:, 0], np.asarray(x, float))


def test_probability_path_matches_hand_derivation():
    check_pins(O)


MUTATIONS = {
    "P^ not rounded to E4M3": (
        "ph = e4m3_decode(e4m3_encode(p8)) if quant else p8", "ph = p8"),
    "row maximum rounded down": (
        "m = np.ceil(s.max(axis=1))", "m = np.floor(s.max(axis=1))"),
    "2^7 probability factor": ("P_SCALE_LOG2 = 8", "P_SCALE_LOG2 = 7"),
    "exact O in D": ('o_for_D = out["O_bf16"][s:e, h] if quant else o', "o_for_D = o"),
    "dV operand not rounded to E4M3": (
        "pbh = e4m3_decode(e4m3_encode(pb)) if quant else pb", "pbh = pb"),
}


def mutated_oracle(old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, f"mutation site not found once: {old!r}"
    mod = types.ModuleType("flamia_oracle_mutant")
    exec(compile(src.replace(old, new), "flamia_oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("what", sorted(MUTATIONS))
def test_planted_mistake_fails_the_pin(what):
    mod = mutated_oracle(*MUTATIONS[what])
    with pytest.raises((AssertionError, ValueError)):
        check_pins(mod)
