"""Pins of the dS rounded-to-zero count (review page, sec. 3.3: with a poorly
set scale small dS elements round to zero; the ablation of sec. 4 takes the
fraction rounded to zero as the diagnostic, 0.4% with the method's scale
against 29% with an oversized one)."""
import numpy as np

from oracle import flamia_oracle as O


def test_counts_by_hand():
    # one 32x32 dS block with largest value 448 (exponent 0): 2^-8 is two
    # E4M3 subnormal steps (2^-9 each) and stays; 2^-11 is a quarter step and
    # rounds to zero
    dS = np.zeros((32, 32))
    dS[0, 0] = 448.0
    dS[1, 0] = 2.0 ** -8
    dS[1, 1] = 2.0 ** -11
    q = O._block_quantize_dS(dS, 0, 0)
    assert q[0, 0] == 448.0 and q[1, 0] == 2.0 ** -8 and q[1, 1] == 0.0
    # an exponent larger by 2 makes 2^-8 exactly half a step: ties to even, zero
    q2 = O._block_quantize_dS(dS, 0, 0, extra=2)
    assert q2[1, 0] == 0.0 and q2[0, 0] == 448.0


def test_fraction_small_with_the_round_up_scale_and_grows_when_oversized():
    rng = np.random.default_rng(5)
    L, d = 256, 64
    x = {n: rng.standard_normal((L, 1, d)) for n in ("q", "k", "v", "do")}
    qz = O.Quantized(x["q"], x["k"], x["v"], x["do"], [0, L])
    nz, z = O.ds_zero_counts(qz, 1.0 / 8.0)
    nz2, z2 = O.ds_zero_counts(qz, 1.0 / 8.0, extra=6)
    assert nz == nz2 == L * (L + 1) // 2   # every visible dS is nonzero here
    assert z / nz < 0.02
    assert z2 / nz2 > 5 * max(z / nz, 1e-3)
