"""Pins of the oracle's number formats and exponent rules against facts the
formats fix by definition (OCP FP8 E4M3FN, E2M1, E8M0) and brute force.

Sources: "FLAMIA ... (jaehun.me review)", sec. 2 (E4M3 maximum 448, floor rule)
and sec. 3.2 (round-up exponents: the scaled maximum never exceeds 448)."""
import os

import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)].astype(np.float64)


def test_e4m3_table_landmarks():
    t = O.E4M3_TABLE
    assert t[0x7E] == 448.0                   # largest finite
    assert t[0x38] == 1.0                     # exponent field 7 = bias
    assert t[0x08] == 2.0 ** -6               # smallest normal
    assert t[0x01] == 2.0 ** -9               # smallest subnormal
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)           # codes 0..126 increase strictly
    assert np.all(t[0x80:0xFF] == -pos)       # sign-magnitude


def _brute_force_rne(values, table_pos):
    """Nearest table value, ties to the code with an even last bit."""
    a = np.abs(values)[:, None]
    dist = np.abs(a - table_pos[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    n = cand.sum(axis=1)
    idx = np.argmax(cand, axis=1)
    two = n == 2
    if np.any(two):
        lo = idx[two]
        idx[two] = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.all(n <= 2)
    return idx | (np.signbit(values).astype(np.int64) << 7)


def test_e4m3_encode_matches_brute_force_on_every_bf16_value():
    v = all_bf16_values()
    v = v[np.abs(v) <= 448.0]
    got = O.e4m3_encode(v).astype(np.int64)
    want = _brute_force_rne(v, O.E4M3_TABLE[:0x7F])
    assert np.array_equal(got, want)


def test_e4m3_exact_midpoints_round_to_even():
    pos = O.E4M3_TABLE[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    got = O.e4m3_encode(mids).astype(np.int64)
    lo = np.arange(0x7E)
    assert np.array_equal(got, np.where(lo % 2 == 0, lo, lo + 1))
    assert O.e4m3_encode(np.array([-0.0, -2.0 ** -11]))[0] == 0x80
    assert O.e4m3_encode(np.array([-2.0 ** -11]))[0] == 0x80
    with pytest.raises(ValueError):
        O.e4m3_encode(np.array([449.0]))
    assert O.e4m3_encode(np.array([1000.0]), saturate=True)[0] == 0x7E


def test_e2m1_table_and_brute_force():
    assert list(O.E2M1_VALUES) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    v = all_bf16_values()
    v = v[np.abs(v) <= 6.0]
    a = np.abs(v)[:, None]
    dist = np.abs(a - O.E2M1_VALUES[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    idx = np.argmax(cand, axis=1)
    two = cand.sum(axis=1) == 2
    idx[two] = np.where(idx[two] % 2 == 0, idx[two], idx[two] + 1)
    want = idx | (np.signbit(v).astype(np.int64) << 3)
    assert np.array_equal(O.e2m1_encode(v).astype(np.int64), want)
    # midpoints 0.25 0.75 1.25 1.75 2.5 3.5 5 go to the even code
    assert list(O.e2m1_decode(O.e2m1_encode(
        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])))) == [0, 1, 1, 2, 2, 4, 4]


def test_e8m0_decode():
    assert O.e8m0_decode(127) == 1.0
    assert O.e8m0_decode(0) == 2.0 ** -127
    assert O.e8m0_decode(254) == 2.0 ** 127


def test_bf16_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(x.astype(np.float64)), ref)


def test_roundup_exponent_never_clips_and_is_minimal():
    v = np.abs(all_bf16_values())
    v = v[(v > 2.0 ** -110) & (v < 2.0 ** 120)]
    e = O.roundup_exponent(v)
    scaled = v * np.ldexp(1.0, -e)
    assert np.all(scaled <= 448.0)            # never clips
    assert np.all(scaled > 224.0)             # one less would clip: minimal
    assert O.roundup_exponent(np.array([0.0]))[0] == -127
    assert O.roundup_exponent(np.array([2.0 ** -130]))[0] == -127


def test_floor_exponent_is_the_ocp_rule():
    assert list(O.floor_exponent(np.array([470.0, 900.0, 1.0, 255.9]))) == [0, 1, -8, -1]


def test_worked_example_golden():
    rows = []
    with open(os.path.join(GOLDEN, "roundup_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    assert len(rows) == 4
    for rule, group, past, e_want, code_want, rec_want in rows:
        vals = np.array([float(g) for g in group.split(",")])
        amax = np.abs(vals).max()
        e = int((O.roundup_exponent if rule == "up" else O.floor_exponent)(np.array([amax]))[0])
        assert e == int(e_want)
        c = O.e4m3_encode(np.array([float(past) * 2.0 ** -e]), saturate=(rule == "floor"))
        assert O.e4m3_decode(c)[0] == float(code_want)
        assert O.e4m3_decode(c)[0] * 2.0 ** e == float(rec_want)


def test_nvfp4_scale_is_smallest_e4m3_at_or_above_amax_over_6():
    v = np.abs(all_bf16_values())
    v = v[v <= 6 * 448.0]
    sc = O.nvfp4_scale_code(v)
    s = O.E4M3_TABLE[sc]
    assert np.all(s >= v / 6.0)
    prev = O.E4M3_TABLE[np.maximum(sc.astype(np.int64) - 1, 0)]
    ok = (sc == 0) | (prev < v / 6.0)
    assert np.all(ok)
    assert O.nvfp4_scale_code(np.array([0.0]))[0] == 0


def test_nvfp4_fp32_division_gives_the_exact_quotient_codes():
    """For every positive E4M3 scale s and every BF16 x with |x| <= 6 s, the
    E2M1 code of the float32 quotient fl32(x / s) equals the code decided by
    exact comparison of x with midpoint * s (a float32 divide never crosses an
    E2M1 rounding midpoint)."""
    v = all_bf16_values()
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    for sc in range(1, 0x7F):
        s = O.E4M3_TABLE[sc]
        x = v[np.abs(v) <= 6.0 * s]
        q32 = (x.astype(np.float32) / np.float32(s)).astype(np.float64)
        got = O.e2m1_encode(q32)
        # exact decision: count midpoints strictly below |x|/s, ties to even
        a = np.abs(x)
        below = (a[:, None] > mids[None, :] * s).sum(axis=1)
        tie = np.any(a[:, None] == mids[None, :] * s, axis=1)
        idx = below.copy()
        idx[tie] = np.where(below[tie] % 2 == 0, below[tie], below[tie] + 1)
        want = idx | (np.signbit(x).astype(np.int64) << 3)
        assert np.array_equal(got.astype(np.int64), want), sc
