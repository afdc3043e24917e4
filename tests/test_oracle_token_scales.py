"""Pins of the oracle's per-token operand scales (review page, sec. 3.2: with
per-token operand scales and query-row dS exponents a future token changes
no earlier output, even inside its own 32-token block).

* the per-token quantiser is the block quantiser with every token its own
  document (a reduction to the pinned block path);
* where every token of a block has the same exponent, every fold factor is 1
  and the token mode equals the block mode with query-row dS exponents, bit
  for bit (pins the folds' bookkeeping: which exponent multiplies what);
* the in-block leakage probe: perturbing token t leaves every earlier row's O,
  LSE and dQ bit for bit, including the rows of t's own block, under each of
  Q, K, V and dO; the block mode moves them (negative control);
* planted mistakes in a copy of the oracle (the V fold over the whole key
  block instead of the keys a row sees; dQ's dS without the K fold) make the
  probe fail;
* the token mode stays as close to exact attention as the block mode.
"""
import os
import types

import numpy as np
import pytest

from oracle import flamia_oracle as O

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle",
                          "flamia_oracle.py")
NAMES = ("q", "k", "v", "do")


def inputs(L=200, H=1, d=64, seed=3):
    rng = np.random.default_rng(seed)
    x = {n: rng.standard_normal((L, H, d)) for n in NAMES}
    for n in x:
        x[n][:, :, 3] *= 8.0
    return x


def run(mod, x, group, cu=None, **kw):
    L = x["q"].shape[0]
    return mod.attention(*[x[n] for n in NAMES], cu or [0, L], 1.0 / 8.0, group=group, **kw)


def test_token_quantiser_is_the_block_quantiser_on_one_token_documents():
    x = inputs(L=100, H=3)["k"]
    c1, s1 = O.quantize_tokenblock(x, [0, 40, 100], group="token")
    c2, s2 = O.quantize_tokenblock(x, list(range(101)), group="block")
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)
    # and each byte is the round-up exponent of that token's own maximum
    e = O.roundup_exponent(np.abs(x).max(axis=2)).T + 127
    assert np.array_equal(s1, e.astype(np.uint8))


def test_equal_exponents_reduce_to_the_block_mode():
    # every token of every tensor has its largest magnitude exactly 1.5 (same
    # per-token exponent across each block): all fold factors are 1
    x = inputs(L=150, H=2)
    for n in x:
        y = np.clip(x[n], -1.0, 1.0)
        y[:, :, 7] = 1.5
        x[n] = y
    for causal in (True, False):
        rt = run(O, x, "token", cu=[0, 70, 150], causal=causal)
        rb = run(O, x, "block", cu=[0, 70, 150], causal=causal, ds_rows=True)
        for n in ("O", "lse", "dQ", "dK", "dV", "D"):
            assert np.array_equal(rt[n], rb[n]), (n, causal)


def probe(mod, group, t=150, names=NAMES):
    """The rows before token t (whose block starts at 128) that change under a
    perturbation of token t, per perturbed tensor."""
    x = inputs()
    base = run(mod, x, group)
    moved = {}
    for name in names:
        y = {n: v.copy() for n, v in x.items()}
        y[name][t] *= 1000.0
        y[name][t, :, 5] += 50.0
        r = run(mod, y, group)
        moved[name] = [what for what, a, b in (("O", r["O"][:t], base["O"][:t]),
                                                ("lse", r["lse"][:, :t], base["lse"][:, :t]),
                                                ("dQ", r["dQ"][:t], base["dQ"][:t]))
                       if not np.array_equal(a, b)]
    return moved


def test_in_block_leakage_probe_token_scales_bitwise():
    assert probe(O, "token") == {n: [] for n in NAMES}


def test_in_block_leakage_probe_block_mode_leaks():
    moved = probe(O, "block")
    for n in NAMES:
        assert moved[n], n   # the shared block exponents let token t reach rows 128..149


def mutated(old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("flamia_oracle_mutant")
    exec(compile(src.replace(old, new), "flamia_oracle_mutant", "exec"), mod.__dict__)
    return mod


def test_planted_fold_over_the_whole_block_leaks():
    mod = mutated("EV = _visible_block_max(dh.ev, rows, cols, dh.causal)",
                  "EV = _visible_block_max(dh.ev, rows, cols, False)")
    assert probe(mod, "token", names=("v",))["v"]


def test_planted_dq_without_the_k_fold_leaks():
    mod = mutated("dQ = dSq @ dh.k[cols]",
                  "dQ = dSk @ (dh.k[cols] * np.ldexp(1.0, dh.ek[cols])[:, None])")
    assert "dQ" in probe(mod, "token", names=("do",))["do"]


def test_token_scales_as_close_to_exact_attention():
    x = inputs()
    ex = O.attention(*[x[n] for n in NAMES], [0, 200], 1.0 / 8.0, quant=False)
    rb, rt = run(O, x, "block"), run(O, x, "token")
    for n in ("O", "dQ", "dK", "dV"):
        cb, ct = O.cosine(rb[n], ex[n]), O.cosine(rt[n], ex[n])
        assert ct >= cb - 5e-4 and ct >= 0.98, (n, cb, ct)


def test_sampled_rows_follow_the_token_mode():
    x = inputs(L=160)
    full = run(O, x, "token")
    qz = O.Quantized(*[x[n] for n in NAMES], [0, 160], group="token")
    res = O.sampled_rows(qz, 0, 0, 1.0 / 8.0, qblocks=[0, 3], kblocks=[1, 4])
    for qb in (0, 3):
        rows = slice(32 * qb, 32 * qb + 32)
        np.testing.assert_allclose(res["O"][qb], full["O"][rows, 0], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(res["dQ"][qb], full["dQ"][rows, 0], rtol=1e-9, atol=1e-12)
    for kb in (1, 4):
        rows = slice(32 * kb, 32 * kb + 32)
        np.testing.assert_allclose(res["dK"][kb], full["dK"][rows, 0], rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(res["dV"][kb], full["dV"][rows, 0], rtol=1e-9, atol=1e-12)
