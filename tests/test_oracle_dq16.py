"""Pins of the oracle's prescaled FP16 dQ accumulator (review page, sec. 3.2
"accumulator leakage", sec. 3.5.3 "Backward pass"): the prescale table from
exponents set by hand, the range the prescale promises on an input built to
reach the bound, the leakage the pages attribute to the sequence-wide
prescale and its removal by causal dQ scaling, and closeness to the float32
accumulator; and of the query-row dS exponents (same page, sec. 3.2: they
remove the leakage inside blocks): exponents by hand and the in-block leak."""
import numpy as np
import pytest

from oracle import flamia_oracle as O


def blocks_with_maxima(rng, lengths, d, exps):
    """[T, 1, d] values whose 32-token blocks (document-aligned) have the
    maximum |x| = 448 * 2^e for the listed exponents, one per block in order."""
    T = sum(lengths)
    x = np.zeros((T, 1, d))
    it = iter(exps)
    s = 0
    for L in lengths:
        for b0 in range(0, L, 32):
            n = min(32, L - b0)
            amax = 448.0 * 2.0 ** next(it)
            blk = rng.uniform(-0.5, 0.5, size=(n, d)) * amax
            blk[rng.integers(n), rng.integers(d)] = amax
            x[s + b0:s + b0 + n, 0] = blk
        s += L
    return x


def test_bound_constant():
    # 16 d 448^3 = 92,073,361,408 (d = 64): 2^36 < it < 2^37; twice that for d = 128
    assert 2 ** 36 < 16 * 64 * 448 ** 3 < 2 ** 37
    assert O.dq16_bound_log2(64) == 37 and O.dq16_bound_log2(128) == 38


def test_prescale_by_hand():
    # documents of 40 and 30 tokens: blocks [0,32) [32,40) | [40,70)
    rng = np.random.default_rng(1)
    L, d = [40, 30], 64
    q = rng.normal(size=(70, 1, d))
    v = blocks_with_maxima(rng, L, d, [-3, 1, -2])
    k = blocks_with_maxima(rng, L, d, [0, -5, 2])
    do = blocks_with_maxima(rng, L, d, [-1, -4, 3])
    qz = O.Quantized(q, k, v, do, [0, 40, 70])
    assert list(qz.vs[0, [0, 32, 40]].astype(int) - 127) == [-3, 1, -2]
    # causal: e_dO + running max e_V + running max e_K, p = 15 - 37 - E
    want = np.array([-18] * 32 + [-19] * 8 + [-25] * 30)   # E = -4, -3, 3
    assert np.array_equal(O.dq_prescale(qz, 0, "causal"), want)
    # non-causal call: maxima over the whole document
    want_nc = np.array([-22] * 32 + [-19] * 8 + [-25] * 30)  # E = 0, -3, 3
    assert np.array_equal(O.dq_prescale(qz, 0, "causal", causal=False), want_nc)
    # sequence-wide: max e_dO 3 + max e_V 1 + max e_K 2
    assert np.array_equal(O.dq_prescale(qz, 0, "sequence"), np.full(70, -28))


def test_prescale_keeps_the_worst_case_in_range():
    # every element of dO, V, K at its block maximum with signs that make each
    # term of dQ = sum_j dS_ij K_j add up: V rows alternate in sign, K rows
    # follow V's sign, and Q = 0 spreads P evenly; |dQ| reaches ~ d 448^3 2^E
    d, L = 64, 256
    a, b, c = -2, 1, -3
    sgn = np.where(np.arange(L) % 2 == 0, 1.0, -1.0)
    q = np.zeros((L, 1, d))
    do = np.full((L, 1, d), 448.0 * 2.0 ** a)
    v = sgn[:, None, None] * np.full((L, 1, d), 448.0 * 2.0 ** b)
    k = sgn[:, None, None] * np.full((L, 1, d), 448.0 * 2.0 ** c)
    qz = O.Quantized(q, k, v, do, [0, L])
    dh = qz.dochead(0, 0)
    rows = np.arange(L)
    o, lse2, _, _ = O.fwd_rows(dh, rows, 1.0)
    D = (dh.do * np.ldexp(1.0, dh.edo)[:, None] * O.bf16_round(o)).sum(axis=1)
    for mode in ("causal", "sequence"):
        p = O.dq_prescale(qz, 0, mode)
        assert np.all(p == 15 - 37 - (a + b + c))
        _, acc = O.dq_fp16_rows(dh, rows, lse2, D, 1.0, p, return_acc=True)
        top = np.abs(acc).max()
        assert np.isfinite(acc).all() and 2.0 ** 10 <= top <= 2.0 ** 15


@pytest.fixture(scope="module")
def mix():
    rng = np.random.default_rng(7)
    lengths = [300, 1, 129, 17, 270, 33]
    T, H, d = sum(lengths), 2, 64
    cu = np.concatenate([[0], np.cumsum(lengths)])
    x = {n: rng.normal(size=(T, H, d)) for n in ("q", "k", "v", "do")}
    x["k"][:, :, 5] *= 20.0  # an outlier channel
    return x, cu, 1.0 / np.sqrt(d)


def run(x, cu, scale, mode):
    return O.attention(x["q"], x["k"], x["v"], x["do"], cu, scale, dq_accum=mode)


def test_fp16_accumulator_close_to_float32(mix):
    x, cu, scale = mix
    ref = run(x, cu, scale, "fp32")
    for mode in ("fp16_sequence", "fp16_causal"):
        r = run(x, cu, scale, mode)
        assert O.cosine(r["dQ"], ref["dQ"]) >= 0.99999
        for h in range(2):
            err = np.abs(r["dQ"][:, h] - ref["dQ"][:, h]).max() / np.abs(ref["dQ"][:, h]).max()
            assert err <= 2e-3, (mode, h, err)
        for n in ("O", "dK", "dV"):  # untouched by the dQ accumulator
            assert np.array_equal(r[n], ref[n])


def test_causal_scaling_removes_the_sequence_dependence(mix):
    # a large later token (block 7 of the first document) must not change the
    # dQ rows of earlier blocks; with the sequence-wide prescale it rounds them
    # differently (review page, sec. 3.2 "accumulator leakage")
    x, cu, scale = mix
    y = {n: t.copy() for n, t in x.items()}
    y["v"][250] *= 64.0
    y["k"][250] *= 64.0
    early = slice(0, 224)
    for mode, same in (("fp32", True), ("fp16_causal", True), ("fp16_sequence", False)):
        a, b = run(x, cu, scale, mode), run(y, cu, scale, mode)
        assert np.array_equal(a["dQ"][early], b["dQ"][early]) == same, mode
    # ... while the late rows themselves change in every mode
    a, b = run(x, cu, scale, "fp16_causal"), run(y, cu, scale, "fp16_causal")
    assert not np.array_equal(a["dQ"][250:300], b["dQ"][250:300])


def test_row_ds_exponents_by_hand():
    # one 2 x 32 dS block: the block rule gives both rows the large row's
    # exponent, the row rule gives each row its own.  E4M3 keeps 3 mantissa
    # bits over its normal range, so a shared exponent only costs precision
    # where it pushes a row below 2^-6 (the subnormals): here by 2^16.
    dS = np.zeros((2, 32))
    dS[0, :] = 1.0 + np.arange(32) / 64.0       # row max 1.484 -> exponent -8
    dS[1, 5] = 1.5 * 2.0 ** 16                  # row max 98304 -> exponent 8
    blk = O._block_quantize_dS(dS, 0, 0)
    row = O._row_quantize_dS(dS, 0)
    assert O.roundup_exponent(np.array([1.484375]))[0] == -8
    assert O.roundup_exponent(np.array([1.5 * 2.0 ** 16]))[0] == 8
    assert np.array_equal(row[0], O.e4m3_decode(O.e4m3_encode(dS[0] * 2.0 ** 8)) * 2.0 ** -8)
    assert np.array_equal(blk[0], O.e4m3_decode(O.e4m3_encode(dS[0] * 2.0 ** -8)) * 2.0 ** 8)
    assert np.array_equal(row[1], blk[1])
    # row 0: within 1/16 relative with its own exponent, subnormal steps of
    # 2^-9 x 2^8 = 1/2 with the shared one
    assert np.abs(row[0] - dS[0]).max() <= dS[0].max() / 16
    assert np.abs(blk[0] - dS[0]).max() >= 0.2


def test_row_ds_exponents_remove_the_in_block_leak(mix):
    # a later query row in the same 32-row block as earlier rows (row 40 of the
    # first document, block [32, 64)): with the block exponents its dO moves
    # the dS exponent that the earlier rows' dQ is rounded with; with query-row
    # exponents only the dO block exponent still links them (the per-token
    # operand scales would remove that), which here shifts a few dO values of
    # rows 32..39 by less than any dS rounding step: their dQ keeps every bit
    x, cu, scale = mix
    y = {n: t.copy() for n, t in x.items()}
    y["do"][40] *= 64.0
    early = slice(32, 40)
    for ds_rows, same in ((False, False), (True, True)):
        a = O.attention(x["q"], x["k"], x["v"], x["do"], cu, scale, ds_rows=ds_rows)
        b = O.attention(y["q"], y["k"], y["v"], y["do"], cu, scale, ds_rows=ds_rows)
        assert np.array_equal(a["dQ"][early], b["dQ"][early]) == same, ds_rows
        assert np.array_equal(a["dQ"][:32], b["dQ"][:32])  # other blocks: never
    r = O.attention(x["q"], x["k"], x["v"], x["do"], cu, scale, ds_rows=True)
    f = O.attention(x["q"], x["k"], x["v"], x["do"], cu, scale)
    assert O.cosine(r["dQ"], f["dQ"]) >= 0.9999
    assert np.array_equal(r["dK"], f["dK"]) and np.array_equal(r["dV"], f["dV"])
