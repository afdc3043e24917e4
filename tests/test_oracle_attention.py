"""Pins of the oracle's attention forward and backward.

Sources: "FLAMIA ... (jaehun.me review)", sec. 1.2 (forward S, P, O and the
backward dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = dS K, dK = dS^T Q),
sec. 3.3 (D_i = dO_i . O_i equals sum_j P_ij dP_ij in exact arithmetic), sec.
3.2 and 4.5 (causal leakage: a masked future token must not change earlier
outputs; tensor-wide scales let one token change all of them), sec. 4.4
(8-bit outputs reach cosine 0.998-0.999 against FP32)."""
import numpy as np
import pytest

from oracle import flamia_oracle as O


def rand(shape, seed, scale=1.0):
    return O.bf16_round(np.random.default_rng(seed).standard_normal(shape) * scale)


def qkvdo(T, H, d, seed=0):
    return [rand((T, H, d), seed + i) for i in range(4)]


# ---------------------------------------------------------------- exact mode

def test_single_token_gives_v():
    q, k, v, do = qkvdo(1, 2, 8)
    r = O.attention(q, k, v, do, [0, 1], 0.3, quant=False)
    assert np.allclose(r["O"], v, rtol=1e-14, atol=0)
    assert np.allclose(r["dV"], do, rtol=1e-14, atol=0)
    assert np.allclose(r["dQ"], 0, atol=1e-15) and np.allclose(r["dK"], 0, atol=1e-15)


def test_zero_keys_give_running_mean_of_v():
    q, k, v, do = qkvdo(50, 1, 8)
    k[:] = 0.0
    r = O.attention(q, k, v, do, [0, 50], 0.3, quant=False)
    want = np.cumsum(v, axis=0) / np.arange(1, 51)[:, None, None]
    assert np.allclose(r["O"], want, rtol=1e-12, atol=1e-14)
    assert np.allclose(r["lse"][0], np.log(np.arange(1, 51)), rtol=1e-12)


def test_one_token_documents():
    q, k, v, do = qkvdo(9, 2, 8)
    r = O.attention(q, k, v, do, list(range(10)), 0.3, quant=False)
    assert np.allclose(r["O"], v, rtol=1e-14)
    assert np.allclose(r["dV"], do, rtol=1e-14)
    assert np.allclose(r["dQ"], 0, atol=1e-15) and np.allclose(r["dK"], 0, atol=1e-15)


def test_gradients_match_central_finite_differences():
    T, H, d = 11, 2, 4
    cu = [0, 6, 11]
    q, k, v, do = qkvdo(T, H, d, seed=5)
    sm = 0.7
    r = O.attention(q, k, v, do, cu, sm, quant=False)

    def loss(qq, kk, vv):
        o = O.attention(qq, kk, vv, None, cu, sm, quant=False, backward=False)["O"]
        return float((o * do).sum())

    h = 1e-6
    for name, g in (("q", r["dQ"]), ("k", r["dK"]), ("v", r["dV"])):
        num = np.zeros_like(g)
        for idx in np.ndindex(*g.shape):
            args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            args[name][idx] += h
            lp = loss(args["q"], args["k"], args["v"])
            args[name][idx] -= 2 * h
            lm = loss(args["q"], args["k"], args["v"])
            num[idx] = (lp - lm) / (2 * h)
        rel = np.abs(num - g).max() / np.abs(g).max()
        assert rel <= 1e-6, (name, rel)


def test_D_identity_exact_and_quantized():
    T, H, d = 96, 1, 16
    q, k, v, do = qkvdo(T, H, d, seed=9)
    cu = [0, 96]
    for quant, tol in ((False, 1e-12), (True, 0.05)):
        r = O.attention(q, k, v, do, cu, 0.25, quant=quant)
        dh = (r["quantized"].dochead(0, 0) if quant else O.exact_dochead(q, k, v, do, cu, 0, 0))
        rows = np.arange(T)
        lse2 = r["lse"][0] / O.LN2
        s = O._scores(dh, rows, rows, 0.25)
        P = np.exp2(s - lse2[:, None])
        dohat = dh.do * np.ldexp(1.0, dh.edo)[:, None]
        vhat = dh.v * np.ldexp(1.0, dh.ev)[:, None]
        rhs = (P * (dohat @ vhat.T)).sum(axis=1)
        err = np.abs(r["D"][0] - rhs).max() / np.abs(rhs).max()
        assert err <= tol, (quant, err)


# ---------------------------------------------------------------- quantised mode

@pytest.mark.parametrize("d", [64, 128])
def test_quantized_cosine_against_exact_on_plain_inputs(d):
    T, H = 768, 2
    q, k, v, do = qkvdo(T, H, d, seed=11)
    cu = [0, 512, 768]
    rq = O.attention(q, k, v, do, cu, d ** -0.5, quant=True)
    rx = O.attention(q, k, v, do, cu, d ** -0.5, quant=False)
    assert O.cosine(rq["O"], rx["O"]) >= 0.998
    for n in ("O", "dQ", "dK", "dV", "lse", "D"):
        assert O.cosine(rq[n], rx[n]) >= 0.996, n
        # magnitudes too: a dropped constant factor leaves the cosine alone
        rel = np.linalg.norm(rq[n] - rx[n]) / np.linalg.norm(rx[n])
        assert rel <= 0.1, (n, rel)


def test_nvfp4_mixed_scores_cosine():
    T, H, d = 512, 1, 64
    q, k, v, do = qkvdo(T, H, d, seed=12)
    cu = [0, 512]
    rq = O.attention(q, k, v, do, cu, d ** -0.5, quant=True, qk_format="nvfp4")
    rx = O.attention(q, k, v, do, cu, d ** -0.5, quant=False)
    assert 0.98 <= O.cosine(rq["O"], rx["O"]) < 0.9999
    r8 = O.attention(q, k, v, do, cu, d ** -0.5, quant=True)
    assert O.cosine(r8["O"], rx["O"]) > O.cosine(rq["O"], rx["O"])


def test_probability_operand_never_exceeds_448():
    q, k, v, do = qkvdo(256, 1, 32, seed=13)
    qz = O.Quantized(q, k, v, do, [0, 256])
    dh = qz.dochead(0, 0)
    rows = np.arange(256)
    s = O._scores(dh, rows, rows, 1.0)
    m = np.ceil(s.max(axis=1))
    p8 = np.ldexp(np.exp2(s - m[:, None]), 8)
    assert p8.max() <= 256.0


def _perturb(x, t, seed):
    y = x.copy()
    y[t] *= 1000.0
    y[t, :, np.random.default_rng(seed).integers(0, x.shape[2])] += 50.0
    return y


def _probe(group, rule="up"):
    T, H, d = 330, 2, 16
    cu = [0, 200, 330]
    base = qkvdo(T, H, d, seed=21)
    t = 150                                   # block [128, 160) of document 0
    r0 = O.attention(*base, cu, 0.25, quant=True, group=group, rule=rule)
    changed = {}
    for i, name in enumerate(("q", "k", "v", "do")):
        args = list(base)
        args[i] = _perturb(base[i], t, i)
        r1 = O.attention(*args, cu, 0.25, quant=True, group=group, rule=rule)
        early = slice(0, 128)
        changed[name] = {
            "O": not np.array_equal(r0["O"][early], r1["O"][early]),
            "lse": not np.array_equal(r0["lse"][:, early], r1["lse"][:, early]),
            "dQ": not np.array_equal(r0["dQ"][early], r1["dQ"][early]),
            "other_doc": any(not np.array_equal(r0[n][200:], r1[n][200:])
                             for n in ("O", "dQ", "dK", "dV")),
        }
    return changed


def test_leakage_probe_token_block_scales_leak_nothing():
    ch = _probe("block")
    for name, c in ch.items():
        assert not any(c.values()), (name, c)


def test_leakage_probe_has_teeth_with_tensor_wide_scales():
    ch = _probe("tensor")
    assert any(c["O"] or c["dQ"] for c in ch.values())
    assert any(c["other_doc"] for c in ch.values())


def test_floor_rule_clamp_leak_inside_a_block():
    """The clamp mechanism of the worked example: with the floor rule a larger
    future value in the same block unclips an earlier code; with round-up the
    earlier code is unchanged."""
    x = np.zeros((32, 1, 4))
    x[3, 0, 0] = 470.0
    y = x.copy()
    y[20, 0, 1] = 900.0
    for rule, leaks in (("floor", True), ("up", False)):
        cx, sx = O.quantize_tokenblock(x, [0, 32], rule=rule)
        cy, sy = O.quantize_tokenblock(y, [0, 32], rule=rule)
        vx = O.dequantize_tokenblock(cx, sx)[3, 0, 0]
        vy = O.dequantize_tokenblock(cy, sy)[3, 0, 0]
        assert (vx != vy) == leaks, rule


def test_sampled_rows_equal_full_attention():
    T, H, d = 300, 1, 16
    cu = [0, 100, 300]
    q, k, v, do = qkvdo(T, H, d, seed=31)
    r = O.attention(q, k, v, do, cu, 0.25, quant=True)
    qz = r["quantized"]
    res = O.sampled_rows(qz, 1, 0, 0.25, qblocks=[0, 3, 6], kblocks=[0, 5, 6])
    s = 100
    for qb in (0, 3, 6):
        rows = slice(s + 32 * qb, min(s + 32 * qb + 32, 300))
        assert np.allclose(res["O"][qb], r["O"][rows, 0], rtol=1e-12, atol=1e-14)
        assert np.allclose(res["lse"][qb], r["lse"][0, rows], rtol=1e-12)
        assert np.allclose(res["dQ"][qb], r["dQ"][rows, 0], rtol=1e-10, atol=1e-13)
    for kb in (0, 5, 6):
        rows = slice(s + 32 * kb, min(s + 32 * kb + 32, 300))
        assert np.allclose(res["dK"][kb], r["dK"][rows, 0], rtol=1e-10, atol=1e-13)
        assert np.allclose(res["dV"][kb], r["dV"][rows, 0], rtol=1e-10, atol=1e-13)


# ------------------------------------------------------------ non-causal mode
# (review page, sec. 4.8: the non-causal packed call; every query sees every
# key of its own document)

def _softmax_attention(q, k, v, do, scale):
    """Plain dense softmax attention of one document and its gradients,
    written out from the definition (float64)."""
    S = scale * q @ k.T
    P = np.exp(S - S.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    o = P @ v
    dP = do @ v.T
    dS = P * (dP - (dP * P).sum(axis=1, keepdims=True))
    return o, scale * dS @ k, scale * dS.T @ q, P.T @ do


def test_noncausal_exact_equals_dense_softmax():
    q, k, v, do = qkvdo(45, 2, 16, seed=31)
    cu = [0, 20, 45]
    r = O.attention(q, k, v, do, cu, 0.37, quant=False, causal=False)
    for b in range(2):
        s, e = cu[b], cu[b + 1]
        for h in range(2):
            o, dq, dk, dv = _softmax_attention(q[s:e, h], k[s:e, h], v[s:e, h], do[s:e, h], 0.37)
            for got, want in ((r["O"], o), (r["dQ"], dq), (r["dK"], dk), (r["dV"], dv)):
                assert np.allclose(got[s:e, h], want, rtol=1e-10, atol=1e-12)


def test_noncausal_outputs_ignore_key_order():
    # permuting the keys (with their values) of a document leaves every
    # non-causal output row unchanged; a causal mask would not
    q, k, v, do = qkvdo(40, 1, 16, seed=33)
    perm = np.random.default_rng(1).permutation(40)
    a = O.attention(q, k, v, do, [0, 40], 0.25, quant=False, causal=False)
    b = O.attention(q, k[perm], v[perm], do, [0, 40], 0.25, quant=False, causal=False)
    assert np.allclose(a["O"], b["O"], rtol=1e-12, atol=1e-14)
    assert np.allclose(a["dQ"], b["dQ"], rtol=1e-10, atol=1e-13)
    assert np.allclose(a["dK"][perm], b["dK"], rtol=1e-10, atol=1e-13)
    c = O.attention(q, k[perm], v[perm], do, [0, 40], 0.25, quant=False)
    assert not np.allclose(a["O"], c["O"])


def test_noncausal_quantised_tracks_exact():
    q, k, v, do = qkvdo(200, 2, 64, seed=35)
    cu = [0, 77, 200]
    ex = O.attention(q, k, v, do, cu, 0.125, quant=False, causal=False)
    qz = O.attention(q, k, v, do, cu, 0.125, causal=False)
    # the method's own level against FP32 (the pages' summary: dQ cosine
    # 0.9979 for MXFP8): O, dV above 0.998, dQ, dK above 0.997
    for n, bar in (("O", 0.998), ("dV", 0.998), ("dQ", 0.997), ("dK", 0.997)):
        assert O.cosine(qz[n], ex[n]) > bar, n
    # documents stay isolated: the first document's rows equal a call on it alone
    one = O.attention(*[x[:77] for x in (q, k, v, do)], [0, 77], 0.125, causal=False)
    for n in ("O", "dQ", "dK", "dV"):
        assert np.array_equal(qz[n][:77], one[n]), n


def test_noncausal_sampled_rows_match_full():
    q, k, v, do = qkvdo(96, 1, 32, seed=37)
    full = O.attention(q, k, v, do, [0, 96], 0.2, causal=False)
    res = O.sampled_rows(full["quantized"], 0, 0, 0.2, [1], [0, 2], causal=False)
    assert np.allclose(res["O"][1], full["O"][32:64, 0], rtol=1e-12, atol=1e-14)
    assert np.allclose(res["dQ"][1], full["dQ"][32:64, 0], rtol=1e-9, atol=1e-12)
    assert np.allclose(res["dK"][0], full["dK"][0:32, 0], rtol=1e-9, atol=1e-12)
    assert np.allclose(res["dV"][2], full["dV"][64:96, 0], rtol=1e-9, atol=1e-12)


# ------------------------------------------------- grouped-query attention
# (K / V with H_kv heads shared by groups of H / H_kv query heads)

@pytest.mark.parametrize("quant", [False, True])
def test_gqa_equals_mha_on_repeated_kv(quant):
    T, H, Hkv, d = 80, 6, 2, 32
    rng = np.random.default_rng(41)
    q, do = [O.bf16_round(rng.standard_normal((T, H, d))) for _ in range(2)]
    k, v = [O.bf16_round(rng.standard_normal((T, Hkv, d))) for _ in range(2)]
    cu = [0, 33, 80]
    g = O.attention(q, k, v, do, cu, 0.2, quant=quant)
    rep = lambda x: np.repeat(x, H // Hkv, axis=1)   # head h -> kv head h // 3
    m = O.attention(q, rep(k), rep(v), do, cu, 0.2, quant=quant)
    assert np.array_equal(g["O"], m["O"]) and np.array_equal(g["dQ"], m["dQ"])
    assert np.array_equal(g["lse"], m["lse"])
    for n in ("dK", "dV"):
        want = m[n].reshape(T, Hkv, H // Hkv, d).sum(axis=2)
        assert g[n].shape == (T, Hkv, d)
        assert np.allclose(g[n], want, rtol=1e-12, atol=1e-14 * np.abs(want).max()), n


def test_gqa_single_kv_head_gradients_sum_over_queries():
    # one K / V head for all query heads: dK, dV are the sums over the heads
    T, H, d = 40, 4, 16
    rng = np.random.default_rng(43)
    q, do = [O.bf16_round(rng.standard_normal((T, H, d))) for _ in range(2)]
    k, v = [O.bf16_round(rng.standard_normal((T, 1, d))) for _ in range(2)]
    g = O.attention(q, k, v, do, [0, T], 0.3, quant=False)
    per_head = [O.attention(q[:, h:h + 1], k, v, do[:, h:h + 1], [0, T], 0.3, quant=False)
                for h in range(H)]
    for n in ("dK", "dV"):
        assert np.allclose(g[n][:, 0], sum(r[n][:, 0] for r in per_head), rtol=1e-12, atol=1e-14)
