"""Pins of the oracle's Hadamard rotation of Q and K.

Source: "FLAMIA ... (jaehun.me review)", sec. 3.4 "Hadamard rotation": the
head-dimension channels of Q and K are mixed by a normalised orthogonal
transform before quantisation; in exact arithmetic dot products are kept and
token positions are not mixed, so no causal dependency appears; it limits how
far one outlier channel sets the scale of a whole block.  The reading fixed
here: the unnormalised Sylvester matrix in float32 butterflies, 1/d folded into
the softmax scale, dQ and dK rotated back."""
import numpy as np
import pytest

from oracle import flamia_oracle as O

scipy_linalg = pytest.importorskip("scipy.linalg")


@pytest.mark.parametrize("d", [1, 2, 4, 8, 64, 128])
def test_matrix_is_the_library_sylvester_matrix(d):
    assert np.array_equal(O.sylvester(d), scipy_linalg.hadamard(d).astype(np.float64))
    h = O.sylvester(d)
    assert np.array_equal(h @ h, d * np.eye(d))


@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_butterflies_equal_the_matrix_product_on_exact_inputs(d):
    # small integers: every float32 partial sum is exact, so the butterfly
    # order cannot show and the result must be x H exactly
    x = np.random.default_rng(d).integers(-64, 64, size=(5, 3, d)).astype(np.float64)
    h = scipy_linalg.hadamard(d).astype(np.float64)
    assert np.array_equal(O.hadamard_fp32(x), x @ h)
    assert np.array_equal(O.hadamard_fp32(O.hadamard_fp32(x)), d * x)


@pytest.mark.parametrize("d", [64, 128])
def test_butterflies_round_in_float32(d):
    rng = np.random.default_rng(7)
    x = O.bf16_round(rng.standard_normal((64, d)) * np.exp(rng.uniform(-8, 8, (64, 1))))
    got = O.hadamard_fp32(x)
    want = x @ scipy_linalg.hadamard(d).astype(np.float64)
    # log2(d) float32 roundings of partial sums bounded by sum |x|
    bound = np.log2(d) * 2.0 ** -24 * np.abs(x).sum(axis=1, keepdims=True)
    assert np.all(np.abs(got - want) <= bound)
    assert np.all(got == got.astype(np.float32))  # float32 values
    # each output is one rounding of a sum of exact terms: not always exact
    assert np.any(got != want)


def _butterflies_loop(x, strides):
    """Element-by-element float32 butterflies in the given stride order."""
    y = [np.float32(v) for v in x]
    for st in strides:
        for i in range(len(y)):
            if i % (2 * st) < st:
                a, b = y[i], y[i + st]
                y[i], y[i + st] = np.float32(a + b), np.float32(a - b)
    return np.array(y, dtype=np.float64)


def test_stride_order_is_increasing():
    # the stage order is a choice (all orders agree in exact arithmetic);
    # find inputs on which the two extreme orders round differently and check
    # that the oracle takes strides 1, 2, 4, ...
    rng = np.random.default_rng(2)
    d = 16
    up, down = [1, 2, 4, 8], [8, 4, 2, 1]
    found = 0
    for _ in range(200):
        x = (rng.standard_normal(d) * np.exp(rng.uniform(-20, 20, d))).astype(np.float32)
        a, b = _butterflies_loop(x, up), _butterflies_loop(x, down)
        if not np.array_equal(a, b):
            found += 1
            assert np.array_equal(O.hadamard_fp32(x[None].astype(np.float64))[0], a)
    assert found > 10


def qkvdo(T, H, d, seed):
    rng = np.random.default_rng(seed)
    return [O.bf16_round(rng.standard_normal((T, H, d))) for _ in range(4)]


@pytest.mark.parametrize("d", [64, 128])
def test_exact_attention_is_unchanged_by_the_rotation(d):
    q, k, v, do = qkvdo(70, 2, d, 3)
    cu = [0, 9, 70]
    a = O.attention(q, k, v, do, cu, 0.125, quant=False)
    b = O.attention(q, k, v, do, cu, 0.125, quant=False, hadamard=True)
    for n in ("O", "dQ", "dK", "dV"):
        assert np.allclose(b[n], a[n], rtol=1e-9, atol=1e-12 * np.abs(a[n]).max()), n
    assert np.allclose(b["lse"], a["lse"], rtol=1e-12)


def test_quantised_rotation_tracks_exact_attention():
    q, k, v, do = qkvdo(128, 2, 64, 5)
    cu = [0, 128]
    ex = O.attention(q, k, v, do, cu, 0.125, quant=False)
    r = O.attention(q, k, v, do, cu, 0.125, quant=True, hadamard=True)
    for n in ("O", "dQ", "dK", "dV"):
        assert O.cosine(r[n], ex[n]) > 0.998, n


def test_rotation_spreads_an_outlier_channel():
    # one channel x 64 in every token dominates the block scale of Q and K;
    # after the rotation the energy is spread over all channels and the
    # scores come out closer to the exact ones
    rng = np.random.default_rng(11)
    T, H, d = 128, 1, 64
    q, k, v, do = [rng.standard_normal((T, H, d)) for _ in range(4)]
    q[:, :, 5] *= 64.0
    k[:, :, 5] *= 64.0
    q, k, v, do = [O.bf16_round(x) for x in (q, k, v, do)]
    cu = [0, T]
    ex = O.attention(q, k, v, do, cu, 0.125, quant=False)
    plain = O.attention(q, k, v, do, cu, 0.125, quant=True)
    rot = O.attention(q, k, v, do, cu, 0.125, quant=True, hadamard=True)
    err = lambda r, n: np.linalg.norm(r[n] - ex[n])
    assert err(rot, "dQ") < err(plain, "dQ")
    assert err(rot, "dK") < err(plain, "dK")


def test_rotated_codes_are_the_quantised_butterflies():
    q = qkvdo(64, 2, 128, 9)[0]
    cu = [0, 40, 64]
    qz = O.Quantized(q, q, q, None, cu)
    rq = O.hadamard_fp32(q)
    c, sb = O.quantize_tokenblock(rq, cu)
    r = O.attention(q, q, q, q, cu, 0.1, quant=True, hadamard=True, backward=False)
    assert np.array_equal(r["quantized"].qc, c) and np.array_equal(r["quantized"].qs, sb)
    assert not np.array_equal(qz.qc, c)
