"""Pins of the oracle's token-block quantiser.

Source: "FLAMIA ... (jaehun.me review)", sec. 3.1 (one power-of-two exponent
per 32 consecutive tokens x full head dimension; the scale is constant along
the head dimension so the codes stay valid under transpose), sec. 3.2
(round-up exponent, nothing clips) and sec. 3.4 "Packed documents" (groups
never cross a document boundary; one dense scale entry per token)."""
import numpy as np

from oracle import flamia_oracle as O


def _data(T=300, H=3, d=16, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H, d)) * np.exp(rng.uniform(-3, 3, (T, 1, 1)))
    return O.bf16_round(x)


CU = [0, 37, 38, 100, 300]


def test_blocks_are_document_local():
    blocks = O.doc_blocks(CU)
    assert blocks[0] == (0, 32) and blocks[1] == (32, 37) and blocks[2] == (37, 38)
    assert blocks[3] == (38, 70) and blocks[4] == (70, 100) and blocks[5] == (100, 132)
    for (b0, b1) in blocks:
        assert 0 < b1 - b0 <= 32
        doc = [i for i in range(len(CU) - 1) if CU[i] <= b0 < CU[i + 1]][0]
        assert b1 <= CU[doc + 1]


def test_scale_is_constant_per_block_and_codes_respect_error_bound():
    x = _data()
    codes, sb = O.quantize_tokenblock(x, CU)
    for (b0, b1) in O.doc_blocks(CU):
        for h in range(x.shape[1]):
            assert len(set(sb[h, b0:b1])) == 1
            e = int(sb[h, b0]) - 127
            amax = np.abs(x[b0:b1, h]).max()
            assert amax * 2.0 ** -e <= 448 and amax * 2.0 ** -e > 224
    xh = O.dequantize_tokenblock(codes, sb)
    scale = O.e8m0_decode(sb).T[:, :, None]
    err = np.abs(xh - x)
    # RNE to 3 mantissa bits: half an ulp, ulp = 2^(E-3) in the normal range,
    # 2^-9 below 2^-6 (all in units of the block scale)
    a = np.abs(x) / scale
    ulp = np.where(a < 2.0 ** -6, 2.0 ** -9, np.ldexp(1.0, np.frexp(a)[1] - 1 - 3))
    assert np.all(err <= 0.5 * ulp * scale * (1 + 1e-12))


def test_no_scale_group_crosses_a_document():
    x = _data()
    codes, sb = O.quantize_tokenblock(x, CU)
    y = x.copy()
    y[40] *= 1000.0                       # doc 2 = [38, 100)
    c2, s2 = O.quantize_tokenblock(y, CU)
    changed = np.any(c2 != codes, axis=(1, 2)) | np.any(s2 != sb, axis=0)
    idx = np.nonzero(changed)[0]
    assert idx.min() >= 38 and idx.max() < 70   # only inside token 40's block


def test_tensor_wide_scale_does_cross_documents():
    x = _data()
    codes, sb = O.quantize_tokenblock(x, CU, group="tensor")
    y = x.copy()
    y[250] *= 1000.0
    c2, s2 = O.quantize_tokenblock(y, CU, group="tensor")
    assert np.any(s2[:, :38] != sb[:, :38])


def test_payload_is_transposable():
    """Dequantising the [token, dim] payload and dequantising the same bytes
    read as the transposed [dim, token] operand (scale along the contraction
    axis, one per 32 tokens) give transposed values: one payload serves both
    the K-major and the MN-major product."""
    x = _data()
    codes, sb = O.quantize_tokenblock(x, CU)
    T, H, d = x.shape
    for h in range(H):
        row_major = O.e4m3_decode(codes[:, h, :]) * O.e8m0_decode(sb[h])[:, None]
        ct = codes[:, h, :].T.copy()                       # [d, T]
        col_scales = O.e8m0_decode(sb[h])[None, :]         # along tokens
        mn_major = O.e4m3_decode(ct) * col_scales
        assert np.array_equal(mn_major.T, row_major)


def test_empty_and_single_token_documents():
    x = _data(T=5)
    cu = [0, 0, 1, 1, 5]
    codes, sb = O.quantize_tokenblock(x, cu)
    xh = O.dequantize_tokenblock(codes, sb)
    e = sb[:, 0].astype(int) - 127
    # a one-token block holds its own maximum: |max| scaled lands in (224, 448]
    for h in range(x.shape[1]):
        assert 224 < np.abs(x[0, h]).max() * 2.0 ** -e[h] <= 448
    assert np.allclose(xh, x, rtol=2 ** -4)


def test_zero_block():
    x = np.zeros((32, 1, 8))
    codes, sb = O.quantize_tokenblock(x, [0, 32])
    assert np.all(codes == 0) and np.all(sb == 0)


def test_compute_D_definition():
    x = _data(T=64, H=2, d=8)
    o = O.bf16_round(_data(T=64, H=2, d=8, seed=3))
    codes, sb = O.quantize_tokenblock(x, [0, 64])
    D = O.compute_D(codes, sb, o)
    xh = O.dequantize_tokenblock(codes, sb)
    for h in range(2):
        for t in (0, 17, 63):
            assert np.isclose(D[h, t], sum(xh[t, h, k] * o[t, h, k] for k in range(8)),
                              rtol=1e-14, atol=0)


def test_nvfp4_roundtrip_and_packing():
    x = _data(T=7, H=2, d=32)
    packed, sc = O.quantize_nvfp4(x)
    assert packed.shape == (7, 2, 16) and sc.shape == (7, 2, 2)
    xh = O.dequantize_nvfp4(packed, sc)
    g = x.reshape(7, 2, 2, 16)
    s = O.E4M3_TABLE[sc][..., None]
    # every element within half an E2M1 step of its scaled value (max step 2 at [4,6])
    assert np.all(np.abs(xh.reshape(7, 2, 2, 16) - g) <= 1.0 * s + 1e-300)
    # element 0 is the low nibble
    c0 = O.e2m1_encode(g[0, 0, 0, 0] / s[0, 0, 0, 0])
    assert (packed[0, 0, 0] & 0xF) == c0
