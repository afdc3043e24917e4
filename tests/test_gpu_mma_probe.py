"""Single-tile tensor-core products against a float64 reference: every
operand major-ness and scale placement the attention kernels use (the review
page, sec. 3.1: one E4M3 payload serves K-major and MN-major products; block
scales per 32 elements; the mixed path's NVFP4 product)."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O

pytestmark = pytest.mark.gpu


def _codes_e4m3(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38  # no NaN codes
    return c


def _run(fl, mode, N, a_mn, b_mn, variant, a, b, sfa, sfb):
    d = torch.empty((128, N), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = lambda z: torch.from_numpy(np.ascontiguousarray(z)).cuda()
    fl.flamia_debug_mma_tile(mode, N, a_mn, b_mn, variant, t(a), t(b),
                             t(sfa) if sfa is not None else None,
                             t(sfb) if sfb is not None else None, d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return d.cpu().numpy().astype(np.float64)


def _reference(mode, N, a_mn, b_mn, a, b, sfa, sfb):
    if mode == 2:
        def unpack(p):
            c = np.empty((p.shape[0], 64), dtype=np.uint8)
            c[:, 0::2] = p & 0xF
            c[:, 1::2] = p >> 4
            return O.e2m1_decode(c)
        A = unpack(a) * np.repeat(O.E4M3_TABLE[sfa], 16, axis=1)
        B = unpack(b) * np.repeat(O.E4M3_TABLE[sfb], 16, axis=1)
        return A @ B.T
    A = O.e4m3_decode(a.T if a_mn else a)          # [128][K]
    B = O.e4m3_decode(b.T if b_mn else b)          # [N][K]
    if mode in (1, 3):
        A = A * np.repeat(np.ldexp(1.0, sfa.astype(int) - 127), 32, axis=1)
        B = B * np.repeat(np.ldexp(1.0, sfb.astype(int) - 127), 32, axis=1)
    return A @ B.T


CASES = [
    # mode, N, a_mn, b_mn
    (0, 128, 0, 0),   # S = Q K^T, d = 128
    (0, 128, 1, 1),
    (1, 128, 0, 1),   # O += P V, d = 128 (V read MN-major)
    (1, 64, 0, 1),    # O += P V, d = 64
    (1, 128, 1, 1),   # dQ = dS K (dS read MN-major)
    (1, 128, 0, 0),
    (2, 128, 0, 0),   # NVFP4 S = Q K^T, d = 64
    (3, 128, 0, 1),   # O += P V with P from tensor memory, d = 128
    (3, 64, 0, 1),    # the same, d = 64
    (3, 128, 0, 0),
    (0, 32, 0, 0),    # S^T = K Q^T with 32-query tiles
    (4, 32, 0, 0),    # the same with K from tensor memory
    (4, 128, 0, 0),
    (1, 32, 1, 1),    # dQ^T = K^T dS^T with 32-query tiles (both MN-major)
    (1, 32, 0, 1),
]


@pytest.mark.parametrize("mode,N,a_mn,b_mn", CASES)
def test_tile_product(lib, mode, N, a_mn, b_mn):
    from precision_causal_attention_block_gb300 import flamia as fl
    rng = np.random.default_rng(mode * 100 + N + 10 * a_mn + b_mn)
    if mode == 2:
        a = rng.integers(0, 256, size=(128, 32), dtype=np.uint8)
        b = rng.integers(0, 256, size=(N, 32), dtype=np.uint8)
        sfa = rng.integers(0x30, 0x48, size=(128, 4), dtype=np.uint8)
        sfb = rng.integers(0x30, 0x48, size=(N, 4), dtype=np.uint8)
    else:
        a = _codes_e4m3(rng, (128, 128))
        b = _codes_e4m3(rng, (128, N) if b_mn else (N, 128))
        sfa = rng.integers(122, 133, size=(128, 4), dtype=np.uint8) if mode in (1, 3) else None
        sfb = rng.integers(122, 133, size=(N, 4), dtype=np.uint8) if mode in (1, 3) else None
    ref = _reference(mode, N, a_mn, b_mn, a, b, sfa, sfb)
    tol = 1e-5 * np.abs(ref).max()
    got = _run(fl, mode, N, a_mn, b_mn, 0, a, b, sfa, sfb)
    if np.abs(got - ref).max() > tol:
        report = {}
        for var in (1, 2, 3):
            try:
                g = _run(fl, mode, N, a_mn, b_mn, var, a, b, sfa, sfb)
                report[var] = float(np.abs(g - ref).max() / np.abs(ref).max())
            except Exception as ex:  # pragma: no cover - diagnostics only
                report[var] = str(ex)
        pytest.fail(f"variant 0 max rel err {np.abs(got - ref).max() / np.abs(ref).max():.3e}; "
                    f"other variants: {report}")


@pytest.mark.parametrize("mode,N", [(1, 128), (3, 128), (3, 64)])
def test_row_scales_from_own_lane_quadrant(lib, mode, N):
    """A's per-row block scales need only be present in the lane quadrant of
    the warp that owns the row (placement 2): each softmax warp can then set
    the scale of its own rows without exchanging them."""
    from precision_causal_attention_block_gb300 import flamia as fl
    rng = np.random.default_rng(7 + mode + N)
    a = _codes_e4m3(rng, (128, 128))
    b = _codes_e4m3(rng, (128, N))
    sfa = rng.integers(118, 137, size=(128, 4), dtype=np.uint8)
    sfb = rng.integers(122, 133, size=(N, 4), dtype=np.uint8)
    ref = _reference(mode, N, 0, 1, a, b, sfa, sfb)
    got = _run(fl, mode, N, 0, 1, 2 << 1, a, b, sfa, sfb)
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()


def test_tmem_max_reducing_load(lib):
    """tcgen05.ld.red (max) returns each thread's 32 loaded values unchanged
    and their maximum: the forward takes its row maximum of unmasked score
    tiles from it (review page, sec. 3.4 "Softmax throughput")."""
    import torch
    from precision_causal_attention_block_gb300 import flamia as fl
    rng = np.random.default_rng(11)
    x = rng.standard_normal((128, 32)).astype(np.float32) * 30.0
    x[5] = -np.abs(x[5])           # an all-negative row
    x[9, :] = -np.inf              # a fully masked row
    x[9, 17] = -3.5
    x[40, 3] = 1e30                # a huge value
    xi = torch.from_numpy(x).cuda()
    vals = torch.empty_like(xi)
    mx = torch.empty(128, dtype=torch.float32, device="cuda")
    fl.flamia_debug_tmem_ldred(xi, vals, mx)
    torch.cuda.synchronize()
    assert np.array_equal(vals.cpu().numpy(), x)
    assert np.array_equal(mx.cpu().numpy(), x.max(axis=1))


def _pair_inputs(shape, rng):
    if shape == 0:
        a, b = _codes_e4m3(rng, (2, 128, 128)), _codes_e4m3(rng, (2, 32, 128))
        return a, b, None, None
    if shape == 1:
        a, b = _codes_e4m3(rng, (2, 128, 64)), _codes_e4m3(rng, (2, 64, 64))
        sfa = rng.integers(120, 135, size=(2, 128, 2), dtype=np.uint8)
        sfb = rng.integers(122, 133, size=(2,), dtype=np.uint8)
        return a, b, sfa, sfb
    a, b = _codes_e4m3(rng, (2, 256, 128)), _codes_e4m3(rng, (2, 256, 32))
    sfa = rng.integers(122, 133, size=(2, 8), dtype=np.uint8)
    sfb = rng.integers(120, 135, size=(2, 8), dtype=np.uint8)
    return a, b, sfa, sfb


def _pair_reference(shape, a, b, sfa, sfb):
    """Per CTA r, the rows it holds: [(D_r, checked column range)]."""
    out = []
    for r in range(2):
        if shape == 0:
            B = O.e4m3_decode(np.concatenate([b[0], b[1]], axis=0))    # [64 N][128 K]
            out.append((O.e4m3_decode(a[r]) @ B.T, slice(0, 64)))
        elif shape == 1:
            A = O.e4m3_decode(a[r]) * np.repeat(np.ldexp(1.0, sfa[r].astype(int) - 127), 32, axis=1)
            B = O.e4m3_decode(np.concatenate([b[0], b[1]], axis=1))    # [64 K][128 N]
            B = B * np.ldexp(1.0, np.repeat(sfb.astype(int) - 127, 32))[:, None]
            out.append((A @ B, slice(0, 128)))
        else:
            A = O.e4m3_decode(a[r]).T * np.ldexp(1.0, np.repeat(sfa[r].astype(int) - 127, 32))[None, :]
            B = O.e4m3_decode(b[r]) * np.ldexp(1.0, np.repeat(sfb[r].astype(int) - 127, 32))[:, None]
            D = np.zeros((128, 64))
            D[:, 32 * r:32 * r + 32] = A @ B
            out.append((D, slice(32 * r, 32 * r + 32)))
    return out


def _pair_run(fl, shape, variant, a, b, sfa, sfb):
    N = 128 if shape == 1 else 64
    t = lambda z: torch.from_numpy(np.ascontiguousarray(z)).cuda()
    d = torch.zeros((2, 128, N), dtype=torch.float32, device="cuda")
    cols = torch.zeros(2, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fl.flamia_debug_pair_mma(shape, variant, t(a), t(b), t(sfa) if sfa is not None else None,
                             t(sfb) if sfb is not None else None, d, cols, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return d.cpu().numpy().astype(np.float64), cols.cpu().numpy()


@pytest.mark.parametrize("shape", [0, 1, 2])
def test_cta_pair_products(lib, shape):
    """The three CTA-pair products of the 2-CTA backward (tcgen05 .cta_group::2;
    review page sec. 3.4 "Backward pass": the pair splits 256 keys): S^T with
    each CTA supplying half of the query columns, dV / dK with each supplying
    half of the head-dimension columns, dQ^T over the pair's 256 keys with each
    CTA keeping the columns it supplied.  Both CTAs see the same tensor-memory
    columns, and each holds the 128 rows of its own A."""
    from precision_causal_attention_block_gb300 import flamia as fl
    rng = np.random.default_rng(40 + shape)
    a, b, sfa, sfb = _pair_inputs(shape, rng)
    got, cols = _pair_run(fl, shape, 0, a, b, sfa, sfb)
    assert cols[0] == cols[1]
    for r, (ref, cs) in enumerate(_pair_reference(shape, a, b, sfa, sfb)):
        err = np.abs(got[r][:, cs] - ref[:, cs]).max() / np.abs(ref[:, cs]).max()
        assert err <= 1e-5, (r, err)
