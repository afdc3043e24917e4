"""GPU token-block quantiser against the oracle: codes, scale bytes and NVFP4
copies bit-exact, D within float32 rounding (review page sec. 3.1, 3.2, 3.4)."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import cu_tensor, dev

pytestmark = pytest.mark.gpu

RAGGED = [1, 31, 32, 33, 0, 100, 5, 300, 127, 128, 129, 2, 257]


def run_quant(x_bf16, cu, fmt=0, o=None):
    from precision_causal_attention_block_gb300 import flamia as fl
    T, H, d = x_bf16.shape
    out = fl.QTensor(T, H, d, nvfp4=(fmt == 1))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    D = torch.empty((H, T), dtype=torch.float32, device="cuda") if o is not None else None
    fl.flamia_quantize_tokenblock(dev(x_bf16), cu_tensor(cu), out, fmt,
                                  o=dev(o) if o is not None else None, D=D, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out, D


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("fmt", [0, 1])
def test_ragged_documents_bit_exact(lib, d, fmt):
    w = W.custom("ragged", RAGGED, 3, d, structure="outlier16x2", seed=3)
    x = W.make_inputs_bf16(w)["q"]
    out, _ = run_quant(x, w.cu_seqlens, fmt)
    xc = x.double().numpy()
    codes, sb = O.quantize_tokenblock(xc, w.cu_seqlens)
    assert np.array_equal(out.codes.cpu().numpy(), codes)
    assert np.array_equal(out.scales.cpu().numpy(), sb)
    if fmt == 1:
        pk, sc = O.quantize_nvfp4(xc)
        assert np.array_equal(out.nvfp4_scales.cpu().numpy(), sc)
        assert np.array_equal(out.nvfp4_codes.cpu().numpy(), pk)


@pytest.mark.parametrize("d", [64, 128])
def test_many_documents_per_segment(lib, d):
    """Each CTA finds the documents of its rows with a warp-wide search and a
    shared-memory copy of their offsets, or, when its rows span more
    documents than the copy holds (here: runs of 300 empty documents), with a
    per-token search: both give the codes of the oracle bit for bit, for
    one-token documents too."""
    # 1,100 tokens, 757 documents (at most T + 1); the rows staged by the
    # CTA of tokens 128 .. 287 span about 380 of them
    lens = [1] * 200 + [0] * 300 + [5, 1, 1] + [40] + [1] * 150 + [0] * 100 + [70, 33] + [600]
    w = W.custom("manydocs", lens, 2, d, structure="outlier16x2", seed=8)
    xs = W.make_inputs_bf16(w)
    x = xs["q"]
    out, D = run_quant(x, w.cu_seqlens, 0, o=xs["k"])
    codes, sb = O.quantize_tokenblock(x.double().numpy(), w.cu_seqlens)
    assert np.array_equal(out.codes.cpu().numpy(), codes)
    assert np.array_equal(out.scales.cpu().numpy(), sb)


def test_extreme_magnitudes_and_zeros(lib):
    w = W.custom("extreme", [40, 70, 1], 2, 64, seed=4)
    x = W.make_inputs_f32(w)["q"]
    x[:32] *= 1e-30           # tiny block (subnormal codes, exponent clamp)
    x[32:40] = 0.0            # all-zero block
    x[40:72] *= 1e30          # huge block
    x[45, 0, 3] = -0.0
    xb = torch.from_numpy(x).to(torch.bfloat16)
    out, _ = run_quant(xb, w.cu_seqlens)
    codes, sb = O.quantize_tokenblock(xb.double().numpy(), w.cu_seqlens)
    assert np.array_equal(out.codes.cpu().numpy(), codes)
    assert np.array_equal(out.scales.cpu().numpy(), sb)


def test_fused_D(lib):
    w = W.custom("ragged", RAGGED, 2, 128, seed=5)
    x = W.make_inputs_bf16(w)
    out, D = run_quant(x["do"], w.cu_seqlens, o=x["v"])
    codes, sb = O.quantize_tokenblock(x["do"].double().numpy(), w.cu_seqlens)
    ref = O.compute_D(codes, sb, x["v"].double().numpy())
    got = D.cpu().numpy().astype(np.float64)
    scale = np.abs(ref).max()
    assert np.abs(got - ref).max() <= 1e-5 * scale


@pytest.mark.parametrize("name", ["tiny", "fixed4x4096", "varlen65536", "onetoken131072",
                                  "long131072"])
def test_full_size_configs(lib, name):
    """Full-size launch; the oracle checks a token window that holds whole
    32-token blocks (documents are independent, blocks are document-local)."""
    w = W.WORKLOADS[name]()
    x = W.make_inputs_bf16(w)["k"]
    fmt = 1 if w.d == 64 else 0
    out, _ = run_quant(x, w.cu_seqlens, fmt)
    cu = list(w.cu_seqlens)
    for (s, e) in ((0, min(w.T, 2048)), (max(0, w.T - 2048), w.T)):
        # widen the window to document boundaries where documents are short,
        # else keep it on the 32-token grid of the single document
        if len(cu) > 2:
            s = max(c for c in cu if c <= s)
            e = min(c for c in cu if c >= e)
            local = [c - s for c in cu if s <= c <= e]
        else:
            s -= s % 32
            local = [0, e - s]
        if e - s > 20000:
            continue
        xs = x[s:e].double().numpy()
        codes, sb = O.quantize_tokenblock(xs, local)
        assert np.array_equal(out.codes[s:e].cpu().numpy(), codes), (s, e)
        assert np.array_equal(out.scales[:, s:e].cpu().numpy(), sb), (s, e)
        if fmt == 1:
            pk, sc = O.quantize_nvfp4(xs)
            assert np.array_equal(out.nvfp4_codes[s:e].cpu().numpy(), pk)
            assert np.array_equal(out.nvfp4_scales[s:e].cpu().numpy(), sc)


def test_bad_seqlens_set_the_status_bit(lib):
    from precision_causal_attention_block_gb300 import flamia as fl
    x = torch.zeros((64, 1, 64), dtype=torch.bfloat16, device="cuda")
    out = fl.QTensor(64, 1, 64)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, 40, 30, 64], dtype=torch.int32, device="cuda")
    fl.flamia_quantize_tokenblock(x, cu, out, 0, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & fl.DEV_BAD_SEQLENS


@pytest.mark.parametrize("d,fmt,H,Hkv", [(128, 0, 4, 2), (64, 1, 3, 3), (128, 0x10, 2, 1),
                                         (64, 0, 6, 3)])
def test_quantize_qkv_one_launch_equals_three_calls(lib, d, fmt, H, Hkv):
    # flamia_quantize_qkv: Q and K with the call's format, V plain MXFP8, K / V
    # with H_kv heads; bit for bit the three single calls, which the tests
    # above pin against the oracle (Q's codes are checked against it here too)
    from precision_causal_attention_block_gb300 import flamia as fl
    w = W.custom("qkv", RAGGED, H, d, structure="outlier16x2", seed=5)
    x = W.make_inputs_bf16(w)
    xq, xk, xv = dev(x["q"]), dev(x["k"][:, :Hkv].contiguous()), dev(x["v"][:, :Hkv].contiguous())
    cu = cu_tensor(w.cu_seqlens)
    nv = (fmt & 0xF) == 1
    q, k, v = fl.QTensor(w.T, H, d, nv), fl.QTensor(w.T, Hkv, d, nv), fl.QTensor(w.T, Hkv, d)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fl.flamia_quantize_qkv(xq, xk, xv, cu, q, k, v, fmt, dev_status=st)
    refs = [fl.QTensor(w.T, H, d, nv), fl.QTensor(w.T, Hkv, d, nv), fl.QTensor(w.T, Hkv, d)]
    for xx, out, f in zip((xq, xk, xv), refs, (fmt, fmt, 0)):
        fl.flamia_quantize_tokenblock(xx, cu, out, f, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for a, b in zip((q, k, v), refs):
        assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
        if a.nvfp4_codes is not None:
            assert torch.equal(a.nvfp4_codes, b.nvfp4_codes)
            assert torch.equal(a.nvfp4_scales, b.nvfp4_scales)
    if fmt != 0x10:
        codes, sb = O.quantize_tokenblock(x["q"].double().numpy(), w.cu_seqlens)
        assert np.array_equal(q.codes.cpu().numpy(), codes)
        assert np.array_equal(q.scales.cpu().numpy(), sb)
