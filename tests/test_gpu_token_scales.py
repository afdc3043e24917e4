"""GPU per-token operand scales (review page, sec. 3.2: with per-token operand
scales and query-row dS exponents a future token changes no earlier output,
also inside its own 32-token block) against the oracle's token mode: codes
and scale bytes bit-exact, outputs at the attention tolerances, and the
in-block leakage probe bit for bit."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import compare, cu_tensor, dev, np64

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "do")
RAGGED = [300, 1, 129, 0, 17, 270, 33, 32, 2, 31]


@pytest.mark.parametrize("d,had", [(64, False), (128, False), (128, True)])
def test_token_codes_bit_exact(lib, d, had):
    from precision_causal_attention_block_gb300 import flamia as fl
    w = W.custom("tok_codes", RAGGED, 3, d, structure="outlier16x2", seed=4)
    x = W.make_inputs_bf16(w)["k"]
    out = fl.QTensor(w.T, w.H, d, nvfp4=False)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fmt = fl.FORMAT_MXFP8 | fl.FORMAT_TOKEN_SCALES | (fl.FORMAT_HADAMARD if had else 0)
    fl.flamia_quantize_tokenblock(dev(x), cu_tensor(w.cu_seqlens), out, fmt, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    xs = x.double().numpy()
    codes, sb = O.quantize_tokenblock(O.hadamard_fp32(xs) if had else xs, w.cu_seqlens,
                                      group="token")
    assert np.array_equal(out.scales.cpu().numpy(), sb)
    assert np.array_equal(out.codes.cpu().numpy(), codes)


def run(w, x, **kw):
    from precision_causal_attention_block_gb300 import flamia as fl
    hkv = x["k"].shape[1]
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale, H_kv=hkv,
                           token_scales=True, **kw)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    return call


@pytest.mark.parametrize("d,kw", [(64, {}), (128, {}), (64, {"causal": False}),
                                  (128, {"hadamard": True}), (64, {"deterministic_dq": True})])
def test_token_attention_against_the_oracle(lib, d, kw):
    # long documents (tensor-core kernels) beside documents of at most one
    # 32-token block (CUDA-core kernels) and one-token documents
    w = W.custom("tok_attn", RAGGED, 2, d, seed=12, structure="outlier16x2")
    x = W.make_inputs_bf16(w)
    call = run(w, x, **kw)
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale,
                      group="token", causal=kw.get("causal", True),
                      hadamard=kw.get("hadamard", False))
    qz = ref["quantized"]
    if not kw.get("hadamard"):
        assert np.array_equal(call.q.codes.cpu().numpy(), qz.qc)
    assert np.array_equal(call.v.scales.cpu().numpy(), qz.vs)
    assert np.array_equal(call.dout.scales.cpu().numpy(), qz.dos)
    rel = 3e-2 if kw.get("hadamard") else 2e-2
    for n, t in (("O", call.o), ("dQ", call.dq), ("dK", call.dk), ("dV", call.dv)):
        compare(n, np64(t), ref[n], rel_max=rel if n in ("dQ", "dK") else 2e-2)
    lse = call.lse.cpu().numpy().astype(np.float64)
    assert np.abs(lse - ref["lse"]).max() <= 1e-4 * max(1.0, np.abs(ref["lse"]).max())


def test_token_grouped_heads(lib):
    w = W.custom("tok_gqa", [300, 17, 200], 4, 128, seed=13)
    x = W.make_inputs_bf16(w)
    x["k"], x["v"] = x["k"][:, :2].contiguous(), x["v"][:, :2].contiguous()
    call = run(w, x)
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale,
                      group="token")
    for n, t in (("O", call.o), ("dQ", call.dq), ("dK", call.dk), ("dV", call.dv)):
        compare(n, np64(t), ref[n])


@pytest.mark.parametrize("d", [64, 128])
def test_token_in_block_leakage_probe_bitwise(lib, d):
    """Perturbing token 450 (block [448, 480) of the first document) leaves
    every output bit of rows 0 .. 449 -- including rows 448 and 449 of its own
    block -- and of the other document unchanged, for each of Q, K, V, dO (dQ
    in the deterministic order)."""
    w = W.custom("tok_probe", [600, 200], 2, d, seed=9)
    x = W.make_inputs_bf16(w)
    base = run(w, x, deterministic_dq=True)
    t = 450
    for name in NAMES:
        y = {n: v.clone() for n, v in x.items()}
        y[name][t] = (y[name][t].float() * 1000.0).to(torch.bfloat16)
        y[name][t, :, 5] += 50.0
        r = run(w, y, deterministic_dq=True)
        for what, a, b in (("O", r.o, base.o), ("dQ", r.dq, base.dq)):
            assert torch.equal(a[:t], b[:t]), (name, what, "earlier rows")
            assert torch.equal(a[600:], b[600:]), (name, what, "other document")
        assert torch.equal(r.lse[:, :t], base.lse[:, :t]), name
        assert torch.equal(r.dk[600:], base.dk[600:]) and torch.equal(r.dv[600:], base.dv[600:])
        later, before = (r.dq, base.dq) if name == "do" else (r.o, base.o)
        assert not torch.equal(later[t:600], before[t:600]), name


@pytest.mark.parametrize("d,kw", [(64, {}), (128, {}), (128, {"ds_rows": True}),
                                  (64, {"token_scales": True}), (64, {"nvfp4_qk": True})])
def test_ds_rounded_to_zero_counts(lib, d, kw):
    """The backward's dS rounded-to-zero diagnostic (review page, sec. 3.3 and
    the dS-scale ablation) against the oracle's count: over every pair a query
    sees, the nonzero dS entries and those whose E4M3 code under the 32 x 32
    block exponent is zero.  Float32 and float64 dS agree except within
    rounding of a code boundary or of float32 underflow, so the counts are
    compared within a small slack."""
    from precision_causal_attention_block_gb300 import flamia as fl
    w = W.custom("dszero", [300, 1, 129, 17, 2, 400], 2, d, seed=31, structure="outlier16x2")
    x = W.make_inputs_bf16(w)
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale,
                           ds_zero_count=True, **kw)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    nz, z = call.ds_zero_counts()
    qz = O.Quantized(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens,
                     qk_format="nvfp4" if kw.get("nvfp4_qk") else "mxfp8",
                     group="token" if kw.get("token_scales") else "block")
    rnz, rz = O.ds_zero_counts(qz, w.sm_scale)
    assert abs(nz - rnz) <= 1e-3 * rnz + 2, (nz, rnz)
    assert abs(z - rz) <= 2e-3 * rnz + 2, (z, rz)
    # an oversized scale in the oracle raises the count: the diagnostic has teeth
    assert O.ds_zero_counts(qz, w.sm_scale, extra=8)[1] > rz
