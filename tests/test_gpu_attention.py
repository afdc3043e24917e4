"""GPU causal forward + backward against the FP64 oracle.

Bar (the review page's accuracy section and the method's numerics): on the
same quantised inputs O, dQ, dK, dV reach cosine >= 0.9995 and max |err| <=
2e-2 max |ref| against the oracle; the codes are bit-exact; on plain normal
inputs the quantised path reaches cosine >= 0.998 against exact attention;
a future token outside a block changes no earlier O / LSE bit (sec. 3.2, 4.5).
"""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import compare, cu_tensor, dev, np64

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "do")


def run_call(w, x, nvfp4=False):
    from precision_causal_attention_block_gb300 import flamia as fl
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale, nvfp4_qk=nvfp4)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    return call


def check_against(call, ref, tok, heads, what=("O", "dQ", "dK", "dV")):
    """Compare GPU outputs on tokens `tok` (slice) and `heads` with an oracle
    result computed on exactly that slice."""
    gpu = {"O": call.o, "dQ": call.dq, "dK": call.dk, "dV": call.dv}
    for n in what:
        compare(n, np64(gpu[n][tok][:, heads]), ref[n])
    lse = call.lse[heads][:, tok].cpu().numpy().astype(np.float64)
    assert np.abs(lse - ref["lse"]).max() <= 1e-4 * max(1.0, np.abs(ref["lse"]).max())


@pytest.mark.parametrize("d", [64, 128])
def test_ragged_small_elementwise(lib, d):
    w = W.custom("ragged_attn", [300, 1, 129, 0, 270, 33, 256], 2, d, seed=7,
                 structure="outlier16x2")
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale)
    qz = ref["quantized"]
    assert np.array_equal(call.q.codes.cpu().numpy(), qz.qc)
    assert np.array_equal(call.v.scales.cpu().numpy(), qz.vs)
    assert np.array_equal(call.dout.codes.cpu().numpy(), qz.doc)
    check_against(call, ref, slice(0, w.T), list(range(w.H)))
    compare("D", call.D.cpu().numpy(), ref["D"], cos_min=0.99999, rel_max=1e-3)


SHORT_MIX = [1, 2, 5, 17, 31, 32, 33, 40, 3, 0, 300, 1]


@pytest.mark.parametrize("d,nvfp4", [(64, False), (128, False), (64, True)])
def test_short_documents_elementwise(lib, d, nvfp4):
    """Documents of at most one 32-token block (one scale per operand) beside
    longer ones: the packed-document case of the review page, sec. 3.4."""
    w = W.custom("short_mix", SHORT_MIX, 3, d, seed=21, structure="outlier16x2")
    x = W.make_inputs_bf16(w)
    call = run_call(w, x, nvfp4=nvfp4)
    fmt = "nvfp4" if nvfp4 else "mxfp8"
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale,
                      qk_format=fmt)
    check_against(call, ref, slice(0, w.T), list(range(w.H)))


def test_all_zero_short_document(lib):
    """An all-zero query block has the smallest scale exponent; its scores are
    0 and attention is uniform over the visible keys (no NaN from masking)."""
    w = W.custom("zero_doc", [7, 20, 45], 2, 128, seed=23)
    x = W.make_inputs_bf16(w)
    x["q"][7:27] = 0
    x["k"][0:7] = 0
    call = run_call(w, x)
    for t in (call.o, call.lse, call.dq, call.dk, call.dv):
        assert torch.isfinite(t.float()).all()
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale)
    check_against(call, ref, slice(0, w.T), list(range(w.H)))
    # uniform attention: O_i = mean of the dequantised V rows up to i
    v = O.dequantize_tokenblock(ref["quantized"].vc, ref["quantized"].vs)
    want = np.cumsum(v[7:27], 0) / np.arange(1, 21)[:, None, None]
    compare("O uniform", np64(call.o[7:27]), want)


@pytest.mark.parametrize("d", [64, 128])
def test_all_zero_blocks_in_long_documents(lib, d):
    """All-zero 32-token blocks get the smallest scale exponent (factor 0 in
    the kernels); on a diagonal tile the masked keys must still give 0, not
    NaN (a masked score times a zero factor)."""
    w = W.custom("zero_blocks", [300, 200], 2, d, seed=29)
    x = W.make_inputs_bf16(w)
    x["k"][128:160] = 0     # key block on the diagonal of query tile 1
    x["q"][160:192] = 0     # a query block
    x["v"][320:352] = 0
    x["do"][64:96] = 0
    call = run_call(w, x)
    for t in (call.o, call.lse, call.dq, call.dk, call.dv):
        assert torch.isfinite(t.float()).all()
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale)
    check_against(call, ref, slice(0, w.T), list(range(w.H)))


def test_tiny_config(lib):
    w = W.tiny()
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale)
    check_against(call, ref, slice(0, w.T), [0, 1])


def test_fixed4x4096_one_document_two_heads(lib):
    w = W.fixed4x4096()
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    heads = [0, 9]
    s, e = 4096, 8192  # document 1
    ref = O.attention(*[x[n][s:e][:, heads].double().numpy() for n in NAMES], [0, e - s],
                      w.sm_scale)
    check_against(call, ref, slice(s, e), heads)


def test_varlen65536_sampled(lib):
    w = W.varlen65536()
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    cu = list(w.cu_seqlens)
    lens = np.diff(cu)
    # one mid-size document in full, plus exact-attention cosine on it
    b = int(np.argmin(np.abs(lens - 2000)))
    s, e = cu[b], cu[b + 1]
    heads = [3]
    sl = [x[n][s:e][:, heads].double().numpy() for n in NAMES]
    ref = O.attention(*sl, [0, e - s], w.sm_scale)
    check_against(call, ref, slice(s, e), heads)
    exact = O.attention(*sl, [0, e - s], w.sm_scale, quant=False)
    for n, t in (("O", call.o), ("dQ", call.dq), ("dK", call.dk), ("dV", call.dv)):
        cos = O.cosine(np64(t[s:e][:, heads]), exact[n])
        method = O.cosine(ref[n], exact[n])
        if n in ("O", "dV"):
            assert cos >= 0.998, (n, cos, method)
        else:
            # the method itself (the oracle) sits at 0.9979 for dQ and dK on
            # these plain normal inputs, the summary page's own dQ figure for
            # MXFP8: the kernel must stay within 2e-4 of it
            assert cos >= method - 2e-4 and cos >= 0.997, (n, cos, method)
    # the longest document: its first and last query blocks, last key blocks
    b = int(np.argmax(lens))
    s, e = cu[b], cu[b + 1]
    L = e - s
    qz = O.Quantized(*[x[n][s:e][:, heads].double().numpy() for n in NAMES], [0, L])
    nb = (L + 31) // 32
    res = O.sampled_rows(qz, 0, 0, w.sm_scale, qblocks=[0, 1, nb - 1], kblocks=[nb - 2, nb - 1])
    for qb in res["O"]:
        rows = slice(s + 32 * qb, min(s + 32 * qb + 32, e))
        compare(f"O[{qb}]", np64(call.o[rows][:, heads[0]]), res["O"][qb])
        compare(f"dQ[{qb}]", np64(call.dq[rows][:, heads[0]]), res["dQ"][qb])
    for kb in res["dK"]:
        rows = slice(s + 32 * kb, min(s + 32 * kb + 32, e))
        compare(f"dK[{kb}]", np64(call.dk[rows][:, heads[0]]), res["dK"][kb])
        compare(f"dV[{kb}]", np64(call.dv[rows][:, heads[0]]), res["dV"][kb])


def test_onetoken131072_slice(lib):
    w = W.onetoken131072()
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    for (s, e) in ((0, 256), (w.T - 256, w.T)):
        sl = [x[n][s:e].double().numpy() for n in NAMES]
        ref = O.attention(*sl, list(range(e - s + 1)), w.sm_scale)
        check_against(call, ref, slice(s, e), list(range(w.H)))
        exact = O.attention(*sl, list(range(e - s + 1)), w.sm_scale, quant=False)
        assert O.cosine(np64(call.o[s:e]), exact["O"]) >= 0.998


def test_long131072_sampled(lib):
    w = W.long131072()
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    heads = [0, 17]
    for h in heads:
        qz = O.Quantized(*[x[n][:, [h]].double().numpy() for n in NAMES], [0, w.T])
        nb = w.T // 32
        res = O.sampled_rows(qz, 0, 0, w.sm_scale, qblocks=[0, 5, nb // 2, nb - 1],
                             kblocks=[nb - 3, nb - 1])
        for qb in res["O"]:
            rows = slice(32 * qb, 32 * qb + 32)
            compare(f"O[{qb}]", np64(call.o[rows][:, h]), res["O"][qb])
            compare(f"dQ[{qb}]", np64(call.dq[rows][:, h]), res["dQ"][qb])
            lse = call.lse[h, rows].cpu().numpy().astype(np.float64)
            assert np.abs(lse - res["lse"][qb]).max() <= 1e-4 * np.abs(res["lse"][qb]).max()
        for kb in res["dK"]:
            rows = slice(32 * kb, 32 * kb + 32)
            compare(f"dK[{kb}]", np64(call.dk[rows][:, h]), res["dK"][kb])
            compare(f"dV[{kb}]", np64(call.dv[rows][:, h]), res["dV"][kb])


def perturbed(x, name, t):
    """A x1000 copy of token t of tensor `name` with one channel shifted by 50."""
    y = {n: v.clone() for n, v in x.items()}
    y[name][t] = (y[name][t].float() * 1000.0).to(torch.bfloat16)
    y[name][t, :, 5] += 50.0
    return y


@pytest.mark.parametrize("d", [128, 64])
def test_leakage_probe_bitwise(lib, d):
    """Review page, sec. 3.2 and 4.5: perturbing a future token outside the
    victim's 32-token block (and in another document) changes no earlier
    output bit.  The dQ partials are summed in a fixed order (deterministic
    mode), so every output is compared bit for bit: O, LSE and dQ of the
    rows before the perturbed token's block, and O, LSE, dQ, dK, dV of the
    other document, under a perturbation of each of Q, K, V and dO."""
    from precision_causal_attention_block_gb300 import flamia as fl
    w = W.custom("probe", [600, 200], 2, d, seed=9)
    x = W.make_inputs_bf16(w)

    def run(xx):
        call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale,
                               deterministic_dq=True)
        xd = {n: dev(t) for n, t in xx.items()}
        call.forward(xd["q"], xd["k"], xd["v"])
        call.backward(xd["do"])
        torch.cuda.synchronize()
        call.check_status()
        return call

    base = run(x)
    t = 450  # block [448, 480) of document 0
    for name in NAMES:
        r = run(perturbed(x, name, t))
        for what, a, b in (("O", r.o, base.o), ("dQ", r.dq, base.dq)):
            assert torch.equal(a[:448], b[:448]), (name, what, "earlier rows")
            assert torch.equal(a[600:], b[600:]), (name, what, "other document")
        assert torch.equal(r.lse[:, :448], base.lse[:, :448]), name
        assert torch.equal(r.lse[:, 600:], base.lse[:, 600:]), name
        assert torch.equal(r.dk[600:], base.dk[600:]), (name, "dK other document")
        assert torch.equal(r.dv[600:], base.dv[600:]), (name, "dV other document")
        # the probe has teeth: the perturbation reaches the later rows
        later, before = (r.dq, base.dq) if name == "do" else (r.o, base.o)
        assert not torch.equal(later[448:600], before[448:600]), name


def test_leakage_probe_atomic_order(lib):
    """The same probe in the default mode, where dQ partials are summed with
    float32 reduce-adds in no fixed order: O, LSE, dK and dV compare bit for
    bit; dQ of the earlier rows may differ from a repeat of the call only by
    the summation-order noise, bounded per element by two BF16 steps of its
    value (a leak of the x1000 token would be orders of magnitude larger)."""
    w = W.custom("probe", [600, 200], 2, 128, seed=9)
    x = W.make_inputs_bf16(w)
    base = run_call(w, x)
    o0, l0, dq0 = base.o.clone(), base.lse.clone(), base.dq.float()
    bound = 2.0 ** -6 * dq0.abs() + 1e-6 * dq0.abs().max()
    for name in NAMES:
        r = run_call(w, perturbed(x, name, 450))
        assert torch.equal(r.o[:448], o0[:448]), name
        assert torch.equal(r.lse[:, :448], l0[:, :448]), name
        assert torch.equal(r.o[600:], o0[600:]), name
        assert torch.equal(r.dk[600:], base.dk[600:]), name
        assert torch.equal(r.dv[600:], base.dv[600:]), name
        diff = (r.dq.float() - dq0).abs()
        assert (diff[:448] <= bound[:448]).all(), (name, diff[:448].max().item())
        assert (diff[600:] <= bound[600:]).all(), (name, diff[600:].max().item())


# ---------------------------------------------------------------- mixed NVFP4 path

def test_nvfp4_mixed_ragged_small(lib):
    """Scores from the NVFP4 copies of Q and K (review page sec. 3.1 mixed
    path); every other product stays MXFP8."""
    w = W.custom("ragged_nvfp4", [300, 1, 129, 0, 270, 33, 256], 2, 64, seed=17)
    x = W.make_inputs_bf16(w)
    call = run_call(w, x, nvfp4=True)
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale,
                      qk_format="nvfp4")
    check_against(call, ref, slice(0, w.T), list(range(w.H)))


def test_nvfp4_mixed_long131072_sampled(lib):
    w = W.long131072()
    x = W.make_inputs_bf16(w)
    call = run_call(w, x, nvfp4=True)
    h = 5
    qz = O.Quantized(*[x[n][:, [h]].double().numpy() for n in NAMES], [0, w.T],
                     qk_format="nvfp4")
    nb = w.T // 32
    res = O.sampled_rows(qz, 0, 0, w.sm_scale, qblocks=[0, 7, nb // 3, nb - 1],
                         kblocks=[nb - 2, nb - 1])
    for qb in res["O"]:
        rows = slice(32 * qb, 32 * qb + 32)
        compare(f"O[{qb}]", np64(call.o[rows][:, h]), res["O"][qb])
        compare(f"dQ[{qb}]", np64(call.dq[rows][:, h]), res["dQ"][qb])
    for kb in res["dK"]:
        rows = slice(32 * kb, 32 * kb + 32)
        compare(f"dK[{kb}]", np64(call.dk[rows][:, h]), res["dK"][kb])
        compare(f"dV[{kb}]", np64(call.dv[rows][:, h]), res["dV"][kb])


def test_nvfp4_flag_needs_head_dim_64(lib):
    from precision_causal_attention_block_gb300 import flamia as fl
    w = W.custom("d128", [64], 1, 128)
    x = W.make_inputs_bf16(w)
    with pytest.raises(RuntimeError, match="unsupported"):
        run_call(w, x, nvfp4=True)


@pytest.mark.parametrize("d,H,Hkv,kw", [(128, 3, 3, {}), (64, 2, 2, {"nvfp4_qk": True}),
                                         (128, 4, 2, {}), (64, 2, 2, {"hadamard": True}),
                                         (64, 2, 2, {"causal": False}),
                                         (128, 2, 2, {"dq_accum": "fp16_causal"}),
                                         (64, 2, 2, {"deterministic_dq": True})])
def test_mostly_one_token_documents(lib, d, H, Hkv, kw):
    """Documents averaging under two tokens (the one-thread kernels take the
    one-token documents; each warp of the short-document kernels scans 32
    (document, head) pairs) with a few longer ones mixed in, element by
    element against the oracle."""
    from precision_causal_attention_block_gb300 import flamia as fl
    rng = np.random.default_rng(7)
    lengths = [1] * 400
    for L, at in zip((2, 5, 17, 31, 32, 0, 3, 40), rng.choice(400, 8, replace=False)):
        lengths[at] = L
    w = W.custom("mostly_one", lengths, H, d, seed=11)
    assert w.T <= 2 * len(lengths)
    x = W.make_inputs_bf16(w)
    x["k"], x["v"] = x["k"][:, :Hkv].contiguous(), x["v"][:, :Hkv].contiguous()
    call = fl.TrainingCall(w.T, H, d, cu_tensor(w.cu_seqlens), w.sm_scale, H_kv=Hkv, **kw)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale,
                      qk_format="nvfp4" if kw.get("nvfp4_qk") else "mxfp8",
                      causal=kw.get("causal", True), hadamard=kw.get("hadamard", False),
                      dq_accum=kw.get("dq_accum", "fp32"))
    rel = 3e-2 if kw.get("hadamard") else 2e-2
    for n, t in (("O", call.o), ("dQ", call.dq), ("dK", call.dk), ("dV", call.dv)):
        compare(n, np64(t), ref[n], rel_max=rel)
