"""GPU prescaled FP16 dQ accumulator (FLAMIA_FLAG_DQ_FP16, with
FLAMIA_FLAG_DQ_CAUSAL_SCALE for causal dQ scaling; review page, sec. 3.2
"accumulator leakage", sec. 3.5.3) against the oracle's model of it: the
prescale table bit for bit, dQ at the attention tolerances on every kernel
(head dims 64 and 128, the mixed NVFP4 path, non-causal, grouped heads, the
rotation, short documents), and the leakage probe bit for bit in the
deterministic mode: causal scaling keeps a later token out of earlier dQ rows,
the sequence-wide prescale lets it in."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import compare, cu_tensor, dev, np64

pytestmark = pytest.mark.gpu

MIX = [300, 1, 129, 0, 17, 270, 33, 32, 530]
NAMES = ("q", "k", "v", "do")


def align256(n):
    return (n + 255) // 256 * 256


def prescale_table(call):
    # the int8 [H, T] part of the backward workspace, after the float32
    # accumulator and the int32 turn counters
    T, H, d = call.T, call.H, call.d
    off = align256(T * H * d * 4) + align256(T * H * 4)
    return call.ws[off:off + H * T].view(torch.int8).reshape(H, T).cpu().numpy().astype(np.int64)


def run(w, x, Hkv=None, **kw):
    from precision_causal_attention_block_gb300 import flamia as fl
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale, H_kv=Hkv, **kw)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    return call


@pytest.mark.parametrize("mode", ["fp16_sequence", "fp16_causal"])
@pytest.mark.parametrize("d,Hkv,kw", [
    (128, None, {}),
    (64, None, {}),
    (64, None, {"nvfp4_qk": True}),
    (128, None, {"causal": False}),
    (128, 2, {}),
    (64, None, {"hadamard": True}),
])
def test_dq16_against_the_oracle(lib, mode, d, Hkv, kw):
    w = W.custom("dq16_mix", MIX, 4, d, seed=31, structure="outlier16x2")
    x = W.make_inputs_bf16(w)
    if Hkv:
        x["k"], x["v"] = x["k"][:, :Hkv].contiguous(), x["v"][:, :Hkv].contiguous()
    call = run(w, x, Hkv, dq_accum=mode, **kw)
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale,
                      qk_format="nvfp4" if kw.get("nvfp4_qk") else "mxfp8",
                      causal=kw.get("causal", True), hadamard=kw.get("hadamard", False),
                      dq_accum=mode)
    assert np.array_equal(prescale_table(call), ref["dq_prescale"])
    rel = 3e-2 if kw.get("hadamard") else 2e-2
    compare("dQ", np64(call.dq), ref["dQ"], rel_max=rel)
    for n, t in (("O", call.o), ("dK", call.dk), ("dV", call.dv)):
        compare(n, np64(t), ref[n], rel_max=rel)


def test_dq16_fixed4x4096_close_to_float32(lib):
    # the full-size shape: the FP16 accumulator against the float32 one of
    # the same call (same codes, same products)
    w = W.fixed4x4096()
    x = W.make_inputs_bf16(w)
    a = run(w, x)
    dq32 = np64(a.dq)
    for mode in ("fp16_sequence", "fp16_causal"):
        b = run(w, x, dq_accum=mode)
        assert torch.equal(a.dk, b.dk) and torch.equal(a.dv, b.dv)
        compare("dQ", np64(b.dq), dq32, cos_min=0.99999, rel_max=5e-3)


def test_dq_leakage_probe_bitwise(lib):
    """A large later token (block [448, 480) of document 0, in K or V) leaves
    every dQ bit of rows 0 .. 447 unchanged with the float32 accumulator and
    with causal dQ scaling, and changes them with the sequence-wide prescale
    (deterministic mode: the sums run in one order)."""
    w = W.custom("probe16", [600, 200], 2, 128, seed=9)
    x = W.make_inputs_bf16(w)
    t = 450
    for mode, same in (("fp32", True), ("fp16_causal", True), ("fp16_sequence", False)):
        base = run(w, x, deterministic_dq=True, dq_accum=mode).dq.clone()
        again = run(w, x, deterministic_dq=True, dq_accum=mode).dq
        assert torch.equal(base, again), mode
        for name in ("k", "v"):
            y = {n: v.clone() for n, v in x.items()}
            y[name][t] = (y[name][t].float() * 1000.0).to(torch.bfloat16)
            r = run(w, y, deterministic_dq=True, dq_accum=mode)
            assert torch.equal(r.dq[:448], base[:448]) == same, (mode, name)
            assert torch.equal(r.dq[600:], base[600:]) == same, (mode, name)
