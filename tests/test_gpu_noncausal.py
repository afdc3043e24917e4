"""GPU non-causal packed call (review page, sec. 4.8 "Batched and non-causal
paths": every query sees every key of its own document) against the oracle's
non-causal mode, at the attention tolerances, on the tensor-core kernels
(documents longer than one block) and the CUDA-core kernels (documents of at
most 32 tokens), head dims 64 and 128 and the mixed NVFP4 path."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import compare, cu_tensor, dev, np64

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "do")
MIX = [300, 1, 129, 0, 17, 270, 33, 32, 256]


def run_call(w, x, nvfp4=False):
    from precision_causal_attention_block_gb300 import flamia as fl
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale, nvfp4_qk=nvfp4,
                           causal=False)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    return call


@pytest.mark.parametrize("d,nvfp4", [(64, False), (128, False), (64, True)])
def test_noncausal_against_the_oracle(lib, d, nvfp4):
    w = W.custom("noncausal_mix", MIX, 2, d, seed=13, structure="outlier16x2")
    x = W.make_inputs_bf16(w)
    call = run_call(w, x, nvfp4)
    xs = [x[n].double().numpy() for n in NAMES]
    ref = O.attention(*xs, w.cu_seqlens, w.sm_scale, causal=False,
                      qk_format="nvfp4" if nvfp4 else "mxfp8")
    gpu = {"O": call.o, "dQ": call.dq, "dK": call.dk, "dV": call.dv}
    for n in ("O", "dQ", "dK", "dV"):
        compare(n, np64(gpu[n]), ref[n])
    lse = call.lse.cpu().numpy().astype(np.float64)
    assert np.abs(lse - ref["lse"]).max() <= 1e-4 * max(1.0, np.abs(ref["lse"]).max())
    # D from its definition on the GPU's own forward output
    qz = ref["quantized"]
    want_D = O.compute_D(qz.doc, qz.dos, np64(call.o))
    compare("D", call.D.cpu().numpy(), want_D, cos_min=0.9999999, rel_max=1e-5)


def test_noncausal_differs_from_causal(lib):
    # the first query of a document sees only itself causally, every key of
    # the document otherwise
    w = W.custom("noncausal_one", [200], 1, 64, seed=17)
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    ref_c = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale)
    assert O.cosine(np64(call.o)[0], ref_c["O"][0]) < 0.9


def test_noncausal_fixed4x4096_sampled(lib):
    # the full-size shape (head dim 128, 4096-token documents): sampled query
    # blocks (O, dQ) and key blocks (dK, dV) of one document, from their own
    # definitions over the whole document
    w = W.fixed4x4096()
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    h, s = 5, 8192
    xs = [x[n][s:s + 4096].double().numpy() for n in NAMES]
    qz = O.Quantized(*xs, [0, 4096])
    res = O.sampled_rows(qz, 0, h, w.sm_scale, [0, 77, 127], [0, 127], causal=False)
    for qb in (0, 77, 127):
        tok = slice(s + 32 * qb, s + 32 * qb + 32)
        compare("O", np64(call.o[tok, h]), res["O"][qb])
        compare("dQ", np64(call.dq[tok, h]), res["dQ"][qb])
    for kb in (0, 127):
        tok = slice(s + 32 * kb, s + 32 * kb + 32)
        compare("dK", np64(call.dk[tok, h]), res["dK"][kb])
        compare("dV", np64(call.dv[tok, h]), res["dV"][kb])
