"""GPU grouped-query attention (K / V heads shared by groups of query heads:
the attention API the pages' method serves) against the oracle's grouped
heads: forward and backward at the attention tolerances, dK / dV of a K / V
head summed over its query heads, on the tensor-core kernels and the
short-document kernels, with the non-causal and rotated variants."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import compare, cu_tensor, dev, np64

pytestmark = pytest.mark.gpu

MIX = [300, 1, 129, 0, 17, 270, 33, 32, 130]


def inputs(w, Hkv):
    x = W.make_inputs_bf16(w)
    x["k"] = x["k"][:, :Hkv].contiguous()
    x["v"] = x["v"][:, :Hkv].contiguous()
    return x


def run(w, x, Hkv, **kw):
    from precision_causal_attention_block_gb300 import flamia as fl
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale, H_kv=Hkv, **kw)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    return call


@pytest.mark.parametrize("d,H,Hkv,kw", [
    (128, 6, 2, {}),
    (64, 4, 1, {}),
    (64, 4, 2, {"nvfp4_qk": True}),
    (128, 4, 2, {"causal": False}),
    (64, 6, 3, {"hadamard": True}),
])
def test_gqa_against_the_oracle(lib, d, H, Hkv, kw):
    w = W.custom("gqa_mix", MIX, H, d, seed=19, structure="outlier16x2")
    x = inputs(w, Hkv)
    call = run(w, x, Hkv, **kw)
    ref = O.attention(*[x[n].double().numpy() for n in ("q", "k", "v", "do")], w.cu_seqlens,
                      w.sm_scale, qk_format="nvfp4" if kw.get("nvfp4_qk") else "mxfp8",
                      causal=kw.get("causal", True), hadamard=kw.get("hadamard", False))
    assert call.dk.shape == (w.T, Hkv, d)
    rel = {"O": 2e-2, "dV": 2e-2, "dQ": 3e-2 if kw.get("hadamard") else 2e-2,
           "dK": 3e-2 if kw.get("hadamard") else 2e-2}
    gpu = {"O": call.o, "dQ": call.dq, "dK": call.dk, "dV": call.dv}
    for n in ("O", "dQ", "dK", "dV"):
        compare(n, np64(gpu[n]), ref[n], rel_max=rel[n])
    lse = call.lse.cpu().numpy().astype(np.float64)
    assert np.abs(lse - ref["lse"]).max() <= 1e-4 * max(1.0, np.abs(ref["lse"]).max())


def test_gqa_one_group_equals_multi_head(lib):
    # H_kv = H through the grouped entry points is the multi-head call, bit for bit
    from precision_causal_attention_block_gb300 import flamia as fl
    w = W.custom("gqa_mha", [200, 31, 90], 2, 64, seed=23)
    x = W.make_inputs_bf16(w)
    a = run(w, x, 2)
    b = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale)
    xd = {n: dev(t) for n, t in x.items()}
    b.q, b.k, b.v = a.q, a.k, a.v  # same quantised operands
    fl.flamia_attn_fwd(b.q, b.k, b.v, b.cu, b.T, b.H, b.d, b.scale, a.wl, b.o, b.lse,
                       dev_status=b.status)
    torch.cuda.synchronize()
    assert torch.equal(a.o, b.o) and torch.equal(a.lse, b.lse)
