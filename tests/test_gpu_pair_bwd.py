"""The 2-CTA backward (review page, sec. 3.4 "Backward pass": a cluster of two
CTAs splits 256 keys and runs its products together) against the FP64 oracle
at the attention tolerances, and against the one-CTA backward of the same
call: the same codes and products per key row, so dK and dV agree to one
BF16 step of each element, and dQ (summed over the pair's 256 keys before its
reduce-add, where one-CTA items add two 128-key partials in either order) to
two."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import compare, cu_tensor, dev, np64

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "do")
# documents whose last 256-key item has no keys in the second CTA (129, 270,
# 300), exactly 256 keys (256, 512), one 128-key tile (33, 100), short ones
MIX = [300, 1, 129, 0, 17, 270, 33, 32, 256, 100, 512, 2]


def run(w, x, ctas, Hkv=None, **kw):
    from precision_causal_attention_block_gb300 import flamia as fl
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale, H_kv=Hkv,
                           bwd_ctas=ctas, **kw)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    return call


@pytest.mark.parametrize("kw", [{}, {"causal": False}, {"hadamard": True}])
def test_pair_against_the_oracle(lib, kw):
    w = W.custom("pair_mix", MIX, 2, 128, seed=33, structure="outlier16x2")
    x = W.make_inputs_bf16(w)
    call = run(w, x, "pair", **kw)
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale,
                      causal=kw.get("causal", True), hadamard=kw.get("hadamard", False))
    rel = 3e-2 if kw.get("hadamard") else 2e-2
    for n, t in (("O", call.o), ("dQ", call.dq), ("dK", call.dk), ("dV", call.dv)):
        compare(n, np64(t), ref[n], rel_max=rel)


def test_pair_grouped_heads(lib):
    w = W.custom("pair_gqa", [700, 17, 300], 4, 128, seed=13)
    x = W.make_inputs_bf16(w)
    x["k"], x["v"] = x["k"][:, :2].contiguous(), x["v"][:, :2].contiguous()
    call = run(w, x, "pair", Hkv=2)
    ref = O.attention(*[x[n].double().numpy() for n in NAMES], w.cu_seqlens, w.sm_scale)
    for n, t in (("O", call.o), ("dQ", call.dq), ("dK", call.dk), ("dV", call.dv)):
        compare(n, np64(t), ref[n])


def _within_bf16_ulps(a, b, ulps):
    """Elementwise |a - b| within `ulps` BF16 spacings of the larger magnitude
    (2^-7 relative per spacing at most), plus float32 noise near zero."""
    lim = ulps * 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-6 * np.abs(a).max()
    return bool(np.all(np.abs(a - b) <= lim))


def _against_one_cta(w, x, **kw):
    a = run(w, x, "one", **kw)
    b = run(w, x, "pair", **kw)
    for n in ("dk", "dv"):
        assert _within_bf16_ulps(np64(getattr(a, n)), np64(getattr(b, n)), 1), n
    # dQ: 256-key sums before one reduce-add against two 128-key partials
    # added in either order, each rounded to BF16 at the end
    assert _within_bf16_ulps(np64(a.dq), np64(b.dq), 2)
    return a, b


def test_pair_matches_one_cta_ragged(lib):
    w = W.custom("pair_vs_one", MIX, 3, 128, seed=5, structure="outlier16x2")
    _against_one_cta(w, W.make_inputs_bf16(w))


def test_pair_fixed4x4096(lib):
    """The 4 x 4096 workload in the pair mode: one document x two heads
    against the oracle, everything against the one-CTA backward."""
    w = W.fixed4x4096()
    x = W.make_inputs_bf16(w)
    _, b = _against_one_cta(w, x)
    heads = [0, 9]
    s, e = 4096, 8192
    ref = O.attention(*[x[n][s:e][:, heads].double().numpy() for n in NAMES], [0, e - s],
                      w.sm_scale)
    for n, t in (("dQ", b.dq), ("dK", b.dk), ("dV", b.dv)):
        compare(n, np64(t[s:e][:, heads]), ref[n])


def test_pair_varlen65536_sampled(lib):
    w = W.varlen65536()
    x = W.make_inputs_bf16(w)
    _, b = _against_one_cta(w, x)
    cu = list(w.cu_seqlens)
    lens = np.diff(cu)
    i = int(np.argmin(np.abs(lens - 1500)))
    s, e = cu[i], cu[i + 1]
    heads = [5]
    ref = O.attention(*[x[n][s:e][:, heads].double().numpy() for n in NAMES], [0, e - s],
                      w.sm_scale)
    for n, t in (("dQ", b.dq), ("dK", b.dk), ("dV", b.dv)):
        compare(n, np64(t[s:e][:, heads]), ref[n])


def test_pair_flag_rejects_other_modes(lib):
    from precision_causal_attention_block_gb300 import flamia as fl
    w = W.custom("pair_rej", [300], 1, 128, seed=1)
    x = W.make_inputs_bf16(w)
    for kw in ({"deterministic_dq": True}, {"dq_accum": "fp16_causal"}, {"ds_rows": True},
               {"schedule": "static"}):
        with pytest.raises(RuntimeError, match="unsupported"):
            run(w, x, "pair", **kw)
    w64 = W.custom("pair_rej64", [300], 1, 64, seed=1)
    with pytest.raises(RuntimeError, match="unsupported"):
        run(w64, W.make_inputs_bf16(w64), "pair")
