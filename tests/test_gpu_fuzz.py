"""Seeded random cases against the oracle: random document mixes (empty,
one-token, block-edge and tile-edge lengths among random ones), head counts,
head dims, grouped K / V heads and call options, each compared element by
element at the attention tolerances.  The case list is fixed by its seeds,
so a failure names a reproducible case."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import compare, cu_tensor, dev, np64

pytestmark = pytest.mark.gpu

EDGES = [0, 1, 2, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 384, 385]
OPTIONS = [{}, {"causal": False}, {"nvfp4_qk": True}, {"hadamard": True},
           {"deterministic_dq": True}, {"dq_accum": "fp16_causal"},
           {"dq_accum": "fp16_sequence", "causal": False}, {"schedule": "static"},
           {"ds_rows": True}, {"token_scales": True}, {"bwd_ctas": "pair"}]


def case(seed):
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(1, 9))
    lengths = [int(rng.choice(EDGES)) if rng.random() < 0.5 else int(rng.integers(0, 700))
               for _ in range(n)]
    if sum(lengths) == 0:
        lengths.append(1)
    opts = dict(OPTIONS[seed % len(OPTIONS)])
    d = int(rng.choice([64, 128]))
    if opts.get("nvfp4_qk"):
        d = 64
    if opts.get("bwd_ctas") == "pair":  # the 2-CTA backward is head dim 128's
        d = 128
    H = int(rng.choice([1, 2, 4]))
    Hkv = int(rng.choice([h for h in (1, 2, 4) if H % h == 0 and h <= H]))
    structure = str(rng.choice(["plain", "rms"]))
    return lengths, H, Hkv, d, structure, opts


@pytest.mark.parametrize("seed", range(4 * len(OPTIONS)))
def test_random_case_against_the_oracle(lib, seed):
    from precision_causal_attention_block_gb300 import flamia as fl
    lengths, H, Hkv, d, structure, opts = case(seed)
    w = W.custom(f"fuzz{seed}", lengths, H, d, structure=structure, seed=seed)
    x = W.make_inputs_bf16(w)
    x["k"], x["v"] = x["k"][:, :Hkv].contiguous(), x["v"][:, :Hkv].contiguous()
    call = fl.TrainingCall(w.T, H, d, cu_tensor(w.cu_seqlens), w.sm_scale, H_kv=Hkv, **opts)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    ref = O.attention(*[x[n].double().numpy() for n in ("q", "k", "v", "do")], w.cu_seqlens,
                      w.sm_scale, qk_format="nvfp4" if opts.get("nvfp4_qk") else "mxfp8",
                      causal=opts.get("causal", True), hadamard=opts.get("hadamard", False),
                      dq_accum=opts.get("dq_accum", "fp32"), ds_rows=opts.get("ds_rows", False),
                      group="token" if opts.get("token_scales") else "block")
    what = f"case {lengths} H={H} H_kv={Hkv} d={d} {structure} {opts}"
    rel = 3e-2 if opts.get("hadamard") else 2e-2
    for n, t in (("O", call.o), ("dQ", call.dq), ("dK", call.dk), ("dV", call.dv)):
        compare(f"{n} ({what})", np64(t), ref[n], rel_max=rel)
    lse = call.lse.cpu().numpy().astype(np.float64)
    assert np.abs(lse - ref["lse"]).max() <= 1e-4 * max(1.0, np.abs(ref["lse"]).max()), what
