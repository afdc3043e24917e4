"""A call past 2^31 elements: T = 2^20 tokens x 32 heads x head dim 64
(256 documents of 4096 tokens), so every element offset and byte offset of
the [T, H, d] tensors needs 64 bits.  The first and the last documents
(first and last heads) against the oracle, and a clean device status."""
import pytest
import torch

from oracle import flamia_oracle as O
from tests.gpu_helpers import compare, np64

pytestmark = pytest.mark.gpu

T, H, D, L = 1 << 20, 32, 64, 4096


def test_more_than_2_31_elements(lib):
    from precision_causal_attention_block_gb300 import flamia as fl
    assert T * H * D == 1 << 31
    g = torch.Generator(device="cuda")
    g.manual_seed(123)
    x = {n: torch.randn((T, H, D), generator=g, device="cuda").to(torch.bfloat16)
         for n in ("q", "k", "v", "do")}
    cu = torch.arange(0, T + 1, L, dtype=torch.int32, device="cuda")
    scale = D ** -0.5
    call = fl.TrainingCall(T, H, D, cu, scale)
    call.forward(x["q"], x["k"], x["v"])
    call.backward(x["do"])
    torch.cuda.synchronize()
    call.check_status()
    for s in (0, T - L):
        for h in (0, H - 1):
            sl = [x[n][s:s + L, h:h + 1].double().cpu().numpy() for n in ("q", "k", "v", "do")]
            ref = O.attention(*sl, [0, L], scale)
            for n, t in (("O", call.o), ("dQ", call.dq), ("dK", call.dk), ("dV", call.dv)):
                compare(f"{n}[{s}, {h}]", np64(t[s:s + L, h:h + 1]), ref[n])
