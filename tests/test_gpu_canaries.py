"""Guard bytes around every buffer a training call writes (compute-sanitizer
is not available on the GPU pool: this is the out-of-bounds check).  Each
output, workspace and quantised operand is a view into a larger allocation
whose margins hold a known pattern; after a full call on ragged documents
(a T that is not a multiple of any tile, documents of 1 to 33 tokens, empty
documents) the margins must be unchanged, in every mode of the call."""
import pytest
import torch

from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import cu_tensor, dev

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side (keeps the 256-byte alignment of the view)
PATTERN = 0xA5
MIX = [300, 1, 129, 0, 17, 270, 33, 32, 131]


class Guarded:
    def __init__(self):
        self.bases = []

    def __call__(self, t):
        """A guarded copy of t's shape and dtype (contents undefined)."""
        if t is None:
            return None
        nbytes = t.numel() * t.element_size()
        base = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=t.device)
        self.bases.append((base, nbytes))
        return base[GUARD:GUARD + nbytes].view(t.dtype).view(t.shape)

    def check(self):
        for i, (base, nbytes) in enumerate(self.bases):
            head, tail = base[:GUARD], base[GUARD + nbytes:]
            assert bool((head == PATTERN).all()) and bool((tail == PATTERN).all()), i


@pytest.mark.parametrize("d,Hkv,kw", [
    (128, None, {}),
    (64, None, {}),
    (64, None, {"nvfp4_qk": True}),
    (128, 2, {"causal": False}),
    (128, None, {"hadamard": True}),
    (128, None, {"deterministic_dq": True, "dq_accum": "fp16_causal"}),
    (64, 2, {"dq_accum": "fp16_sequence"}),
])
def test_no_write_outside_the_buffers(lib, d, Hkv, kw):
    from precision_causal_attention_block_gb300 import flamia as fl
    w = W.custom("guard", MIX, 4, d, seed=37)
    x = W.make_inputs_bf16(w)
    hkv = Hkv or w.H
    x["k"], x["v"] = x["k"][:, :hkv].contiguous(), x["v"][:, :hkv].contiguous()
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale, H_kv=Hkv, **kw)
    g = Guarded()
    for qt in (call.q, call.k, call.v, call.dout):
        for name in ("codes", "scales", "nvfp4_codes", "nvfp4_scales"):
            setattr(qt, name, g(getattr(qt, name)))
    for name in ("wl", "ws", "o", "lse", "D", "dq", "dk", "dv"):
        setattr(call, name, g(getattr(call, name)))
    xd = {n: dev(t) for n, t in x.items()}
    for _ in range(2):  # the second call reuses the work list's counters
        call.forward(xd["q"], xd["k"], xd["v"])
        call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    g.check()
