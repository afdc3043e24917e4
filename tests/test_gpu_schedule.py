"""GPU work distribution of the persistent kernels: the static snake over
the cost-sorted item list (FLAMIA_FLAG_SCHEDULE_STATIC), the dynamic claims
(the default) and the pages' rule (FLAMIA_FLAG_SCHEDULE_RULE (review page,
sec. 3.4 "Work scheduling" and sec. 4.3: dynamic for causal calls; for
non-causal calls only when the longest document is at least 4x the average))
give the same results: O, LSE, dK and dV bit for bit (each element is
computed by one item whichever CTA takes it), dQ within the float32 atomic
order, and the oracle's values."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import compare, cu_tensor, dev, np64

pytestmark = pytest.mark.gpu

MIX = [300, 1, 129, 0, 17, 270, 33, 32, 530]


def run(w, x, **kw):
    from precision_causal_attention_block_gb300 import flamia as fl
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale, **kw)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    return call


@pytest.mark.parametrize("d,causal", [(128, True), (64, False), (128, False)])
def test_static_schedule_against_the_oracle(lib, d, causal):
    # plain data: on outlier data this seed puts one dQ element 2.7% of max|dQ|
    # off the oracle under either schedule, identically (a dS code decided in
    # float32 on the GPU and in float64 in the oracle, one E4M3 step apart,
    # times an outlier K channel); the outlier cases live in the other tests
    w = W.custom("sched_mix", MIX, 3, d, seed=41, structure="plain")
    x = W.make_inputs_bf16(w)
    call = run(w, x, causal=causal, schedule="static")
    ref = O.attention(*[x[n].double().numpy() for n in ("q", "k", "v", "do")], w.cu_seqlens,
                      w.sm_scale, causal=causal)
    for n, t in (("O", call.o), ("dQ", call.dq), ("dK", call.dk), ("dV", call.dv)):
        compare(n, np64(t), ref[n])


@pytest.mark.parametrize("wname,causal", [("fixed4x4096", True), ("fixed4x4096", False),
                                          ("varlen65536", False)])
def test_schedules_agree_at_full_size(lib, wname, causal):
    w = getattr(W, wname)()
    x = W.make_inputs_bf16(w)
    calls = {s: run(w, x, causal=causal, schedule=s) for s in ("static", "dynamic", "rule")}
    a = calls["dynamic"]
    for s in ("static", "rule"):
        b = calls[s]
        for n in ("o", "lse", "dk", "dv"):
            assert torch.equal(getattr(a, n), getattr(b, n)), (s, n)
        da, db = np64(a.dq), np64(b.dq)
        assert O.cosine(da, db) >= 0.999999
        assert np.abs(da - db).max() <= 1e-2 * np.abs(da).max()
