"""Failure detection on the GPU without a fault: the library's bounded waits
(an mbarrier that nothing completes, a dQ turn that nothing passes) give up
after their time limit, report FLAMIA_DEV_TIMEOUT in the status word and
return; the context stays usable, as a correct call right after shows."""
import time

import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import compare, cu_tensor, dev, np64

pytestmark = pytest.mark.gpu


def test_bounded_waits_time_out_and_report(lib):
    from precision_causal_attention_block_gb300 import flamia as fl
    turn = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    fl.flamia_debug_bounded_waits(turn, st)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == fl.DEV_TIMEOUT
    assert 3.5 <= dt <= 60.0, dt  # two waits of about 2 s each
    # the same context runs a call correctly afterwards
    w = W.custom("after_timeout", [200, 17, 90], 2, 64, seed=3)
    x = W.make_inputs_bf16(w)
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    ref = O.attention(*[x[n].double().numpy() for n in ("q", "k", "v", "do")], w.cu_seqlens,
                      w.sm_scale)
    for n, t in (("O", call.o), ("dQ", call.dq), ("dK", call.dk), ("dV", call.dv)):
        compare(n, np64(t), ref[n])
    assert np.isfinite(np64(call.o)).all()
