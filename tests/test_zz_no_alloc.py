"""The allocation-free work-list entry point (flamia_build_worklist_static).

It exists for callers that cannot allocate device memory (a framework whose
caching allocator owns the device memory, a plugin host without an allocator,
a loop that cannot take cudaMalloc's device synchronisation): its scratch is a
fixed 8 MiB array in the library.  It must give exactly the output of
flamia_build_worklist, call after call, whatever an earlier call left in the
shared array.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from precision_causal_attention_block_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _lists(wl_u8):
    raw = wl_u8.cpu().numpy()
    hdr = raw[:64].view(np.int32)
    nf, nb, capf, capb = int(hdr[0]), int(hdr[1]), int(hdr[2]), int(hdr[3])
    al = lambda x: (x + 255) // 256 * 256
    fwd = raw[64:64 + 16 * nf].view(np.int32).reshape(-1, 4)
    off_bwd = al(64 + 16 * capf)
    bwd = raw[off_bwd:off_bwd + 16 * nb].view(np.int32).reshape(-1, 4)
    # the lists without short documents follow, sized by header words 5 and 6
    off_tf = al(off_bwd + 16 * capb)
    off_tb = al(off_tf + 16 * capf)
    tf = raw[off_tf:off_tf + 16 * int(hdr[5])]
    tb = raw[off_tb:off_tb + 16 * int(hdr[6])]
    return hdr[:7].copy(), np.concatenate([fwd.ravel(), tf.view(np.int32)]), \
        np.concatenate([bwd.ravel(), tb.view(np.int32)])


def _call_both(lib, cu_list, T):
    from precision_causal_attention_block_gb300 import flamia as fl
    cu = torch.tensor(cu_list, dtype=torch.int32, device="cuda")
    n = fl.flamia_worklist_bytes(T, len(cu_list) - 1)
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    ref = torch.full((n,), 0x5A, dtype=torch.uint8, device="cuda")
    fl.flamia_build_worklist(cu, T, ref, dev_status=st[0:1])
    out = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")
    # through the C ABI directly
    rc = lib.flamia_build_worklist_static(ctypes.c_void_p(cu.data_ptr()), len(cu_list) - 1, T,
                                          ctypes.c_void_p(out.data_ptr()), n,
                                          ctypes.c_void_p(st[1:2].data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0]
    return _lists(ref), _lists(out)


def test_matches_the_allocating_builder_twice_in_a_row(lib):
    from oracle import flamia_oracle as O
    cases = [list(W.varlen65536().cu_seqlens), [0, 300, 301, 1000], list(W.onetoken131072().cu_seqlens)]
    for cu in cases:  # consecutive calls reuse the same static scratch
        (h0, f0, b0), (h1, f1, b1) = _call_both(lib, cu, cu[-1])
        assert np.array_equal(h0, h1)
        assert np.array_equal(f0, f1) and np.array_equal(b0, b1)
        assert len(f0) > 0
        # and both are the oracle's lists (the item arrays lead each vector)
        rf, rb = O.build_worklist(cu)
        assert np.array_equal(f1[:rf.size], rf.ravel()) and np.array_equal(b1[:rb.size], rb.ravel())


def test_rejects_layouts_beyond_the_static_scratch(lib):
    """A million one-token documents need more scratch than the array holds:
    the call returns FLAMIA_ERR_WORKSPACE before launching anything.  Every
    buffer passed is real and of its declared size."""
    from precision_causal_attention_block_gb300 import flamia as fl
    T = 1 << 20
    cu = torch.arange(T + 1, dtype=torch.int32, device="cuda")
    n = fl.flamia_worklist_bytes(T, T)
    wl = torch.zeros(n, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.flamia_build_worklist_static(ctypes.c_void_p(cu.data_ptr()), T, T,
                                          ctypes.c_void_p(wl.data_ptr()), n,
                                          ctypes.c_void_p(st.data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 3  # FLAMIA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(wl.count_nonzero().item()) == 0
