"""GPU work list against the oracle, bit-exact (review page sec. 3.4 "Work
scheduling")."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import cu_tensor

pytestmark = pytest.mark.gpu

HDR_BYTES = 64


def build(cu, T):
    from precision_causal_attention_block_gb300 import flamia as fl
    ndocs = len(cu) - 1
    wl = torch.empty(fl.flamia_worklist_bytes(T, ndocs), dtype=torch.uint8, device="cuda")
    wl.fill_(0xAB)  # garbage: the builder must not rely on a cleared buffer
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fl.flamia_build_worklist(cu_tensor(cu), T, wl, dev_status=st)
    torch.cuda.synchronize()
    raw = wl.cpu().numpy()
    hdr = raw[:HDR_BYTES].view(np.int32)
    nf, nb, capf, capb = (int(v) for v in hdr[:4])
    fwd = raw[HDR_BYTES:HDR_BYTES + 16 * nf].view(np.int32).reshape(-1, 4)
    al = lambda x: (x + 255) // 256 * 256
    off_bwd = al(HDR_BYTES + 16 * capf)
    bwd = raw[off_bwd:off_bwd + 16 * nb].view(np.int32).reshape(-1, 4)
    off_tf = al(off_bwd + 16 * capb)
    off_tb = al(off_tf + 16 * capf)
    ntf, ntb = int(hdr[5]), int(hdr[6])
    tiles = (raw[off_tf:off_tf + 16 * ntf].view(np.int32).reshape(-1, 4),
             raw[off_tb:off_tb + 16 * ntb].view(np.int32).reshape(-1, 4))
    return fwd, bwd, int(st.item()), int(hdr[4]), tiles


def tile_list(items, cu, short=32):
    """The lists the tile kernels walk: the same order without the items of
    documents of at most `short` tokens (those run on the CUDA-core path)."""
    keep = [i for i, it in enumerate(items) if cu[it[0] + 1] - cu[it[0]] > short]
    return items[keep]


@pytest.mark.parametrize("cu", [
    [0, 300, 301, 1000],
    [0, 0, 5, 5, 5],
    [0, 1],
    [0, 256, 512, 513, 900, 900, 2049],
])
def test_small_lists(lib, cu):
    fwd, bwd, st, maxc, (tf, tb) = build(cu, cu[-1])
    rf, rb = O.build_worklist(cu)
    assert st == 0
    assert np.array_equal(fwd, rf) and np.array_equal(bwd, rb)
    assert maxc == (rf[0, 3] if len(rf) else 0)
    assert np.array_equal(tf, tile_list(rf, cu)) and np.array_equal(tb, tile_list(rb, cu))


@pytest.mark.parametrize("name", ["tiny", "fixed4x4096", "varlen65536", "onetoken131072",
                                  "long131072"])
def test_configs(lib, name):
    w = W.WORKLOADS[name]()
    cu = list(w.cu_seqlens)
    fwd, bwd, st, _, (tf, tb) = build(cu, w.T)
    rf, rb = O.build_worklist(cu)
    assert st == 0
    assert np.array_equal(fwd, rf) and np.array_equal(bwd, rb)
    assert np.array_equal(tf, tile_list(rf, cu)) and np.array_equal(tb, tile_list(rb, cu))


def test_bad_seqlens_flagged(lib):
    _, _, st, _, _ = build([0, 10, 5, 20], 20)
    assert st & 1
