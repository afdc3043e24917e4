"""Shared helpers of the GPU parity tests: device transfer and oracle runs on
self-contained slices (documents are independent, so the oracle can run on
one document's tokens and a subset of heads)."""
import numpy as np
import torch

from oracle import flamia_oracle as O

DEV = "cuda"


def dev(t):
    return t.to(DEV)


def cu_tensor(cu):
    return torch.tensor(list(cu), dtype=torch.int32, device=DEV)


def np64(t):
    return t.detach().double().cpu().numpy()


def oracle_slice(x, s, e, heads, local_cu, sm_scale, quant=True, qk_format="mxfp8"):
    """Oracle forward+backward of tokens [s, e) on the listed heads; local_cu
    are the document offsets inside the slice (the slice must hold whole
    documents, or, for one long document, start on a 32-token boundary of it
    and be used only for the forward rows it fully contains)."""
    sl = [x[n][s:e][:, heads].double().numpy() for n in ("q", "k", "v", "do")]
    return O.attention(*sl, local_cu, sm_scale, quant=quant, qk_format=qk_format)


def compare(name, got, ref, cos_min=0.9995, rel_max=2e-2):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    cos = O.cosine(got, ref)
    denom = np.abs(ref).max()
    err = np.abs(got - ref).max() / denom if denom > 0 else np.abs(got).max()
    assert cos >= cos_min and err <= rel_max, f"{name}: cosine {cos:.6f}, max rel err {err:.3e}"
    return cos, err
