"""GPU Hadamard rotation of Q and K (review page, sec. 3.4 "Hadamard
rotation" and "Quantization fusion": the quantiser mixes the head-dim channels
of Q and K with an orthogonal transform before the block statistics) against
the oracle: rotated codes and scale bytes bit-exact, attention outputs within
the attention tolerances, and the rotated call close to exact attention."""
import numpy as np
import pytest
import torch

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W
from tests.gpu_helpers import compare, cu_tensor, dev, np64

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "do")
RAGGED = [1, 31, 32, 33, 0, 100, 5, 300, 127, 128, 129, 2, 257]


@pytest.mark.parametrize("d", [64, 128])
def test_rotated_codes_bit_exact(lib, d):
    from precision_causal_attention_block_gb300 import flamia as fl
    w = W.custom("ragged_had", RAGGED, 3, d, structure="outlier16x2", seed=5)
    x = W.make_inputs_bf16(w)["k"]
    out = fl.QTensor(w.T, w.H, d, nvfp4=False)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fl.flamia_quantize_tokenblock(dev(x), cu_tensor(w.cu_seqlens), out,
                                  fl.FORMAT_MXFP8 | fl.FORMAT_HADAMARD, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    codes, sb = O.quantize_tokenblock(O.hadamard_fp32(x.double().numpy()), w.cu_seqlens)
    assert np.array_equal(out.scales.cpu().numpy(), sb)
    assert np.array_equal(out.codes.cpu().numpy(), codes)


def test_rotation_rejects_nvfp4_and_fused_D(lib):
    from precision_causal_attention_block_gb300 import flamia as fl
    T, H, d = 64, 1, 64
    x = torch.zeros((T, H, d), dtype=torch.bfloat16, device="cuda")
    cu = cu_tensor([0, T])
    with pytest.raises(RuntimeError):
        fl.flamia_quantize_tokenblock(x, cu, fl.QTensor(T, H, d, nvfp4=True),
                                      fl.FORMAT_MXFP8_NVFP4 | fl.FORMAT_HADAMARD)
    D = torch.empty((H, T), dtype=torch.float32, device="cuda")
    with pytest.raises(RuntimeError):
        fl.flamia_quantize_tokenblock(x, cu, fl.QTensor(T, H, d, nvfp4=False),
                                      fl.FORMAT_MXFP8 | fl.FORMAT_HADAMARD, o=x, D=D)


def run_call(w, x):
    from precision_causal_attention_block_gb300 import flamia as fl
    call = fl.TrainingCall(w.T, w.H, w.d, cu_tensor(w.cu_seqlens), w.sm_scale, hadamard=True)
    xd = {n: dev(t) for n, t in x.items()}
    call.forward(xd["q"], xd["k"], xd["v"])
    call.backward(xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    return call


@pytest.mark.parametrize("d", [64, 128])
def test_rotated_attention_against_the_oracle(lib, d):
    # long documents (tensor-core kernels) beside short ones (CUDA-core kernels)
    w = W.custom("had_attn", [300, 1, 129, 0, 17, 270, 33, 32], 2, d, seed=9,
                 structure="outlier16x2")
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    xs = [x[n].double().numpy() for n in NAMES]
    ref = O.attention(*xs, w.cu_seqlens, w.sm_scale, hadamard=True)
    qz = ref["quantized"]
    assert np.array_equal(call.q.codes.cpu().numpy(), qz.qc)
    assert np.array_equal(call.k.scales.cpu().numpy(), qz.ks)
    gpu = {"O": call.o, "dQ": call.dq, "dK": call.dk, "dV": call.dv}
    for n in ("O", "dQ", "dK", "dV"):
        compare(n, np64(gpu[n]), ref[n], rel_max=ROTATED_REL_MAX[n])
    lse = call.lse.cpu().numpy().astype(np.float64)
    assert np.abs(lse - ref["lse"]).max() <= 1e-4 * max(1.0, np.abs(ref["lse"]).max())


@pytest.mark.parametrize("d", [64, 128])
def test_rotated_attention_tracks_exact_attention(lib, d):
    # on plain normal inputs the rotated method is as close to exact attention
    # as the unrotated one (within 5e-4 in cosine).  (With a few x16 channels
    # in every token the E4M3 blocks already cope without rotation, and the
    # rotation, which gives every channel a share of the outliers, lowers the
    # cosine from about 0.995 to 0.985: the oracle shows the same.)
    w = W.custom("had_plain", [300, 1, 129, 0, 17, 270, 33, 32], 2, d, seed=9, structure="plain")
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    xs = [x[n].double().numpy() for n in NAMES]
    ex = O.attention(*xs, w.cu_seqlens, w.sm_scale, quant=False)
    plain = O.attention(*xs, w.cu_seqlens, w.sm_scale)
    gpu = {"O": call.o, "dQ": call.dq, "dK": call.dk, "dV": call.dv}
    for n in ("O", "dQ", "dK", "dV"):
        assert O.cosine(np64(gpu[n]), ex[n]) >= O.cosine(plain[n], ex[n]) - 5e-4, n
        assert O.cosine(np64(gpu[n]), ex[n]) >= 0.997, n


def test_rotated_fixed4x4096_one_document(lib):
    """The full-size shape's kernels (head dim 128, 4096-token documents) with
    the rotation, the pages' default at head dim 128 (review page, sec. 3.4),
    against the oracle and against exact attention on one document.  Head 1
    (a x20 channel in dO only) reaches cosine >= 0.998 to exact attention on
    all four outputs, and so does the kernel.  Head 13 has x20 channels in Q,
    K and V: there the method itself stays below 0.998 (the rotation spreads
    the Q and K outliers over every channel; the oracle gives dK 0.911), so
    the kernel is held to the oracle's own distance from exact attention."""
    w = W.fixed4x4096()
    x = W.make_inputs_bf16(w)
    call = run_call(w, x)
    tok, heads = slice(4096, 8192), [1, 13]
    xs = [x[n][tok][:, heads].double().numpy() for n in NAMES]
    ref = O.attention(*xs, [0, 4096], w.sm_scale, hadamard=True)
    ex = O.attention(*xs, [0, 4096], w.sm_scale, quant=False)
    gpu = {"O": call.o, "dQ": call.dq, "dK": call.dk, "dV": call.dv}
    for n in ("O", "dQ", "dK", "dV"):
        got = np64(gpu[n][tok][:, heads])
        compare(n, got, ref[n], rel_max=ROTATED_REL_MAX[n])
        assert O.cosine(got[:, 0], ex[n][:, 0]) >= 0.998, (n, "head 1")
        method = O.cosine(ref[n][:, 1], ex[n][:, 1])
        assert O.cosine(got[:, 1], ex[n][:, 1]) >= method - 2e-4, (n, "head 13", method)


# The rotation back makes every element of dQ and dK a +-1 sum over all d
# columns of dQ_r / dK_r, so the GPU's and the oracle's few differing dS codes
# (round-to-nearest ties decided in float32 on the GPU) land in every element
# of the row, while the largest element of the reference shrinks towards the
# row's RMS: the max-error bound of the unrotated outputs (2e-2 of the largest
# reference element) becomes 3e-2 for these two.
ROTATED_REL_MAX = {"O": 2e-2, "dV": 2e-2, "dQ": 3e-2, "dK": 3e-2}
