"""Seeded synthetic inputs for the packed causal attention workloads.

This module only draws numbers: it holds none of the attention or quantisation
arithmetic, so both the CUDA path and the CPU oracle can take their inputs from
it without sharing any of the method.

Shapes follow the FLAMIA pages' packed causal workloads (16 heads, head dim
128; a one-document 131,072-token row; one-token documents for the
work-list stress case).  The pages measure on captured activations that are
not available here, so these draws stand in for them:

* every tensor is BF16, rounded to nearest-even from float32 standard normals
  drawn with ``numpy.random.default_rng(seed)``;
* the draw order is: document lengths (variable-length case only), then Q, K,
  V, dO, each followed by its own structure draw (outlier channels or per-head
  RMS).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

TENSOR_NAMES = ("q", "k", "v", "do")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    d: int
    cu_seqlens: tuple  # int document offsets, len = ndocs + 1
    sm_scale: float
    structure: str      # "outlier16x2" | "outlier20pct1" | "plain" | "rms"
    seed: int = 0

    @property
    def ndocs(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def doc_lengths(self):
        c = self.cu_seqlens
        return [c[i + 1] - c[i] for i in range(len(c) - 1)]

    @property
    def sum_sq_len(self) -> int:
        return sum(L * L for L in self.doc_lengths)

    def causal_flops(self) -> float:
        """fwd 4*H*d*L^2/2 + bwd 10*H*d*L^2/2 (causal half of the L^2 pairs)."""
        return 7.0 * self.H * self.d * self.sum_sq_len


def loguniform_lengths(rng, total: int, max_len: int):
    """Document lengths drawn log-uniform in [1, max_len] until they fill ``total``."""
    out, acc = [], 0
    while acc < total:
        u = rng.uniform(0.0, math.log(max_len))
        n = int(min(max(round(math.exp(u)), 1), max_len))
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def offsets(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    return tuple(cu)


def tiny():
    """1 document, T=256, H=2, d=64; 2 of 64 channels x16 per tensor."""
    return Workload("tiny_T256_H2_d64", 256, 2, 64, (0, 256), 1.0 / 8.0, "outlier16x2")


def fixed4x4096():
    """4 equal documents of 4096 tokens, H=16, d=128; 1% of H*d channels x20."""
    return Workload("fixed_4x4096_H16_d128", 16384, 16, 128,
                    (0, 4096, 8192, 12288, 16384), 1.0 / math.sqrt(128.0), "outlier20pct1")


def varlen65536(seed: int = 0):
    """65,536 tokens in log-uniform documents of 1..16384 tokens, H=16, d=128."""
    rng = np.random.default_rng(seed)
    cu = offsets(loguniform_lengths(rng, 65536, 16384))
    return Workload("varlen_65536_H16_d128", 65536, 16, 128, cu,
                    1.0 / math.sqrt(128.0), "plain", seed)


def onetoken131072():
    """131,072 one-token documents, H=16, d=128."""
    return Workload("onetoken_131072_H16_d128", 131072, 16, 128,
                    tuple(range(131073)), 1.0 / math.sqrt(128.0), "plain")


def long131072():
    """One causal document of 131,072 tokens, H=32, d=64; per-head RMS in [0.5, 2]."""
    return Workload("long_131072_H32_d64", 131072, 32, 64, (0, 131072), 1.0 / 8.0, "rms")


def long16384():
    """The long-context shape cut to one 16,384-token document (H=32, d=64, per-head
    RMS in [0.5, 2]): a case small enough for detailed kernel profiles."""
    return Workload("long_16384_H32_d64", 16384, 32, 64, (0, 16384), 1.0 / 8.0, "rms")


def skewed8192():
    """The training-call table's most skewed packing: one 8,192-token document
    followed by 224 documents of 256 tokens (T = 65,536), H=16, d=128."""
    return Workload("skewed_8192_224x256_H16_d128", 65536, 16, 128,
                    offsets([8192] + [256] * 224), 1.0 / math.sqrt(128.0), "plain")


def custom(name, lengths, H, d, structure="plain", seed=0, sm_scale=None):
    """Small ragged cases for parity tests."""
    cu = offsets(lengths)
    return Workload(name, cu[-1], H, d, cu,
                    sm_scale if sm_scale is not None else 1.0 / math.sqrt(d), structure, seed)


WORKLOADS = {
    "tiny": tiny,
    "fixed4x4096": fixed4x4096,
    "varlen65536": varlen65536,
    "onetoken131072": onetoken131072,
    "long131072": long131072,
    "long16384": long16384,
    "skewed8192": skewed8192,
}


def _draw_tensor(rng, w: Workload) -> np.ndarray:
    x = rng.standard_normal((w.T, w.H, w.d), dtype=np.float32)
    if w.structure == "outlier16x2":
        ch = rng.choice(w.d, 2, replace=False)
        x[:, :, ch] *= 16.0
    elif w.structure == "outlier20pct1":
        n = max(1, round(0.01 * w.H * w.d))
        flat = rng.choice(w.H * w.d, n, replace=False)
        for c in flat:
            x[:, c // w.d, c % w.d] *= 20.0
    elif w.structure == "rms":
        rms = rng.uniform(0.5, 2.0, size=w.H).astype(np.float32)
        x *= rms[None, :, None]
    elif w.structure != "plain":
        raise ValueError(w.structure)
    return x


def _skip_lengths(rng, w: Workload):
    # The variable-length case drew its lengths from the same generator first.
    if w.name.startswith("varlen"):
        loguniform_lengths(rng, w.T, 16384)


def make_inputs_f32(w: Workload):
    """Q, K, V, dO as float32 numpy arrays [T, H, d] (not yet rounded to BF16)."""
    rng = np.random.default_rng(w.seed)
    _skip_lengths(rng, w)
    return {n: _draw_tensor(rng, w) for n in TENSOR_NAMES}


def make_inputs_bf16(w: Workload):
    """Q, K, V, dO as torch.bfloat16 CPU tensors [T, H, d] (round-to-nearest-even)."""
    import torch
    out = {}
    rng = np.random.default_rng(w.seed)
    _skip_lengths(rng, w)
    for n in TENSOR_NAMES:
        out[n] = torch.from_numpy(_draw_tensor(rng, w)).to(torch.bfloat16)
    return out


def cu_seqlens_array(w: Workload) -> np.ndarray:
    return np.asarray(w.cu_seqlens, dtype=np.int32)
