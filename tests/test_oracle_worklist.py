"""Pins of the oracle's work list.

Source: "FLAMIA ... (jaehun.me review)", sec. 3.4 "Work scheduling": a work
item is 256 consecutive queries of one document, its cost the number of key
blocks it visits, sorted by descending cost."""
import os

import numpy as np

from oracle import flamia_oracle as O
from precision_causal_attention_block_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_small_golden():
    want = {"fwd": [], "bwd": []}
    with open(os.path.join(GOLDEN, "worklist_small.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                kind, *vals = line.split()
                want[kind].append([int(v) for v in vals])
    fwd, bwd = O.build_worklist([0, 300, 301, 1000])
    assert fwd.tolist() == want["fwd"]
    assert bwd.tolist() == want["bwd"]


def _generated(cu):
    fwd, bwd = [], []
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        fwd += [(b, q0) for q0 in range(s, e, 256)]
        bwd += [(b, k0) for k0 in range(s, e, 128)]
    return fwd, bwd


def test_varlen_recipe_facts():
    w = W.varlen65536()
    assert w.ndocs == 30 and max(w.doc_lengths) == 15946 and w.sum_sq_len == 620059716
    assert w.T == 65536 and min(w.doc_lengths) >= 1


def test_invariants_on_the_varlen_workload():
    cu = list(W.varlen65536().cu_seqlens)
    fwd, bwd = O.build_worklist(cu)
    gf, gb = _generated(cu)
    for items, gen, tile in ((fwd, gf, 256), (bwd, gb, 128)):
        # a permutation of the generated items
        assert sorted((int(a), int(b)) for a, b, _, _ in items) == sorted(gen)
        cost = items[:, 3]
        assert np.all(np.diff(cost) <= 0)                       # descending
        order = {g: i for i, g in enumerate(gen)}
        for c in np.unique(cost):                               # stable
            pos = [order[(int(a), int(b))] for a, b, _, cc in items if cc == c]
            assert pos == sorted(pos)
        # items cover each document exactly once, end clipped to the document
        for b, st, en, c in items:
            assert cu[b] <= st < en <= cu[b + 1] and en - st <= tile
    # costs: forward = key blocks seen by the last query, backward = query blocks seeing the tile
    for b, q0, q1, c in fwd:
        assert c == -(-(q1 - cu[b]) // 128)
    for b, k0, k1, c in bwd:
        assert c == -(-(cu[b + 1] - k0) // 128)
    assert len(fwd) == 276 and len(bwd) == 532


def test_closed_form_one_token_documents():
    n = 131072
    fwd, bwd = O.build_worklist(list(range(n + 1)))
    want = np.stack([np.arange(n), np.arange(n), np.arange(1, n + 1), np.ones(n, int)], 1)
    assert np.array_equal(fwd, want) and np.array_equal(bwd, want)


def test_empty_documents_give_no_items():
    fwd, bwd = O.build_worklist([0, 0, 5, 5, 5])
    assert fwd.tolist() == [[1, 0, 5, 1]] and bwd.tolist() == [[1, 0, 5, 1]]
    fwd, bwd = O.build_worklist([0])
    assert fwd.shape == (0, 4) and bwd.shape == (0, 4)
