"""The C-ABI library builds, loads without a GPU, exports every declared
symbol, and rejects bad arguments on the host (no kernel is launched)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cpu_lib():
    from precision_causal_attention_block_gb300 import build, flamia
    build.build()
    return flamia.load()


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(flamia_[a-z_0-9]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(cpu_lib):
    names = declared_symbols()
    assert "flamia_attn_fwd" in names and "flamia_quantize_tokenblock" in names
    for n in names:
        assert hasattr(cpu_lib, n), n


def test_size_queries(cpu_lib):
    from precision_causal_attention_block_gb300 import flamia as fl
    # float32 dQ accumulator, int32 turn counters, int8 prescale table, 3 H
    # ints, each 256-byte padded
    th = 16384 * 16
    # (+ 256 bytes for the two dS counters at the end)
    assert fl.flamia_bwd_workspace_bytes(16384, 16, 128) == th * 128 * 4 + th * 4 + th + 512
    assert fl.flamia_bwd_workspace_bytes(3, 1, 64) == 768 + 256 + 256 + 256 + 256
    assert fl.flamia_bwd_ds_counts_offset(3, 1, 64) == 768 + 256 + 256 + 256
    assert fl.flamia_bwd_workspace_bytes(10, 1, 96) == 0
    wl = fl.flamia_worklist_bytes(65536, 30)
    assert wl >= 64 + 16 * (65536 // 256 + 31) + 16 * (65536 // 128 + 31)
    assert fl.flamia_worklist_bytes(0, 1) == 0
    # the forward needs no workspace at any size
    assert fl.flamia_fwd_workspace_bytes(16384, 16, 128) == 0
    assert fl.flamia_fwd_workspace_bytes(1 << 20, 32, 64) == 0


def test_status_strings(cpu_lib):
    for s in range(5):
        assert cpu_lib.flamia_status_str(s)
    assert cpu_lib.flamia_status_str(99) == b"unknown status"


def test_host_side_argument_checks(cpu_lib):
    from precision_causal_attention_block_gb300 import flamia as fl
    q = fl.QTensorStruct()
    null = ctypes.c_void_p(None)
    # unsupported head dim
    assert cpu_lib.flamia_quantize_tokenblock(null, 16, 1, 96, null, 1, 0, null, null,
                                              ctypes.byref(q), null, null) == 2
    # null input
    assert cpu_lib.flamia_quantize_tokenblock(null, 16, 1, 64, null, 1, 0, null, null,
                                              ctypes.byref(q), null, null) == 1
    # work list: null / buffer too small / more tokens than the one limit
    # (real, if host-side, buffers: these checks return before any launch)
    assert cpu_lib.flamia_build_worklist(null, 1, 16, null, 0, null, null) == 1
    cu = np.array([0, 16], dtype=np.int32)
    big = np.zeros(fl.flamia_worklist_bytes(16, 1) + 256, dtype=np.uint8)
    big_al = ctypes.c_void_p((big.ctypes.data + 255) // 256 * 256)
    assert cpu_lib.flamia_build_worklist(cu.ctypes.data_as(ctypes.c_void_p), 1, 16, big_al, 8,
                                         null, null) == 3
    for fn in (cpu_lib.flamia_build_worklist, cpu_lib.flamia_build_worklist_static):
        assert fn(cu.ctypes.data_as(ctypes.c_void_p), 1, (1 << 20) + 1, big_al, big.nbytes - 256,
                  null, null) == 1
    assert cpu_lib.flamia_quantize_tokenblock(null, (1 << 20) + 1, 1, 64, null, 1, 0, null,
                                              null, ctypes.byref(q), null, null) == 1
    # flags not supported (an unknown bit; static and dynamic scheduling at
    # once; the ordered dQ turns with the static schedule) / bad scale
    for flags in (0x4000, 0x40 | 0x80, 0x800):  # the CTA-pair flag is the backward's
        assert cpu_lib.flamia_attn_fwd(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), null, 1,
                                       16, 1, 64, ctypes.c_float(0.1), flags, null, null, null,
                                       null, null) == 2
    assert cpu_lib.flamia_attn_bwd(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q),
                                   ctypes.byref(q), null, null, null, 1, 16, 1, 64,
                                   ctypes.c_float(0.1), 0x8 | 0x40, null, null, null, null, null,
                                   0, null, null) == 2
    assert cpu_lib.flamia_attn_bwd(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q),
                                   ctypes.byref(q), null, null, null, 1, 16, 1, 64,
                                   ctypes.c_float(-1.0), 0, null, null, null, null, null, 0, null,
                                   null) == 1
    # the 2-CTA backward: not with head dim 64, the ordered dQ, query-row dS
    # exponents, or the one-CTA flag
    for d, flags in ((64, 0x800), (128, 0x800 | 0x8), (128, 0x800 | 0x100), (128, 0x800 | 0x1000)):
        assert cpu_lib.flamia_attn_bwd(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q),
                                       ctypes.byref(q), null, null, null, 1, 16, 1, d,
                                       ctypes.c_float(0.1), flags, null, null, null, null, null,
                                       0, null, null) == 2


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "precision_causal_attention_block_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"(import|from)\s+oracle|oracle/|flamia_oracle", src), f


def test_binding_constants_match_the_header():
    # every FLAMIA_FLAG_* / FLAMIA_FORMAT_* / FLAMIA_DEV_* macro of flamia.h has
    # the same value in the Python binding, and the binding declares a
    # signature for every exported function
    from precision_causal_attention_block_gb300 import flamia as fl
    src = open(os.path.join(ROOT, "include", "flamia.h")).read()
    macros = dict(re.findall(r"#define FLAMIA_((?:FLAG|FORMAT|DEV)_[A-Z0-9_]+)\s+(0x[0-9A-Fa-f]+|\d+)",
                             src))
    assert len(macros) >= 14
    for name, val in macros.items():
        assert getattr(fl, name, None) == int(val, 0), name
    for n in declared_symbols():
        assert n in fl.SIGNATURES, n
