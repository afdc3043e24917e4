"""FP64 CPU oracle for token-block microscaled causal flash attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA path; the two meet only
in the seeded input generators (``workloads.py``), which hold no arithmetic of
the method.

What it follows (citations name the page and its section):

* "FLAMIA ... (jaehun.me review)", sec. 3.1 "Reduce quantization duplication
  with token-block scales": Q, K, V, dO are E4M3 codes with one power-of-two
  exponent per 32 consecutive tokens x the full head dimension; dS has one
  scale per 32x32 block; probability operands are E4M3; outputs and gradients
  are BF16.  Mixed path: Q, K for the score product are NVFP4 (one scale per
  16 head-dim elements of a token).
* same page, sec. 3.1: the score is the plain E4M3 dot product times a row
  factor (query block exponent, folded with the softmax scale) and a column
  factor (key block exponent).  The printed formula is missing from the page;
  the reading used here is S_ij = scale * 2^eQ(i) * 2^eK(j) * sum_k q_ik k_jk.
* same page, sec. 3.2: exponents are rounded up so that the scaled maximum
  never exceeds 448 (E4M3 max) -- nothing clips.
* same page, sec. 1.2 and 3.3: forward S, P, O, row statistics; backward
  recomputes P, dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = dS K,
  dK = dS^T Q, with D_i = dO_i . O_i from the same quantised dO.
* same page, sec. 3.4 "Packed documents": scale groups never cross a document
  boundary; rows outside a document get an infinite log-sum-exp.
* same page, sec. 3.4 "Work scheduling": a work item is 256 consecutive
  queries of one document, its cost the number of key blocks it visits,
  sorted by descending cost.
* same page, sec. 3.4 "Hadamard rotation" and "Quantization fusion": the
  head-dimension channels of Q and K are mixed by a normalised orthogonal
  transform inside the quantiser (dot products preserved, token positions
  not mixed), on by default at head dim 128.
* grouped-query attention (GQA), part of the attention API the method
  serves (the pages give no numerics for it): K and V carry H_kv heads,
  query head h reads K / V head h // (H / H_kv), and dK, dV of a K / V head
  sum the contributions of its H / H_kv query heads.
* same page, sec. 4.8 "Batched and non-causal paths": the non-causal packed
  call, where every query sees every key of its own document.
* same page, sec. 3.2 "accumulator leakage" and sec. 3.5.3 "Backward
  pass": dQ partial sums reduced in FP16 behind a power-of-two prescale set
  from sequence-wide maxima, or ("causal dQ scaling") from the keys visible
  to each query row.
* same page, sec. 2 "A small example": the floor exponent rule
  e = floor(log2 amax) - emax with clipping at 448, used here only as the
  negative control of the leakage probe.

Readings where the pages are silent:
* code rounding is round-to-nearest-even; -0 keeps its sign bit;
* amax == 0 gives exponent -127 (byte 0) and all-zero codes; exponents are
  clamped to [-127, 127];
* the running row maximum is an integer ceil of the log2-domain score, and the
  probability operand is RNE_E4M3(2^8 * exp2(s - m)); l sums the unquantised
  exp2(s - m); O = 2^-8 * sum_j P^_ij V^_j / l; LSE = (m + log2 l) * ln 2;
* the backward probability is exp2(s - lse2) (normalised); the dV operand is
  RNE_E4M3(2^8 P); dS uses the unquantised P;
* the dS block exponent uses the same round-up rule on the 32x32 block
  maximum (masked entries are 0); the softmax scale is applied after the
  dQ / dK products;
* query-row dS exponents (an option): for the dQ product only, one round-up
  exponent per query row and 32-key block; dK keeps the 32x32 block ones
  (only dQ of an earlier row can see a later row through a shared exponent);
* the NVFP4 scale is the smallest E4M3 value >= amax / 6, no tensor-wide
  scale;
* the rotation is the unnormalised Sylvester-Hadamard matrix H_d (entries
  +-1, H_d H_d = d I), applied to each (token, head) row of Q and K in float32
  by butterflies of stride 1, 2, ..., d/2 in that order (the GPU quantiser
  takes the same steps, so the codes match bit for bit); the 1/d that
  normalises it is folded into the softmax scale (exact for d a power of
  two), and the backward returns dQ = dQ_r H_d, dK = dK_r H_d for the
  gradients dQ_r, dK_r of the rotated operands;
* the FP16 dQ accumulator (an option; float32 is the default): prescale
  2^p with p = 15 - ceil(log2(16 d 448^3)) - (e_dO + max e_V + max e_K), the
  maxima sequence-wide or over the keys the row sees, key-tile partials
  rounded to float32 then FP16 and added in FP16 (see dq_prescale);
* work items: forward q0 = s + 256k, q1 = min(q0 + 256, e), cost =
  ceil((q1 - s) / 128); backward k0 = s + 128k, k1 = min(k0 + 128, e),
  cost = ceil((e - k0) / 128); stable sort by descending cost.

Parity pins for every function live in tests/test_oracle_*.py.
"""
from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)
LN2 = math.log(2.0)
E4M3_MAX = 448.0
E2M1_MAX = 6.0
P_SCALE_LOG2 = 8  # 2^8: largest power of two <= 448, multiplies P before E4M3


# ----------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------

def _e4m3_value(code: int) -> float:
    """OCP FP8 E4M3FN: sign, 4-bit exponent (bias 7), 3-bit mantissa; 0x7F/0xFF NaN."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(y, saturate: bool = False) -> np.ndarray:
    """Round-to-nearest-even of float64 values to E4M3 codes (uint8).

    Values above 448 in magnitude are an error unless ``saturate`` (then they
    clip to +-448, the behaviour of the floor-rule negative control).
    """
    y = np.asarray(y, dtype=np.float64)
    sign = np.signbit(y)
    a = np.abs(y)
    if np.any(~np.isfinite(a)):
        raise ValueError("non-finite value to E4M3")
    if saturate:
        a = np.minimum(a, E4M3_MAX)
    elif np.any(a > E4M3_MAX):
        raise ValueError("value above 448 would clip")
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # subnormal range: multiples of 2^-9
    q = np.rint(a[sub] * 2.0 ** 9)          # 0..8, rint = ties to even
    code[sub] = q.astype(np.int64)          # q == 8 is the smallest normal (exp 1, man 0)
    nrm = ~sub
    an = a[nrm]
    _, ex = np.frexp(an)                    # an = f * 2^ex, f in [0.5, 1)
    E = ex - 1                              # an in [2^E, 2^(E+1))
    t = np.rint((an / np.ldexp(1.0, E) - 1.0) * 8.0)   # mantissa in eighths, ties to even
    carry = t >= 8
    E = np.where(carry, E + 1, E)
    t = np.where(carry, 0, t)
    code[nrm] = ((E + 7) << 3) | t.astype(np.int64)
    if saturate:
        code = np.minimum(code, 0x7E)
    return (code | (sign.astype(np.int64) << 7)).astype(np.uint8)


E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_TABLE = np.concatenate([E2M1_VALUES, -E2M1_VALUES])


def e2m1_decode(codes) -> np.ndarray:
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def e2m1_encode(y) -> np.ndarray:
    """Round-to-nearest-even to E2M1 (sign, 2-bit exponent bias 1, 1-bit mantissa).

    Saturates at +-6 (the NVFP4 scale keeps |y| <= 6, so it never triggers
    except when the scale itself saturated at 448)."""
    y = np.asarray(y, dtype=np.float64)
    sign = np.signbit(y)
    a = np.minimum(np.abs(y), E2M1_MAX)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 1.0
    code[sub] = np.rint(a[sub] * 2.0).astype(np.int64)      # 0, 0.5, (1.0 -> code 2)
    nrm = ~sub
    an = a[nrm]
    _, ex = np.frexp(an)
    E = ex - 1                                              # 0, 1, 2
    t = np.rint((an / np.ldexp(1.0, E) - 1.0) * 2.0)        # halves, ties to even
    carry = t >= 2
    E = np.where(carry, E + 1, E)
    t = np.where(carry, 0, t)
    code[nrm] = ((E + 1) << 1) | t.astype(np.int64)
    return (code | (sign.astype(np.int64) << 3)).astype(np.uint8)


def e8m0_decode(byte) -> np.ndarray:
    b = np.asarray(byte, dtype=np.int64)
    return np.ldexp(1.0, b - 127)


def bf16_round(x) -> np.ndarray:
    """float64 -> nearest BF16 value (8 significant bits, ties to even), as float64."""
    x = np.asarray(x, dtype=np.float64)
    f, e = np.frexp(x)
    return np.ldexp(np.rint(f * 256.0) / 256.0, e)


def hadamard_fp32(x) -> np.ndarray:
    """x H_d along the last axis (H_d the unnormalised Sylvester-Hadamard
    matrix, d a power of two), computed in float32 by butterflies of stride
    1, 2, ..., d/2 in that order: within each pair (i, i + s) with
    i mod 2s < s the new values are (x_i + x_{i+s}, x_i - x_{i+s}).
    Returns float64 (exact copies of the float32 results)."""
    y = np.asarray(x, dtype=np.float32)
    d = y.shape[-1]
    assert d > 0 and d & (d - 1) == 0, d
    lead = y.shape[:-1]
    s = 1
    while s < d:
        z = y.reshape(lead + (d // (2 * s), 2, s))
        a, b = z[..., 0, :], z[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(lead + (d,))
        s *= 2
    return y.astype(np.float64)


def sylvester(d: int) -> np.ndarray:
    """H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]] (float64)."""
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


# ----------------------------------------------------------------------------
# Exponent rules
# ----------------------------------------------------------------------------

def roundup_exponent(amax) -> np.ndarray:
    """Smallest integer e with amax <= 448 * 2^e, clamped to [-127, 127];
    amax == 0 gives -127."""
    amax = np.asarray(amax, dtype=np.float64)
    e = np.full(amax.shape, -127, dtype=np.int64)
    pos = amax > 0
    _, ex = np.frexp(amax[pos])         # amax < 2^ex
    cand = ex - 10                      # 448 * 2^(ex-10) < 2^(ex-1) <= amax: too small
    for _ in range(4):                  # step up until the bound holds (at most 3 steps)
        bad = amax[pos] > E4M3_MAX * np.ldexp(1.0, cand)
        cand = np.where(bad, cand + 1, cand)
    e[pos] = cand
    return np.clip(e, -127, 127)


def floor_exponent(amax) -> np.ndarray:
    """OCP microscaling rule e = floor(log2 amax) - 8 (8 = E4M3 emax); negative control."""
    amax = np.asarray(amax, dtype=np.float64)
    e = np.full(amax.shape, -127, dtype=np.int64)
    pos = amax > 0
    _, ex = np.frexp(amax[pos])
    e[pos] = (ex - 1) - 8
    return np.clip(e, -127, 127)


# ----------------------------------------------------------------------------
# Token-block quantiser
# ----------------------------------------------------------------------------

def doc_blocks(cu_seqlens, size: int = 32):
    """Document-local blocks [s + size*b, min(s + size*(b+1), e)) in token order."""
    out = []
    cu = list(cu_seqlens)
    for i in range(len(cu) - 1):
        s, e = int(cu[i]), int(cu[i + 1])
        for b0 in range(s, e, size):
            out.append((b0, min(b0 + size, e)))
    return out


def quantize_tokenblock(x, cu_seqlens, rule: str = "up", group: str = "block"):
    """E4M3 codes [T, H, d] and E8M0 scale bytes [H, T] (one byte per token).

    group="block": one exponent per (document-local 32-token block, head).
    group="token": one exponent per (token, head) over its d elements (the
    per-token operand scales of the precision options).
    group="tensor": one exponent per head over all tokens (negative control).
    rule="up": round-up exponent (never clips); rule="floor": floor rule with
    clipping at 448 (negative control).
    """
    x = np.asarray(x, dtype=np.float64)
    T, H, d = x.shape
    codes = np.zeros((T, H, d), dtype=np.uint8)
    sbytes = np.zeros((H, T), dtype=np.uint8)
    if group == "block":
        blocks = doc_blocks(cu_seqlens, 32)
    elif group == "token":
        blocks = doc_blocks(cu_seqlens, 1)
    elif group == "tensor":
        blocks = [(0, T)] if T > 0 else []
    else:
        raise ValueError(group)
    expfn = roundup_exponent if rule == "up" else floor_exponent
    for (b0, b1) in blocks:
        xb = x[b0:b1]                                   # [n, H, d]
        amax = np.abs(xb).max(axis=(0, 2))              # per head
        e = expfn(amax)                                 # [H]
        scaled = xb * np.ldexp(1.0, -e)[None, :, None]
        codes[b0:b1] = e4m3_encode(scaled, saturate=(rule != "up"))
        sbytes[:, b0:b1] = (e + 127).astype(np.uint8)[:, None]
    return codes, sbytes


def dequantize_tokenblock(codes, sbytes) -> np.ndarray:
    """code value * 2^(byte - 127); the scale depends only on the token."""
    return e4m3_decode(codes) * e8m0_decode(sbytes).T[:, :, None]


def compute_D(do_codes, do_sbytes, o_bf16) -> np.ndarray:
    """D[h, t] = sum_k dequant(dO)[t, h, k] * O[t, h, k] (O = the forward's BF16 output)."""
    return np.einsum("thk,thk->ht", dequantize_tokenblock(do_codes, do_sbytes),
                     np.asarray(o_bf16, dtype=np.float64))


# ----------------------------------------------------------------------------
# NVFP4 quantiser (mixed path: Q, K for the score product)
# ----------------------------------------------------------------------------

def nvfp4_scale_code(amax) -> np.ndarray:
    """E4M3 code of the smallest E4M3 value >= amax / 6 (exact quotient);
    amax == 0 gives 0; quotients above 448 saturate to 448."""
    amax = np.asarray(amax, dtype=np.float64)
    pos_vals = E4M3_TABLE[:0x7F]                       # codes 0x00..0x7E, increasing
    q = amax / 6.0
    idx = np.searchsorted(pos_vals, q, side="left")   # first value >= q
    return np.minimum(idx, 0x7E).astype(np.uint8)


def quantize_nvfp4(x):
    """Packed E2M1 codes [T, H, d/2] (element 2i in the low nibble) and E4M3
    scale codes [T, H, d/16]."""
    x = np.asarray(x, dtype=np.float64)
    T, H, d = x.shape
    g = x.reshape(T, H, d // 16, 16)
    sc = nvfp4_scale_code(np.abs(g).max(axis=3))
    s = e4m3_decode(sc)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(s > 0, g / s, 0.0)
    c = e2m1_encode(y).reshape(T, H, d)
    packed = (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    return packed, sc


def dequantize_nvfp4(packed, sc) -> np.ndarray:
    T, H, d2 = packed.shape
    c = np.empty((T, H, 2 * d2), dtype=np.uint8)
    c[..., 0::2] = packed & 0xF
    c[..., 1::2] = packed >> 4
    v = e2m1_decode(c).reshape(T, H, 2 * d2 // 16, 16)
    return (v * e4m3_decode(sc)[..., None]).reshape(T, H, 2 * d2)


# ----------------------------------------------------------------------------
# Work list
# ----------------------------------------------------------------------------

def build_worklist(cu_seqlens):
    """Forward and backward items, int64 arrays [n, 4] = (doc, start, end, cost),
    each sorted by descending cost, stable over generation order."""
    cu = [int(c) for c in cu_seqlens]
    fwd, bwd = [], []
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        for q0 in range(s, e, 256):
            q1 = min(q0 + 256, e)
            fwd.append((b, q0, q1, -(-(q1 - s) // 128)))
        for k0 in range(s, e, 128):
            k1 = min(k0 + 128, e)
            bwd.append((b, k0, k1, -(-(e - k0) // 128)))
    fwd.sort(key=lambda it: -it[3])   # Python's sort is stable
    bwd.sort(key=lambda it: -it[3])
    return (np.array(fwd, dtype=np.int64).reshape(-1, 4),
            np.array(bwd, dtype=np.int64).reshape(-1, 4))


# ----------------------------------------------------------------------------
# Attention, one (document, head) at a time
# ----------------------------------------------------------------------------

class DocHead:
    """Operands of one document and one head, as exact values split into a
    code part and a per-token power-of-two exponent (for the unquantised mode
    the code part is the raw value and the exponent is 0)."""

    def __init__(self, q, eq, k, ek, v, ev, do=None, edo=None, qs=None, ks=None):
        self.q, self.eq = q, eq          # [L, d], [L] int
        self.k, self.ek = k, ek
        self.v, self.ev = v, ev
        self.do, self.edo = do, edo
        # score operands when they differ from q/k (NVFP4 mixed path): exact values
        self.qs, self.ks = qs, ks
        self.L = q.shape[0]
        self.causal = True  # False: every query sees every key of the document
        # per-token operand scales: the per-token factors along a contraction are
        # folded into the opposite operand before its E4M3 rounding
        self.token = False


def _scores(dh: DocHead, rows: np.ndarray, cols: np.ndarray, sm_scale: float) -> np.ndarray:
    """log2-domain scores s_ij = S_ij * log2(e), -inf where j > i (causal)."""
    if dh.qs is not None:
        S = sm_scale * (dh.qs[rows] @ dh.ks[cols].T)
    else:
        dots = dh.q[rows] @ dh.k[cols].T                       # code dot products
        S = sm_scale * dots * np.ldexp(1.0, dh.eq[rows])[:, None] \
            * np.ldexp(1.0, dh.ek[cols])[None, :]              # row factor x column factor
    s = S * LOG2E
    if dh.causal:
        s[cols[None, :] > rows[:, None]] = -np.inf
    return s


def fwd_rows(dh: DocHead, rows: np.ndarray, sm_scale: float, quant: bool = True):
    """Forward output rows: O [R, d], lse2 [R] (log2 units), m [R], l [R]."""
    rows = np.asarray(rows, dtype=np.int64)
    if not dh.causal:
        cols = np.arange(dh.L)
    else:
        cols = np.arange(int(rows.max()) + 1 if rows.size else 0)
    s = _scores(dh, rows, cols, sm_scale)
    m = np.ceil(s.max(axis=1))                                 # integer row maximum
    pt = np.exp2(s - m[:, None])                               # 0 where masked
    l = pt.sum(axis=1)                                         # unquantised sum
    if quant and dh.token:
        # V's per-key factor 2^eV(j) folded into P^ relative to the largest
        # exponent EV(i, b) among the keys of its 32-key block that row i sees
        EV = _visible_block_max(dh.ev, rows, cols, dh.causal)
        fold = np.ldexp(1.0, dh.ev[cols][None, :] - EV)
        ph = e4m3_decode(e4m3_encode(np.ldexp(pt * fold, P_SCALE_LOG2)))
        o = np.ldexp((ph * np.ldexp(1.0, EV)) @ dh.v[cols], -P_SCALE_LOG2) / l[:, None]
        return o, m + np.log2(l), m, l
    p8 = np.ldexp(pt, P_SCALE_LOG2)
    ph = e4m3_decode(e4m3_encode(p8)) if quant else p8         # E4M3 probability operand
    vhat = dh.v[cols] * np.ldexp(1.0, dh.ev[cols])[:, None]
    o = np.ldexp(ph @ vhat, -P_SCALE_LOG2) / l[:, None]
    return o, m + np.log2(l), m, l


def _visible_block_max(e, rows, cols, causal):
    """[R, C] int: for row i and column j, the largest e[j'] over the columns j'
    of j's document-aligned 32-column block that row i sees (j' <= i when
    causal); 0 where row i sees no column of the block.  rows / cols are
    doc-local, cols a contiguous range starting on a 32 boundary."""
    out = np.zeros((len(rows), len(cols)), dtype=np.int64)
    c0 = int(cols[0]) if len(cols) else 0
    for j0 in range(0, len(cols), 32):
        blk = e[cols[j0:j0 + 32]].astype(np.int64)
        if causal:
            pm = np.maximum.accumulate(blk)                    # prefix maxima
            last = np.asarray(rows) - (c0 + j0)                # last visible column in the block
            vis = last >= 0
            val = np.where(vis, pm[np.clip(last, 0, len(blk) - 1)], 0)
        else:
            val = np.full(len(rows), blk.max())
        out[:, j0:j0 + 32] = val[:, None]
    return out


def _query_block_max(e, rows):
    """[R] int: the largest e over each row's document-aligned 32-row block
    (rows doc-local, contiguous, starting on a 32 boundary, whole blocks
    except at the document end)."""
    out = np.empty(len(rows), dtype=np.int64)
    for i0 in range(0, len(rows), 32):
        out[i0:i0 + 32] = e[rows[i0:i0 + 32]].max()
    return out


def _block_quantize_dS(dS: np.ndarray, r0: int, c0: int, extra: int = 0) -> np.ndarray:
    """dS rounded through E4M3 with one round-up exponent per 32x32 block whose
    origin is aligned to the document start (r0, c0 are doc-local offsets of
    the rectangle and must be multiples of 32).  extra > 0 enlarges every
    block exponent by that much (the oversized scale of the pages' dS-scale
    ablation; never used by the method)."""
    assert r0 % 32 == 0 and c0 % 32 == 0
    out = np.empty_like(dS)
    R, C = dS.shape
    for i0 in range(0, R, 32):
        for j0 in range(0, C, 32):
            blk = dS[i0:i0 + 32, j0:j0 + 32]
            e = int(roundup_exponent(np.abs(blk).max())) + extra
            out[i0:i0 + 32, j0:j0 + 32] = e4m3_decode(e4m3_encode(blk * 2.0 ** -e)) * 2.0 ** e
    return out


def ds_zero_counts(qz: "Quantized", sm_scale: float, extra: int = 0, heads=None,
                   causal: bool = True):
    """Review page, sec. 3.3 and the dS-scale ablation of sec. 4: over every
    pair a query sees, the number of dS entries that are nonzero, and of those
    the number whose E4M3 code under the 32x32 block exponent is zero (rounded
    to zero).  extra: an oversized block exponent (see _block_quantize_dS).
    With per-token operand scales the block payload is dK's folded operand.
    Returns (nonzero, zero)."""
    T, H, _ = qz.qc.shape
    nz = zero = 0
    for b in range(len(qz.cu) - 1):
        s, e = qz.cu[b], qz.cu[b + 1]
        if e == s:
            continue
        for h in (range(H) if heads is None else heads):
            dh = qz.dochead(b, h)
            dh.causal = causal
            rows = np.arange(e - s)
            o, lse2, _, _ = fwd_rows(dh, rows, sm_scale, True)
            dohat = dh.do * np.ldexp(1.0, dh.edo)[:, None]
            D = (dohat * bf16_round(o)).sum(axis=1)
            _, _, _, dS = bwd_rect(dh, rows, rows, lse2, D, sm_scale, True)
            if dh.token:  # the block payload is dK's operand, dS 2^(eQ - EQ)
                dSh = _block_quantize_dS(
                    np.ldexp(dS, (dh.eq[rows] - _query_block_max(dh.eq, rows))[:, None]), 0, 0,
                    extra)
            else:
                dSh = _block_quantize_dS(dS, 0, 0, extra)
            live = dS != 0
            nz += int(live.sum())
            zero += int((live & (dSh == 0)).sum())
    return nz, zero


def _row_quantize_dS(dS: np.ndarray, c0: int) -> np.ndarray:
    """dS rounded through E4M3 with one round-up exponent per query row and
    32-column block aligned to the document start (c0: doc-local offset of the
    first column, a multiple of 32): review page, sec. 3.2, the query-row-wise
    dS exponents that remove the leakage inside blocks."""
    assert c0 % 32 == 0
    out = np.empty_like(dS)
    for j0 in range(0, dS.shape[1], 32):
        blk = dS[:, j0:j0 + 32]
        e = roundup_exponent(np.abs(blk).max(axis=1))[:, None]
        out[:, j0:j0 + 32] = e4m3_decode(e4m3_encode(blk * np.ldexp(1.0, -e))) * np.ldexp(1.0, e)
    return out


def bwd_rect(dh: DocHead, rows: np.ndarray, cols: np.ndarray, lse2_rows: np.ndarray,
             D_rows: np.ndarray, sm_scale: float, quant: bool = True, raw_dq: bool = False,
             ds_rows: bool = False):
    """Backward contributions of the rectangle rows x cols.

    rows and cols are contiguous doc-local ranges starting on a 32 boundary.
    Returns (dQ partial [R, d] over these cols, dK partial [C, d] and dV
    partial [C, d] over these rows, dS [R, C]); with raw_dq the dQ partial is
    the product dS^ K^ before the softmax scale.  ds_rows: the dQ product takes
    dS rounded with query-row exponents (dK keeps the 32x32 block ones)."""
    s = _scores(dh, rows, cols, sm_scale)
    P = np.exp2(s - lse2_rows[:, None])                        # normalised, 0 where masked
    if quant and dh.token:
        return _bwd_rect_token(dh, rows, cols, P, D_rows, sm_scale, raw_dq)
    pb = np.ldexp(P, P_SCALE_LOG2)
    pbh = e4m3_decode(e4m3_encode(pb)) if quant else pb        # dV operand
    dohat = dh.do[rows] * np.ldexp(1.0, dh.edo[rows])[:, None]
    vhat = dh.v[cols] * np.ldexp(1.0, dh.ev[cols])[:, None]
    dP = dohat @ vhat.T
    dS = P * (dP - D_rows[:, None])
    dSh = _block_quantize_dS(dS, int(rows[0]), int(cols[0])) if quant else dS
    qhat = dh.q[rows] * np.ldexp(1.0, dh.eq[rows])[:, None]
    khat = dh.k[cols] * np.ldexp(1.0, dh.ek[cols])[:, None]
    dV = np.ldexp(pbh.T @ dohat, -P_SCALE_LOG2)
    dK = sm_scale * (dSh.T @ qhat)
    dSq = _row_quantize_dS(dS, int(cols[0])) if (quant and ds_rows) else dSh
    dQ = (dSq @ khat) if raw_dq else sm_scale * (dSq @ khat)
    return dQ, dK, dV, dS


def _bwd_rect_token(dh: DocHead, rows, cols, P, D_rows, sm_scale, raw_dq):
    """bwd_rect with per-token operand scales: each per-token factor along a
    contraction is folded into the opposite operand before that operand's
    E4M3 rounding (review page, sec. 3.2: scales folded into the opposite
    operand; per-token operand scales with query-row dS exponents close the
    leakage inside blocks).
      dV = 2^-8 sum_i P^b_ij 2^EdO(qb) dO_i,  P^b = RNE(2^8 P 2^(e_dO(i) - EdO(qb)));
      dK = scale sum_i dS^K_ij 2^EQ(qb) Q_i,  dS^K = dS 2^(eQ(i) - EQ(qb)) rounded
           with one exponent per 32x32 block;
      dQ = scale sum_j dS^Q_ij K_j (codes),   dS^Q = dS 2^eK(j) rounded with one
           exponent per (query row, 32-key block);
    EdO, EQ: the largest exponent of the query's 32-row block (dV and dK sum
    every later query by definition, so a block-wide choice cannot leak)."""
    edo_b = _query_block_max(dh.edo, rows)
    eq_b = _query_block_max(dh.eq, rows)
    pbh = e4m3_decode(e4m3_encode(np.ldexp(P, P_SCALE_LOG2 + (dh.edo[rows] - edo_b)[:, None])))
    dohat = dh.do[rows] * np.ldexp(1.0, dh.edo[rows])[:, None]
    vhat = dh.v[cols] * np.ldexp(1.0, dh.ev[cols])[:, None]
    dP = dohat @ vhat.T
    dS = P * (dP - D_rows[:, None])
    dSk = _block_quantize_dS(np.ldexp(dS, (dh.eq[rows] - eq_b)[:, None]), int(rows[0]),
                             int(cols[0]))
    dSq = _row_quantize_dS(np.ldexp(dS, dh.ek[cols][None, :]), int(cols[0]))
    dV = np.ldexp((pbh * np.ldexp(1.0, edo_b)[:, None]).T @ dh.do[rows], -P_SCALE_LOG2)
    dK = sm_scale * ((dSk * np.ldexp(1.0, eq_b)[:, None]).T @ dh.q[rows])
    dQ = dSq @ dh.k[cols]
    return (dQ if raw_dq else sm_scale * dQ), dK, dV, dS


# ----------------------------------------------------------------------------
# FP16 dQ accumulation (precision option)
# ----------------------------------------------------------------------------
# Review page, sec. 3.2 "accumulator leakage" and sec. 3.5.3 "Backward pass":
# the dQ partial sums of the key tiles are reduced in FP16 (half the traffic of
# float32), pre-multiplied by a power of two that keeps them inside FP16's
# range; by default the power comes from sequence-wide maxima of dO, V and K,
# so a later token changes the rounding of earlier rows; "causal dQ scaling"
# takes it from the keys each query row sees.
# Reading: the magnitudes are the operands' block exponents (every element of
# a block satisfies |x| <= 448 * 2^e), which bound the raw partial sums
# rigorously and make the prescale an integer function of the scale tables:
#   |sum_j dS^_ij K^_jk| <= 16 d 448^3 2^E,  E = e_dO(i) + max e_V + max e_K
# (|dP_ij|, |D_i| <= d 448^2 2^(e_dO + max e_V) (1 + 2^-4 for O), P sums to 1,
# RNE_E4M3 of dS adds at most 2^-4 relative plus half a subnormal step per
# element, which the factor 16 covers up to 2^20 keys), and
#   p(i) = 15 - ceil(log2(16 d 448^3)) - E   keeps |2^p acc| <= 2^15 < 65504.
# The maxima run over the head's whole packed sequence ("sequence") or over
# the keys the row sees ("causal": keys s .. i of its document, all of the
# document in a non-causal call); p is clamped to [-126, 126].  The 128-key
# tiles (from the document start) add their partials, rounded to float32 then
# to FP16, to the FP16 accumulator in descending tile order (the deterministic
# order; any other order is equally valid); dQ = softmax_scale 2^-p acc.

DQ16_KEY_TILE = 128


def dq16_bound_log2(d: int) -> int:
    """ceil(log2(16 d 448^3)): the raw dQ bound is 2^(this + E)."""
    return int(math.ceil(math.log2(16 * d * E4M3_MAX ** 3)))


def dq_prescale(qz: "Quantized", h: int, mode: str, causal: bool = True) -> np.ndarray:
    """Prescale exponents p [T] (int64) of query head h; mode "sequence" or
    "causal" (see above)."""
    T, H, d = qz.qc.shape
    hk = h // (H // qz.kc.shape[1])
    edo = qz.dos[h].astype(np.int64) - 127
    ev = qz.vs[hk].astype(np.int64) - 127
    ek = qz.ks[hk].astype(np.int64) - 127
    if mode == "sequence":
        E = np.full(T, edo.max() + ev.max() + ek.max() if T else 0, dtype=np.int64)
    elif mode == "causal":
        E = np.zeros(T, dtype=np.int64)
        for b in range(len(qz.cu) - 1):
            s, e = qz.cu[b], qz.cu[b + 1]
            if e == s:
                continue
            if causal:
                mv, mk = np.maximum.accumulate(ev[s:e]), np.maximum.accumulate(ek[s:e])
            else:
                mv, mk = ev[s:e].max(), ek[s:e].max()
            E[s:e] = edo[s:e] + mv + mk
    else:
        raise ValueError(mode)
    return np.clip(15 - dq16_bound_log2(d) - E, -126, 126)


def fp16_round(x) -> np.ndarray:
    """Round to the nearest FP16 value (ties to even), returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def dq_fp16_rows(dh: DocHead, rows: np.ndarray, lse2_rows: np.ndarray, D_rows: np.ndarray,
                 sm_scale: float, p_rows: np.ndarray, return_acc: bool = False,
                 ds_rows: bool = False):
    """dQ of the given rows (doc-local, from 0, a multiple-of-32 start)
    through the prescaled FP16 accumulator."""
    f = np.ldexp(1.0, np.asarray(p_rows, dtype=np.int64))[:, None]
    acc = np.zeros((len(rows), dh.q.shape[1]))
    for t0 in reversed(range(0, dh.L, DQ16_KEY_TILE)):
        cols = np.arange(t0, min(t0 + DQ16_KEY_TILE, dh.L))
        part, _, _, _ = bwd_rect(dh, rows, cols, lse2_rows, D_rows, sm_scale, True, raw_dq=True,
                                 ds_rows=ds_rows)
        x = fp16_round((part * f).astype(np.float32))
        acc = fp16_round(acc + x)                    # the sum of two FP16 values is exact here
    dq = sm_scale * acc / f
    return (dq, acc) if return_acc else dq


# ----------------------------------------------------------------------------
# Whole-tensor entry points
# ----------------------------------------------------------------------------

class Quantized:
    """Token-block quantised operands of one attention call (+ optional NVFP4 Q, K)."""

    def __init__(self, q, k, v, do, cu_seqlens, qk_format: str = "mxfp8",
                 rule: str = "up", group: str = "block"):
        self.cu = [int(c) for c in cu_seqlens]
        self.group = group
        self.qc, self.qs = quantize_tokenblock(q, self.cu, rule, group)
        self.kc, self.ks = quantize_tokenblock(k, self.cu, rule, group)
        self.vc, self.vs = quantize_tokenblock(v, self.cu, rule, group)
        self.doc, self.dos = (quantize_tokenblock(do, self.cu, rule, group)
                              if do is not None else (None, None))
        self.qk_format = qk_format
        if qk_format == "nvfp4":
            self.q4 = dequantize_nvfp4(*quantize_nvfp4(q))
            self.k4 = dequantize_nvfp4(*quantize_nvfp4(k))

    def dochead(self, b: int, h: int) -> DocHead:
        """Query head h with its K / V head h // (H / H_kv)."""
        s, e = self.cu[b], self.cu[b + 1]
        hk = h // (self.qc.shape[1] // self.kc.shape[1])
        ex = lambda sb, hh: sb[hh, s:e].astype(np.int64) - 127
        dh = DocHead(e4m3_decode(self.qc[s:e, h]), ex(self.qs, h),
                     e4m3_decode(self.kc[s:e, hk]), ex(self.ks, hk),
                     e4m3_decode(self.vc[s:e, hk]), ex(self.vs, hk),
                     e4m3_decode(self.doc[s:e, h]) if self.doc is not None else None,
                     ex(self.dos, h) if self.doc is not None else None)
        if self.qk_format == "nvfp4":
            dh.qs, dh.ks = self.q4[s:e, h], self.k4[s:e, hk]
        dh.token = self.group == "token"
        return dh


def exact_dochead(q, k, v, do, cu, b, h) -> DocHead:
    s, e = cu[b], cu[b + 1]
    hk = h // (q.shape[1] // k.shape[1])
    z = np.zeros(e - s, dtype=np.int64)
    f = lambda x, hh: np.asarray(x[s:e, hh], dtype=np.float64)
    return DocHead(f(q, h), z, f(k, hk), z, f(v, hk), z, f(do, h) if do is not None else None, z)


def attention(q, k, v, do, cu_seqlens, sm_scale: float, quant: bool = True,
              qk_format: str = "mxfp8", rule: str = "up", group: str = "block",
              heads=None, docs=None, backward: bool = True, hadamard: bool = False,
              causal: bool = True, dq_accum: str = "fp32", ds_rows: bool = False):
    """Full forward (+ backward) over packed [T, H, d] float64 inputs.

    Returns a dict with O [T, H, d] (float64), O_bf16, lse [H, T] (natural log,
    +inf where not computed) and, with backward, dQ, dK, dV [T, H, d] and D
    [H, T].  ``heads`` / ``docs`` restrict the work (other entries stay 0).
    ``hadamard``: Q and K are rotated by H_d before quantisation (float32
    butterflies; exactly, in float64, when quant is False), the scores use
    sm_scale / d, and dQ, dK are rotated back by H_d.  ``causal=False``: every
    query sees every key of its document.  k and v may have H_kv heads (H_kv
    dividing H): query head h then reads head h // (H / H_kv), and dK, dV
    ([T, H_kv, d]) sum over the query heads of each K / V head.
    ``dq_accum``: "fp32" (float32 sums, no prescale), "fp16_sequence" or
    "fp16_causal" (the prescaled FP16 accumulator of dq_fp16_rows, with the
    prescale table returned as ``dq_prescale`` [H, T]).  ``ds_rows``: dQ from
    dS rounded with query-row exponents (see _row_quantize_dS).
    ``group="token"``: per-token operand scales (one exponent per token and
    head; the factors along each contraction folded into the opposite operand,
    see fwd_rows and _bwd_rect_token; dQ always takes query-row exponents)."""
    q = np.asarray(q, dtype=np.float64)
    T, H, d = q.shape
    Hkv = np.asarray(k).shape[1]
    assert H % Hkv == 0 and np.asarray(v).shape[1] == Hkv
    if hadamard:
        rot = hadamard_fp32 if quant else (lambda x: np.asarray(x, dtype=np.float64) @ sylvester(d))
        r = attention(rot(q), rot(k), v, do, cu_seqlens, sm_scale / d, quant, qk_format, rule,
                      group, heads, docs, backward, hadamard=False, causal=causal,
                      dq_accum=dq_accum, ds_rows=ds_rows)
        if backward:
            hd = sylvester(d)
            r["dQ"] = r["dQ"] @ hd
            r["dK"] = r["dK"] @ hd
        return r
    cu = [int(c) for c in cu_seqlens]
    heads = range(H) if heads is None else heads
    docs = range(len(cu) - 1) if docs is None else docs
    qz = Quantized(q, k, v, do if backward else None, cu, qk_format, rule, group) if quant else None
    out = {n: np.zeros((T, H, d)) for n in ("O", "O_bf16", "dQ")}
    out.update({n: np.zeros((T, Hkv, d)) for n in ("dK", "dV")})
    out["lse"] = np.full((H, T), np.inf)
    out["D"] = np.zeros((H, T))
    assert dq_accum in ("fp32", "fp16_sequence", "fp16_causal")
    dq16 = backward and dq_accum != "fp32"
    if dq16:
        assert quant, "the FP16 accumulator belongs to the quantised method"
        out["dq_prescale"] = np.zeros((H, T), dtype=np.int64)
        for h in heads:
            out["dq_prescale"][h] = dq_prescale(qz, h, dq_accum[5:], causal)
    for b in docs:
        s, e = cu[b], cu[b + 1]
        if e == s:
            continue
        for h in heads:
            dh = qz.dochead(b, h) if quant else exact_dochead(q, k, v, do, cu, b, h)
            dh.causal = causal
            rows = np.arange(e - s)
            o, lse2, _, _ = fwd_rows(dh, rows, sm_scale, quant)
            out["O"][s:e, h] = o
            out["O_bf16"][s:e, h] = bf16_round(o)
            out["lse"][h, s:e] = lse2 * LN2
            if not backward:
                continue
            dohat = dh.do * np.ldexp(1.0, dh.edo)[:, None]
            # D uses the forward's BF16 output in the quantised method and the
            # exact output in the unquantised reference
            o_for_D = out["O_bf16"][s:e, h] if quant else o
            D = (dohat * o_for_D).sum(axis=1)
            out["D"][h, s:e] = D
            dQ, dK, dV, _ = bwd_rect(dh, rows, rows, lse2, D, sm_scale, quant, ds_rows=ds_rows)
            if dq16:
                dQ = dq_fp16_rows(dh, rows, lse2, D, sm_scale, out["dq_prescale"][h, s:e],
                                  ds_rows=ds_rows)
            hk = h // (H // Hkv)
            out["dQ"][s:e, h] = dQ
            out["dK"][s:e, hk] += dK
            out["dV"][s:e, hk] += dV
    if quant:
        out["quantized"] = qz
    return out


def sampled_rows(qz: Quantized, b: int, h: int, sm_scale: float, qblocks, kblocks,
                 causal: bool = True):
    """Outputs of selected 32-token query blocks (O, lse, dQ) and 32-token key
    blocks (dK, dV) of document b, head h, each computed from its own
    definition (every key a query row sees, every query row a key sees).

    qblocks / kblocks are doc-local block indices.  Returns dicts keyed by the
    doc-local block index."""
    dh = qz.dochead(b, h)
    dh.causal = causal
    L = dh.L
    res = {"O": {}, "lse": {}, "dQ": {}, "dK": {}, "dV": {}}

    def stats(rows):
        o, lse2, _, _ = fwd_rows(dh, rows, sm_scale, True)
        dohat = dh.do[rows] * np.ldexp(1.0, dh.edo[rows])[:, None]
        D = (dohat * bf16_round(o)).sum(axis=1)
        return o, lse2, D

    for qb in qblocks:
        rows = np.arange(32 * qb, min(32 * qb + 32, L))
        o, lse2, D = stats(rows)
        cols = np.arange(0, int(rows[-1]) + 1 if causal else L)
        dQ, _, _, _ = bwd_rect(dh, rows, cols, lse2, D, sm_scale, True)
        res["O"][qb], res["lse"][qb], res["dQ"][qb] = o, lse2 * LN2, dQ
    for kb in kblocks:
        cols = np.arange(32 * kb, min(32 * kb + 32, L))
        rows = np.arange(32 * kb if causal else 0, L)
        _, lse2, D = stats(rows)
        _, dK, dV, _ = bwd_rect(dh, rows, cols, lse2, D, sm_scale, True)
        res["dK"][kb], res["dV"][kb] = dK, dV
    return res


def cosine(a, b) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))
