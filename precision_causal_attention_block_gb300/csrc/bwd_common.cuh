// Pieces shared by the backward kernels (attn_bwd.cu: head dims 64 and the
// mixed NVFP4 path; attn_bwd128.cu: the pipelined head-dim-128 kernel).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "short_docs.cuh"

namespace flamia {

struct BwdParams {
  const uint8_t* q_scales;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  const uint8_t* do_scales;
  const uint32_t* q4_scales;  // NVFP4: 4 E4M3 scales per (token, head) as one word (d = 64)
  const uint32_t* k4_scales;
  const float* D;
  const float* lse;
  const int32_t* cu;
  int* wl_header;  // list sizes, and the claim counters this kernel updates
  const int4* items;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int T, H, ndocs, cap;
  int Hkv, G;        // K / V heads; K / V head hk serves query heads hk G .. hk G + G - 1
  float scale_log2;  // softmax_scale * log2(e)
  float sm_scale;
  int hadamard;  // dK (and, in the conversion, dQ) rotated back by H_d
  int causal;    // 0: every query sees every key of its document
  int* dq_turns;  // deterministic dQ: [T][H] turn counters (per tile's first query), else null
  const int8_t* dq_pre;  // FP16 dQ accumulator: prescale exponents [H, T], else null (float32)
  int sched;             // kSchedDynamic / kSchedRule / kSchedStatic
  int ds_rows;           // dQ's dS operand with query-row exponents
  int token;             // per-token operand scales (implies ds_rows)
  unsigned long long* ds_count;  // dS rounded-to-zero diagnostic: [nonzero, zero], else null
  int* status;
};

// dS rounded-to-zero diagnostic of one 32-column chunk: among the chunk's dS
// values (float, dv) the nonzero ones, and of those the ones whose E4M3 code
// in the block payload (dw, four per word) is +-0; summed over the warp and
// added to a shared-memory pair by lane 0.
__device__ __forceinline__ void count_ds_zero(const uint32_t (&dv)[32], const uint32_t (&dw)[8],
                                              unsigned long long* cnt, int lane) {
  uint32_t nz = 0, z = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const bool live = __uint_as_float(dv[i]) != 0.f;
    const bool zero = ((dw[i >> 2] >> (8 * (i & 3))) & 0x7Fu) == 0u;
    nz += live ? 1u : 0u;
    z += (live && zero) ? 1u : 0u;
  }
  nz = __reduce_add_sync(0xffffffffu, nz);
  z = __reduce_add_sync(0xffffffffu, z);
  if (lane == 0) {
    atomicAdd(cnt, static_cast<unsigned long long>(nz));
    atomicAdd(cnt + 1, static_cast<unsigned long long>(z));
  }
}

__device__ __forceinline__ float pow2_or_zero(int k) { return k < -126 ? 0.f : exp2i(k); }

// One 32-column chunk of a key row: P (operand codes), dS (float, 2^8-scaled)
// and the chunk's |dS| maximum.  MASK: diagonal tile, query < key is masked.
template <bool MASK>
__device__ __forceinline__ float bwd_chunk(const uint32_t (&sv)[32], uint32_t (&dv)[32],
                                           const float* nl, const float* dd, float fS, float fP,
                                           int col0, int key, uint32_t (&pw)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const float4 n4 = *reinterpret_cast<const float4*>(nl + i);
    const float4 d4 = *reinterpret_cast<const float4*>(dd + i);
    float2 s01 = __ffma2_rn(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])),
                            make_float2(fS, fS), make_float2(n4.x, n4.y));
    float2 s23 = __ffma2_rn(make_float2(__uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3])),
                            make_float2(fS, fS), make_float2(n4.z, n4.w));
    if (MASK) {
      if (col0 + i + 0 < key) s01.x = -INFINITY;
      if (col0 + i + 1 < key) s01.y = -INFINITY;
      if (col0 + i + 2 < key) s23.x = -INFINITY;
      if (col0 + i + 3 < key) s23.y = -INFINITY;
    }
    const float2 p01 = make_float2(ex2_approx(s01.x), ex2_approx(s01.y));
    const float2 p23 = make_float2(ex2_approx(s23.x), ex2_approx(s23.y));
    const float2 g01 = __ffma2_rn(make_float2(__uint_as_float(dv[i]), __uint_as_float(dv[i + 1])),
                                  make_float2(fP, fP), make_float2(-d4.x, -d4.y));
    const float2 g23 =
        __ffma2_rn(make_float2(__uint_as_float(dv[i + 2]), __uint_as_float(dv[i + 3])),
                   make_float2(fP, fP), make_float2(-d4.z, -d4.w));
    const float2 d01 = __fmul2_rn(p01, g01);
    const float2 d23 = __fmul2_rn(p23, g23);
    amax = fmax3(fabsf(d01.x), fabsf(d01.y), amax);
    amax = fmax3(fabsf(d23.x), fabsf(d23.y), amax);
    dv[i] = __float_as_uint(d01.x);
    dv[i + 1] = __float_as_uint(d01.y);
    dv[i + 2] = __float_as_uint(d23.x);
    dv[i + 3] = __float_as_uint(d23.y);
    pw[i / 4] = cvt_e4m3x4(p01.x, p01.y, p23.x, p23.y);
  }
  return amax;
}

// Per-token operand scales: one 32-column chunk of a key row with per-column
// (query) factors.  s = S 2^eQ(i) rowf + nl, dP 2^eD(i) rowg - D; dv gets
// dS (2^8-scaled, unfolded) and pw the dV operand RNE_E4M3(P8 2^(eD(i) -
// EdO)).  qf, df, pf: the chunk's 2^eQ(i), 2^eD(i), 2^(eD(i) - EdO).
template <bool MASK>
__device__ __forceinline__ void bwd_chunk_tok(const uint32_t (&sv)[32], uint32_t (&dv)[32],
                                              const float* nl, const float* dd, const float* qf,
                                              const float* df, const float* pf, float rowf,
                                              float rowg, int col0, int key, uint32_t (&pw)[8]) {
  const float2 rf2 = make_float2(rowf, rowf), rg2 = make_float2(rowg, rowg);
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const float4 n4 = *reinterpret_cast<const float4*>(nl + i);
    const float4 d4 = *reinterpret_cast<const float4*>(dd + i);
    const float4 q4 = *reinterpret_cast<const float4*>(qf + i);
    const float4 g4 = *reinterpret_cast<const float4*>(df + i);
    const float4 p4 = *reinterpret_cast<const float4*>(pf + i);
    float2 s01 = __fmul2_rn(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])),
                            make_float2(q4.x, q4.y));
    float2 s23 = __fmul2_rn(make_float2(__uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3])),
                            make_float2(q4.z, q4.w));
    s01 = __ffma2_rn(s01, rf2, make_float2(n4.x, n4.y));
    s23 = __ffma2_rn(s23, rf2, make_float2(n4.z, n4.w));
    if (MASK) {
      if (col0 + i + 0 < key) s01.x = -INFINITY;
      if (col0 + i + 1 < key) s01.y = -INFINITY;
      if (col0 + i + 2 < key) s23.x = -INFINITY;
      if (col0 + i + 3 < key) s23.y = -INFINITY;
    }
    const float2 p01 = make_float2(ex2_approx(s01.x), ex2_approx(s01.y));
    const float2 p23 = make_float2(ex2_approx(s23.x), ex2_approx(s23.y));
    float2 g01 = __fmul2_rn(make_float2(__uint_as_float(dv[i]), __uint_as_float(dv[i + 1])),
                            make_float2(g4.x, g4.y));
    float2 g23 = __fmul2_rn(make_float2(__uint_as_float(dv[i + 2]), __uint_as_float(dv[i + 3])),
                            make_float2(g4.z, g4.w));
    g01 = __ffma2_rn(g01, rg2, make_float2(-d4.x, -d4.y));
    g23 = __ffma2_rn(g23, rg2, make_float2(-d4.z, -d4.w));
    const float2 d01 = __fmul2_rn(p01, g01);
    const float2 d23 = __fmul2_rn(p23, g23);
    dv[i] = __float_as_uint(d01.x);
    dv[i + 1] = __float_as_uint(d01.y);
    dv[i + 2] = __float_as_uint(d23.x);
    dv[i + 3] = __float_as_uint(d23.y);
    const float2 b01 = __fmul2_rn(p01, make_float2(p4.x, p4.y));
    const float2 b23 = __fmul2_rn(p23, make_float2(p4.z, p4.w));
    pw[i / 4] = cvt_e4m3x4(b01.x, b01.y, b23.x, b23.y);
  }
}

// One backward work item (128-key tile of one document x one head), decoded
// identically by every role; false for items of short documents, which the
// CUDA-core kernel handles.
struct BwdItem {
  int hk, s, e, k0, k1, qs, nq;  // hk: K / V head; qs: the first query that sees the key
                                  // tile; nq: 128-query tiles per query head
};

__device__ __forceinline__ bool decode_bwd_item(const BwdParams& prm, int n_items, int idx,
                                                BwdItem& it) {
  const int T = prm.T;
  it.hk = idx / n_items;  // head-major: a wave of CTAs touches the Q / dO / dQ of few heads
  // each head's list longest first; in the deterministic dQ mode shortest
  // first, so a document's key tiles are claimed in descending order, the
  // order of their dQ turns (a turn never waits for an item claimed later)
  const int pos = idx % n_items;
  const int4 item = prm.items[prm.dq_turns != nullptr ? n_items - 1 - pos : pos];
  // clamped: a malformed work list or offsets cannot index outside [0, T)
  const int doc = min(max(item.x, 0), prm.ndocs - 1);
  it.s = min(max(prm.cu[doc], 0), T);
  it.e = min(max(prm.cu[doc + 1], it.s), T);
  if (it.e - it.s <= kShortDoc) return false;
  it.k0 = it.s + ((min(max(item.y, it.s), it.e) - it.s) & ~(kTile - 1));
  it.k1 = min(max(item.z, it.k0), min(it.k0 + kTile, it.e));
  // causal: query tiles from the diagonal to the end; else the whole document
  it.qs = prm.causal ? it.k0 : it.s;
  it.nq = (it.e - it.qs + kTile - 1) / kTile;
  return true;
}

// Deterministic dQ: the key tiles of a document add their partials to the
// query tile starting at q0 in descending key-tile order, the order in which
// their walks from the diagonal reach it; key tile r waits until the tiles
// above it have added (causal: the tiles up to the one holding q0; else all).
__device__ __forceinline__ int dq_turn(const BwdParams& prm, const BwdItem& it, int q0) {
  const int top = prm.causal ? (q0 - it.s) / kTile : (it.e - it.s - 1) / kTile;
  return top - (it.k0 - it.s) / kTile;
}

// Consumer roles of a backward kernel's item ring: the MMA issuer and one
// leader thread per compute group (the leader hands the item to its group
// through shared memory and a named barrier, so a group's warps never
// disagree on the item and never miss a barrier).

// The 2-CTA backward (head dim 128): whether the call's modes allow it, and
// its launch (grid: as many CTA pairs as can be resident).
bool bwd_pair_supported(const BwdParams& prm);
cudaError_t launch_bwd128_pair(const BwdParams& prm, const flamia_qtensor* q,
                               const flamia_qtensor* k, const flamia_qtensor* v,
                               const flamia_qtensor* dout, float* acc, cudaStream_t stream);

// Pipelined backward for head dim 128 (MXFP8 score product); grid = CTAs.
cudaError_t launch_bwd128_pipelined(const BwdParams& prm, const flamia_qtensor* q,
                                    const flamia_qtensor* k, const flamia_qtensor* v,
                                    const flamia_qtensor* dout, float* acc, unsigned grid,
                                    cudaStream_t stream);

}  // namespace flamia
