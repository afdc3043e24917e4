// Documents of at most 32 tokens (FLAMIA review page, sec. 3.4 "Packed
// documents"): one 32-token scale block covers the whole document, so every
// operand of the document has a single power-of-two scale per head and the
// work is a handful of tiny dot products -- not a dense contraction.  One
// warp handles one (document, head) on the CUDA cores with the same numerics
// as the tile kernels: E4M3 codes decoded exactly, float32 sums, the integer
// running maximum, P^ = RNE_E4M3(2^8 exp2(s - m)), dS rounded with one
// round-up exponent for the document's single 32x32 block.
// Lanes split the head dimension (d / 32 consecutive elements per lane).
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "short_docs.cuh"

namespace flamia {
namespace {

constexpr int kShortWarps = 4;  // warps (documents x heads) per CTA

__device__ __forceinline__ float pow2_or_zero_s(int k) { return k < -126 ? 0.f : exp2i(k); }

struct ShortParams {
  const uint8_t *qc, *kc, *vc, *doc_;           // E4M3 codes [T, H, d]
  const uint8_t *qs, *ks, *vs, *dos;            // E8M0 bytes [H, T]
  const uint8_t *q4c, *k4c;                     // NVFP4 codes [T, H, d/2] (mixed path, d = 64)
  const uint8_t *q4s, *k4s;                     // NVFP4 E4M3 scales [T, H, d/16]
  const int32_t* cu;
  int T, H, ndocs;
  int Hkv, G;  // K / V heads; query head h reads K / V head h / G
  float scale_log2, sm_scale;
  // forward
  __nv_bfloat16* o;
  float* lse;
  // backward
  const float *lse_in, *D;
  float* dq_acc;  // float32 [T, H, d]: dS K sums (softmax_scale comes in the conversion)
  const int8_t* dq_pre;  // FP16 accumulator: prescale exponents [H, T] (else null: float32)
  __nv_bfloat16 *dk, *dv;
  int hadamard;  // dK rotated back by H_d (Q and K were quantised rotated)
  int causal;    // 0: every query sees every key of its document
  int skip_single;  // one-token documents were done by the one-thread kernels
  int ds_rows;      // dQ from dS rounded with one exponent per query row
  int ppw;          // (document, head) pairs per warp: 32 when documents average <= 2
                    // tokens (almost every pair is skipped), else 1
  int token;        // per-token operand scales: one exponent per token, the factors
                    // along each contraction folded into the opposite operand
  unsigned long long* ds_count;  // dS rounded-to-zero diagnostic [nonzero, zero], or null
};

// d/32 E4M3 codes of one row (this lane's slice) decoded to floats.
template <int DIM>
__device__ __forceinline__ void load_codes(const uint8_t* __restrict__ base, size_t row,
                                           int lane, float (&x)[DIM / 32]) {
  if constexpr (DIM == 128) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(base + row * DIM + 4 * lane);
    const float2 a = e4m3x2_to_float2(w & 0xFFFFu), b = e4m3x2_to_float2(w >> 16);
    x[0] = a.x;
    x[1] = a.y;
    x[2] = b.x;
    x[3] = b.y;
  } else {
    const uint32_t w = *reinterpret_cast<const uint16_t*>(base + row * DIM + 2 * lane);
    const float2 a = e4m3x2_to_float2(w);
    x[0] = a.x;
    x[1] = a.y;
  }
}

// d = 64 NVFP4 row slice of this lane: 2 elements (one byte) times the E4M3
// scale of its 16-element group.
__device__ __forceinline__ void load_nvfp4(const uint8_t* __restrict__ codes,
                                           const uint8_t* __restrict__ scales, size_t row,
                                           int lane, float (&x)[2]) {
  const float2 v = e2m1x2_to_float2(codes[row * 32 + lane]);
  const float sc = e4m3x2_to_float2(scales[row * 4 + lane / 8]).x;
  x[0] = v.x * sc;
  x[1] = v.y * sc;
}

// Score operand rows: E4M3 codes, or the NVFP4 values on the mixed path.
template <int DIM, bool NVF4>
__device__ __forceinline__ void load_score_rows(const ShortParams& prm, bool is_q, size_t row,
                                                int lane, float (&x)[DIM / 32]) {
  if constexpr (NVF4) {
    static_assert(DIM == 64, "the NVFP4 score product is built for head dim 64");
    load_nvfp4(is_q ? prm.q4c : prm.k4c, is_q ? prm.q4s : prm.k4s, row, lane, x);
  } else {
    load_codes<DIM>(is_q ? prm.qc : prm.kc, row, lane, x);
  }
}

template <int DIM>
__device__ __forceinline__ float warp_dot(const float (&a)[DIM / 32], const float (&b)[DIM / 32]) {
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < DIM / 32; ++i) acc = fmaf(a[i], b[i], acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
}

template <int DIM>
__device__ __forceinline__ void store_bf16(__nv_bfloat16* __restrict__ dst, size_t row, int lane,
                                           const float (&x)[DIM / 32]) {
  if constexpr (DIM == 128) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
    *reinterpret_cast<uint2*>(dst + row * DIM + 4 * lane) =
        make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
    *reinterpret_cast<uint32_t*>(dst + row * DIM + 2 * lane) = *reinterpret_cast<uint32_t*>(&a);
  }
}


// The short-document kernels give each warp prm.ppw consecutive (document,
// head) pairs: each of those lanes reads one pair's length, and the warp then
// does, one after another, the pairs whose documents it handles (1 .. 32
// tokens; from 2 when the one-thread kernels took the one-token documents).
// Many pairs per warp only pay when nearly all are skipped (documents of
// about one token); otherwise one pair per warp keeps the pairs in parallel.
// Returns the mask of the lanes whose pair is done.
__device__ __forceinline__ unsigned short_pairs(const ShortParams& prm, long long p0, int units,
                                                int lane) {
  const long long pr = p0 + lane;
  int L = 0;
  if (lane < prm.ppw && pr < static_cast<long long>(prm.ndocs) * units) {
    const int doc = static_cast<int>(pr / units);
    const int s = min(max(prm.cu[doc], 0), prm.T);
    L = min(max(prm.cu[doc + 1], s), prm.T) - s;
  }
  return __ballot_sync(0xffffffffu, L >= (prm.skip_single ? 2 : 1) && L <= kShortDoc);
}

template <int DIM, bool NVF4>
__device__ __forceinline__ void fwd_short_pair(const ShortParams& prm, int doc, int h, int lane) {
  const int H = prm.H, T = prm.T;
  const int s = min(max(prm.cu[doc], 0), T);
  const int e = min(max(prm.cu[doc + 1], s), T);
  const int L = e - s;
  const size_t hT = static_cast<size_t>(h) * T;
  const int hk = h / prm.G, Hkv = prm.Hkv;
  const size_t hkT = static_cast<size_t>(hk) * T;
  // one scale block per operand: the exponents of the document's first token
  // (on the mixed path the NVFP4 values carry their own scales)
  const float cf0 = NVF4 ? prm.scale_log2
                         : prm.scale_log2 * pow2_or_zero_s(static_cast<int>(prm.qs[hT + s]) - 127) *
                               pow2_or_zero_s(static_cast<int>(prm.ks[hkT + s]) - 127);
  const float vsc0 = pow2_or_zero_s(static_cast<int>(prm.vs[hkT + s]) - 127);
  // per-token operand scales: lane j holds key j's K and V exponents
  const int ekj = prm.token && lane < L ? static_cast<int>(prm.ks[hkT + s + lane]) - 127 : 0;
  const int evj = prm.token && lane < L ? static_cast<int>(prm.vs[hkT + s + lane]) : 0;  // byte
  for (int i = 0; i < L; ++i) {
    float cf = cf0, vsc = vsc0;
    if (prm.token)
      cf = prm.scale_log2 * pow2_or_zero_s(static_cast<int>(prm.qs[hT + s + i]) - 127) *
           pow2_or_zero_s(ekj);
    float q[DIM / 32];
    load_score_rows<DIM, NVF4>(prm, true, static_cast<size_t>(s + i) * H + h, lane, q);
    // lane j keeps the raw score of key j (visible keys: j <= i, or j < L)
    const int last = prm.causal ? i : L - 1;
    float sj = 0.f;
    const bool vis = lane <= last;
    for (int j = 0; j <= last; ++j) {
      float k[DIM / 32];
      load_score_rows<DIM, NVF4>(prm, false, static_cast<size_t>(s + j) * Hkv + hk, lane, k);
      const float dot = warp_dot<DIM>(q, k);
      if (lane == j) sj = dot;
    }
    float mx = vis ? sj * cf : -INFINITY;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m = ceilf(mx);
    const float p8 = vis ? ex2_approx(fmaf(sj, cf, -(m - 8.f))) : 0.f;
    float l8 = p8;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l8 += __shfl_xor_sync(0xffffffffu, l8, off);
    float fold = 1.f;
    if (prm.token) {
      // V's per-key factor folded into P^ relative to the largest exponent
      // among the keys row i sees
      int ev = vis ? evj : 0;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ev = max(ev, __shfl_xor_sync(0xffffffffu, ev, off));
      fold = vis ? pow2_or_zero_s(evj - ev) : 0.f;
      vsc = pow2_or_zero_s(ev - 127);
    }
    const float ph = e4m3x2_to_float2(cvt_e4m3x2(p8 * fold, 0.f)).x;  // the E4M3 operand value
    float acc[DIM / 32] = {};
    for (int j = 0; j <= last; ++j) {
      const float pj = __shfl_sync(0xffffffffu, ph, j);
      float v[DIM / 32];
      load_codes<DIM>(prm.vc, static_cast<size_t>(s + j) * Hkv + hk, lane, v);
#pragma unroll
      for (int c = 0; c < DIM / 32; ++c) acc[c] = fmaf(pj, v[c], acc[c]);
    }
    const float inv = vsc / l8;
#pragma unroll
    for (int c = 0; c < DIM / 32; ++c) acc[c] *= inv;
    store_bf16<DIM>(prm.o, static_cast<size_t>(s + i) * H + h, lane, acc);
    if (lane == 0) prm.lse[hT + s + i] = (m - 8.f + __log2f(l8)) * 0.69314718055994530942f;
  }
}

template <int DIM, bool NVF4>
__global__ void __launch_bounds__(32 * kShortWarps)
    attn_fwd_short_kernel(const ShortParams prm) {
  const int lane = threadIdx.x & 31;
  const long long p0 =
      (static_cast<long long>(blockIdx.x) * kShortWarps + (threadIdx.x >> 5)) * prm.ppw;
  if (p0 >= static_cast<long long>(prm.ndocs) * prm.H) return;
  for (unsigned todo = short_pairs(prm, p0, prm.H, lane); todo != 0; todo &= todo - 1) {
    const long long pr = p0 + __ffs(todo) - 1;
    fwd_short_pair<DIM, NVF4>(prm, static_cast<int>(pr / prm.H), static_cast<int>(pr % prm.H),
                              lane);
  }
}

// One (document, head) pair of the backward, by the whole warp.  GQA: the
// pair is (document, K / V head) and walks the group's query heads; the dK /
// dV rows of the document (at most 32) sum over them in this warp's part of
// the dynamic shared memory (DIM floats per row, lane l owns its DIM / 32
// columns).  s_p / s_ds: this warp's 2^8 P (the dV operand before rounding)
// and dS of the document.
template <int DIM, bool NVF4, bool GQA>
__device__ __forceinline__ void bwd_short_pair(const ShortParams& prm, int doc, int u, int lane,
                                               int w, float (*s_p)[kShortDoc + 1],
                                               float (*s_ds)[kShortDoc + 1], float* s_acc) {
  const int H = prm.H, T = prm.T, Hkv = prm.Hkv, G = GQA ? prm.G : 1;
  const int hk = GQA ? u : u / prm.G;  // K / V head
  const int s = min(max(prm.cu[doc], 0), T);
  const int e = min(max(prm.cu[doc + 1], s), T);
  const int L = e - s;
  constexpr int N = DIM / 32;
  float* acck = s_acc + static_cast<size_t>(w) * 2 * kShortDoc * DIM;
  float* accv = acck + kShortDoc * DIM;
  if (GQA) {
    for (int j = 0; j < L; ++j)
#pragma unroll
      for (int c = 0; c < N; ++c) acck[j * DIM + N * lane + c] = accv[j * DIM + N * lane + c] = 0.f;
  }
  const size_t hkT = static_cast<size_t>(hk) * T;
  const int ek = static_cast<int>(prm.ks[hkT + s]) - 127, ev = static_cast<int>(prm.vs[hkT + s]) - 127;
  const float LOG2E = 1.4426950408889634f;
  for (int gq = 0; gq < G; ++gq) {
    const int h = GQA ? hk * G + gq : u;
    const size_t hT = static_cast<size_t>(h) * T;
    int eq = static_cast<int>(prm.qs[hT + s]) - 127;
    int edo = static_cast<int>(prm.dos[hT + s]) - 127;
    // per-token operand scales: eq, edo become the document's largest query
    // and dO exponents (the scales of Q and dO in dK and dV; each token's own
    // factor relative to them is folded into dS and P^b)
    if (prm.token) {
      int a = lane < L ? static_cast<int>(prm.qs[hT + s + lane]) : 0;
      int b = lane < L ? static_cast<int>(prm.dos[hT + s + lane]) : 0;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        a = max(a, __shfl_xor_sync(0xffffffffu, a, off));
        b = max(b, __shfl_xor_sync(0xffffffffu, b, off));
      }
      eq = a - 127;
      edo = b - 127;
    }
    const float cf = NVF4 ? prm.scale_log2 : prm.scale_log2 * pow2_or_zero_s(eq) * pow2_or_zero_s(ek);
    const float gp = pow2_or_zero_s(ev) * pow2_or_zero_s(edo);
    // P (x 2^8) and dS (x 2^8) of every visible pair, lane = key
    float amax = 0.f;
    for (int i = 0; i < L; ++i) {
      float q[N], g[N];
      load_score_rows<DIM, NVF4>(prm, true, static_cast<size_t>(s + i) * H + h, lane, q);
      load_codes<DIM>(prm.doc_, static_cast<size_t>(s + i) * H + h, lane, g);
      const float nl = 8.f - prm.lse_in[hT + s + i] * LOG2E;
      const float Di = prm.D[hT + s + i];
      // per-token operand scales: query i's own exponents against the
      // document's largest (dQ_i / dO_i factors in S and dP, folds for dK, dV)
      const int eqi = prm.token ? static_cast<int>(prm.qs[hT + s + i]) - 127 : eq;
      const int edoi = prm.token ? static_cast<int>(prm.dos[hT + s + i]) - 127 : edo;
      const float fk = pow2_or_zero_s(eqi - eq);
      for (int j = 0; j <= (prm.causal ? i : L - 1); ++j) {
        float k[N], v[N];
        load_score_rows<DIM, NVF4>(prm, false, static_cast<size_t>(s + j) * Hkv + hk, lane, k);
        load_codes<DIM>(prm.vc, static_cast<size_t>(s + j) * Hkv + hk, lane, v);
        const float sd = warp_dot<DIM>(q, k);
        const float dp = warp_dot<DIM>(g, v);
        float cfij = cf, gpij = gp;
        if (prm.token) {
          const int ekj = static_cast<int>(prm.ks[hkT + s + j]) - 127;
          const int evj = static_cast<int>(prm.vs[hkT + s + j]) - 127;
          cfij = prm.scale_log2 * pow2_or_zero_s(eqi) * pow2_or_zero_s(ekj);
          gpij = pow2_or_zero_s(evj) * pow2_or_zero_s(edoi);
        }
        const float p8 = ex2_approx(fmaf(sd, cfij, nl));
        const float d8 = p8 * fmaf(dp, gpij, -Di);
        if (lane == 0) {
          s_p[i][j] = p8;
          s_ds[i][j] = d8;
        }
        amax = fmaxf(amax, fabsf(d8 * fk));  // dK's operand (fk = 1 without token scales)
      }
    }
    __syncwarp();
    // the document is one 32x32 dS block: one round-up exponent
    const int eb = max(roundup_exponent(amax) - 8, -127);
    const float inv = exp2i(-(eb + 8)), dsc = pow2_or_zero_s(eb);
    // dQ_i = scale * sum_j dS^_ij K^_j  (float32 rows of the accumulator)
    for (int i = 0; i < L; ++i) {
      float acc[N] = {};
      float inv_i = inv, dsc_i = dsc;
      // per-token operand scales: K's per-key factor folded into dQ's dS
      // operand, which then takes query-row exponents
      auto kfold = [&](int j) {
        return prm.token ? pow2_or_zero_s(static_cast<int>(prm.ks[hkT + s + j]) - 127) : 1.f;
      };
      if (prm.ds_rows || prm.token) {  // row i's own exponent (the whole document is one key block)
        float am = 0.f;
        for (int j = 0; j <= (prm.causal ? i : L - 1); ++j)
          am = fmaxf(am, fabsf(s_ds[i][j] * kfold(j)));
        const int er = max(roundup_exponent(am) - 8, -127);
        inv_i = exp2i(-(er + 8));
        dsc_i = pow2_or_zero_s(er);
      }
      for (int j = 0; j <= (prm.causal ? i : L - 1); ++j) {
        const float dsh =
            e4m3x2_to_float2(cvt_e4m3x2(s_ds[i][j] * kfold(j) * inv_i, 0.f)).x * dsc_i;
        float k[N];
        load_codes<DIM>(prm.kc, static_cast<size_t>(s + j) * Hkv + hk, lane, k);
#pragma unroll
        for (int c = 0; c < N; ++c) acc[c] = fmaf(dsh, k[c], acc[c]);
      }
      // softmax_scale: in the BF16 conversion
      const float mul = prm.token ? 1.f : pow2_or_zero_s(ek);
      const size_t at = (static_cast<size_t>(s + i) * H + h) * DIM + N * lane;
      if (prm.dq_pre == nullptr) {
        float* dst = prm.dq_acc + at;
#pragma unroll
        for (int c = 0; c < N; ++c) dst[c] = acc[c] * mul;
      } else {  // the document's one key tile: its prescaled sum is the FP16 row
        const float pre = exp2i(prm.dq_pre[hT + s + i]);
        __half* dst = reinterpret_cast<__half*>(prm.dq_acc) + at;
#pragma unroll
        for (int c = 0; c < N; ++c) dst[c] = __float2half_rn((acc[c] * mul) * pre);
      }
    }
    // dK_j = scale * sum_i dS^_ij Q^_i,  dV_j = 2^-8 sum_i P^b_ij dO^_i
    unsigned long long cnz = 0, cz = 0;  // dS rounded-to-zero diagnostic
    for (int j = 0; j < L; ++j) {
      float ak[N] = {}, av[N] = {};
      for (int i = prm.causal ? j : 0; i < L; ++i) {
        // per-token operand scales: Q's and dO's per-query factors folded
        // into dS and P^b relative to the document's largest exponents
        float fq = 1.f, fdo = 1.f;
        if (prm.token) {
          fq = pow2_or_zero_s(static_cast<int>(prm.qs[hT + s + i]) - 127 - eq);
          fdo = pow2_or_zero_s(static_cast<int>(prm.dos[hT + s + i]) - 127 - edo);
        }
        const float dsh = e4m3x2_to_float2(cvt_e4m3x2(s_ds[i][j] * fq * inv, 0.f)).x * dsc;
        const float pb = e4m3x2_to_float2(cvt_e4m3x2(s_p[i][j] * fdo, 0.f)).x;
        if (s_ds[i][j] != 0.f) {
          ++cnz;
          if (dsh == 0.f) ++cz;
        }
        float q[N], g[N];
        load_codes<DIM>(prm.qc, static_cast<size_t>(s + i) * H + h, lane, q);
        load_codes<DIM>(prm.doc_, static_cast<size_t>(s + i) * H + h, lane, g);
#pragma unroll
        for (int c = 0; c < N; ++c) {
          ak[c] = fmaf(dsh, q[c], ak[c]);
          av[c] = fmaf(pb, g[c], av[c]);
        }
      }
      const float mk = prm.sm_scale * pow2_or_zero_s(eq), mv = pow2_or_zero_s(edo) * (1.f / 256.f);
      if (GQA) {
#pragma unroll
        for (int c = 0; c < N; ++c) {
          acck[j * DIM + N * lane + c] += ak[c] * mk;
          accv[j * DIM + N * lane + c] += av[c] * mv;
        }
      } else {
#pragma unroll
        for (int c = 0; c < N; ++c) {
          ak[c] *= mk;
          av[c] *= mv;
        }
        if (prm.hadamard) fwht_row<N, 32>(ak, lane);  // dK = dK_r H_d (the whole warp)
        store_bf16<DIM>(prm.dk, static_cast<size_t>(s + j) * Hkv + hk, lane, ak);
        store_bf16<DIM>(prm.dv, static_cast<size_t>(s + j) * Hkv + hk, lane, av);
      }
    }
    if (prm.ds_count != nullptr && lane == 0) {
      atomicAdd(prm.ds_count, cnz);
      atomicAdd(prm.ds_count + 1, cz);
    }
    __syncwarp();  // s_p / s_ds are rewritten by the next head
  }
  if (GQA) {
    for (int j = 0; j < L; ++j) {
      float ak[N], av[N];
#pragma unroll
      for (int c = 0; c < N; ++c) {
        ak[c] = acck[j * DIM + N * lane + c];
        av[c] = accv[j * DIM + N * lane + c];
      }
      if (prm.hadamard) fwht_row<N, 32>(ak, lane);
      store_bf16<DIM>(prm.dk, static_cast<size_t>(s + j) * Hkv + hk, lane, ak);
      store_bf16<DIM>(prm.dv, static_cast<size_t>(s + j) * Hkv + hk, lane, av);
    }
  }
}

template <int DIM, bool NVF4, bool GQA>
__global__ void __launch_bounds__(32 * kShortWarps)
    attn_bwd_short_kernel(const ShortParams prm) {
  __shared__ float s_p[kShortWarps][kShortDoc][kShortDoc + 1];
  __shared__ float s_ds[kShortWarps][kShortDoc][kShortDoc + 1];
  extern __shared__ float s_acc[];  // GQA: [warp][dK | dV][row][DIM]
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int units = GQA ? prm.Hkv : prm.H;
  const long long p0 = (static_cast<long long>(blockIdx.x) * kShortWarps + w) * prm.ppw;
  if (p0 >= static_cast<long long>(prm.ndocs) * units) return;
  for (unsigned todo = short_pairs(prm, p0, units, lane); todo != 0; todo &= todo - 1) {
    const long long pr = p0 + __ffs(todo) - 1;
    bwd_short_pair<DIM, NVF4, GQA>(prm, static_cast<int>(pr / units), static_cast<int>(pr % units),
                                   lane, w, s_p[w], s_ds[w], s_acc);
  }
}

// ------------------------------------------------------ one-token documents
// A document of one token is one score per head: one thread per (document,
// head) does it with whole-row loads, the same numerics as the warp kernels
// (integer maximum, E4M3 P^, the document's one dS exponent); only the order
// of the float32 dot-product sums differs.  Packed E4M3 codes of a row,
// 16 at a time.
template <int DIM>
__device__ __forceinline__ void decode16(const uint4 w, float (&x)[16]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = e4m3x2_to_float2(u[i] & 0xFFFFu), b = e4m3x2_to_float2(u[i] >> 16);
    x[4 * i] = a.x;
    x[4 * i + 1] = a.y;
    x[4 * i + 2] = b.x;
    x[4 * i + 3] = b.y;
  }
}

template <int DIM>
__device__ __forceinline__ float row_dot(const uint8_t* __restrict__ a, const uint8_t* __restrict__ b) {
  float acc = 0.f;
#pragma unroll 4
  for (int c = 0; c < DIM / 16; ++c) {
    float x[16], y[16];
    decode16<DIM>(__ldg(reinterpret_cast<const uint4*>(a) + c), x);
    decode16<DIM>(__ldg(reinterpret_cast<const uint4*>(b) + c), y);
#pragma unroll
    for (int i = 0; i < 16; ++i) acc = fmaf(x[i], y[i], acc);
  }
  return acc;
}

// f * codes of a row, as BF16, 16 elements (32 bytes) at a time.
template <int DIM>
__device__ __forceinline__ void store_scaled_bf16(__nv_bfloat16* __restrict__ dst,
                                                  const uint8_t* __restrict__ src, float p,
                                                  float f) {
#pragma unroll 2
  for (int c = 0; c < DIM / 16; ++c) {
    float x[16];
    decode16<DIM>(__ldg(reinterpret_cast<const uint4*>(src) + c), x);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // (p code) rounded as the warp kernels' fmaf(p, code, 0), then times f
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(p, x[2 * i]) * f,
                                                      __fmul_rn(p, x[2 * i + 1]) * f);
      w[i] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    uint4* d4 = reinterpret_cast<uint4*>(dst) + 2 * c;
    d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <int DIM>
__global__ void __launch_bounds__(256, 4) attn_fwd_single_kernel(const ShortParams prm) {
  const long long pair = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int H = prm.H, T = prm.T;
  if (pair >= static_cast<long long>(prm.ndocs) * H) return;
  const int doc = static_cast<int>(pair / H), h = static_cast<int>(pair % H);
  const int s = min(max(prm.cu[doc], 0), T);
  const int e = min(max(prm.cu[doc + 1], s), T);
  if (e - s != 1) return;
  const int hk = h / prm.G;
  const size_t hT = static_cast<size_t>(h) * T, hkT = static_cast<size_t>(hk) * T;
  const size_t qrow = static_cast<size_t>(s) * H + h, krow = static_cast<size_t>(s) * prm.Hkv + hk;
  const float cf = prm.scale_log2 * pow2_or_zero_s(static_cast<int>(prm.qs[hT + s]) - 127) *
                   pow2_or_zero_s(static_cast<int>(prm.ks[hkT + s]) - 127);
  const float vsc = pow2_or_zero_s(static_cast<int>(prm.vs[hkT + s]) - 127);
  const float sj = row_dot<DIM>(prm.qc + qrow * DIM, prm.kc + krow * DIM);
  const float m = ceilf(sj * cf);
  const float p8 = ex2_approx(fmaf(sj, cf, -(m - 8.f)));
  const float ph = e4m3x2_to_float2(cvt_e4m3x2(p8, 0.f)).x;
  store_scaled_bf16<DIM>(prm.o + qrow * DIM, prm.vc + krow * DIM, ph, vsc / p8);
  prm.lse[hT + s] = (m - 8.f + __log2f(p8)) * 0.69314718055994530942f;
}

// Multi-head attention without the rotation (the warp kernel does the rest).
template <int DIM>
__global__ void __launch_bounds__(256, 4) attn_bwd_single_kernel(const ShortParams prm) {
  const long long pair = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int H = prm.H, T = prm.T;
  if (pair >= static_cast<long long>(prm.ndocs) * H) return;
  const int doc = static_cast<int>(pair / H), h = static_cast<int>(pair % H);
  const int s = min(max(prm.cu[doc], 0), T);
  const int e = min(max(prm.cu[doc + 1], s), T);
  if (e - s != 1) return;
  const size_t hT = static_cast<size_t>(h) * T, row = static_cast<size_t>(s) * H + h;
  const int eq = static_cast<int>(prm.qs[hT + s]) - 127, ek = static_cast<int>(prm.ks[hT + s]) - 127;
  const int ev = static_cast<int>(prm.vs[hT + s]) - 127, edo = static_cast<int>(prm.dos[hT + s]) - 127;
  const float cf = prm.scale_log2 * pow2_or_zero_s(eq) * pow2_or_zero_s(ek);
  const float gp = pow2_or_zero_s(ev) * pow2_or_zero_s(edo);
  const float sd = row_dot<DIM>(prm.qc + row * DIM, prm.kc + row * DIM);
  const float dp = row_dot<DIM>(prm.doc_ + row * DIM, prm.vc + row * DIM);
  const float nl = 8.f - prm.lse_in[hT + s] * 1.4426950408889634f;
  const float p8 = ex2_approx(fmaf(sd, cf, nl));
  const float d8 = p8 * fmaf(dp, gp, -prm.D[hT + s]);
  // the document's one 32x32 dS block holds this one element
  const int eb = max(roundup_exponent(fabsf(d8)) - 8, -127);
  const float dsh = e4m3x2_to_float2(cvt_e4m3x2(d8 * exp2i(-(eb + 8)), 0.f)).x * pow2_or_zero_s(eb);
  const float pb = e4m3x2_to_float2(cvt_e4m3x2(p8, 0.f)).x;
  if (prm.ds_count != nullptr) {  // dS rounded-to-zero diagnostic, one add per warp
    const unsigned act = __activemask();
    const unsigned lnz = __ballot_sync(act, d8 != 0.f);
    const unsigned lz = __ballot_sync(act, d8 != 0.f && dsh == 0.f);
    if ((threadIdx.x & 31) == __ffs(act) - 1) {
      atomicAdd(prm.ds_count, static_cast<unsigned long long>(__popc(lnz)));
      atomicAdd(prm.ds_count + 1, static_cast<unsigned long long>(__popc(lz)));
    }
  }
  // dQ row of the accumulator: dS^ K^ (softmax_scale comes in the conversion)
  const float mul = pow2_or_zero_s(ek);
  const uint8_t* kc = prm.kc + row * DIM;
#pragma unroll 2
  for (int c = 0; c < DIM / 16; ++c) {
    float x[16];
    decode16<DIM>(__ldg(reinterpret_cast<const uint4*>(kc) + c), x);
    if (prm.dq_pre == nullptr) {
      float4* d4 = reinterpret_cast<float4*>(prm.dq_acc + row * DIM) + 4 * c;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        d4[i] = make_float4(__fmul_rn(dsh, x[4 * i]) * mul, __fmul_rn(dsh, x[4 * i + 1]) * mul,
                            __fmul_rn(dsh, x[4 * i + 2]) * mul, __fmul_rn(dsh, x[4 * i + 3]) * mul);
    } else {
      const float pre = exp2i(prm.dq_pre[hT + s]);
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const __half2 h2 = __floats2half2_rn((__fmul_rn(dsh, x[2 * i]) * mul) * pre,
                                             (__fmul_rn(dsh, x[2 * i + 1]) * mul) * pre);
        w[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      uint4* d4 = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(prm.dq_acc) + row * DIM) + 2 * c;
      d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
      d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
  // dK = scale 2^eq dS^ Q^,  dV = 2^(edo - 8) P^b dO^
  store_scaled_bf16<DIM>(prm.dk + row * DIM, prm.qc + row * DIM, dsh,
                         prm.sm_scale * pow2_or_zero_s(eq));
  store_scaled_bf16<DIM>(prm.dv + row * DIM, prm.doc_ + row * DIM, pb,
                         pow2_or_zero_s(edo) * (1.f / 256.f));
}

// Pairs per warp of the short-document kernels (see short_pairs).
inline int short_ppw(int T, int ndocs) { return static_cast<long long>(T) <= 2ll * ndocs ? 32 : 1; }

ShortParams make_params(const flamia_qtensor* q, const flamia_qtensor* k, const flamia_qtensor* v,
                        const int32_t* cu, int ndocs, int T, int H, int Hkv,
                        float softmax_scale) {
  ShortParams p{};
  p.q4c = q->nvfp4_codes;
  p.k4c = k->nvfp4_codes;
  p.q4s = q->nvfp4_scales;
  p.k4s = k->nvfp4_scales;
  p.qc = q->codes;
  p.kc = k->codes;
  p.vc = v->codes;
  p.qs = q->scales;
  p.ks = k->scales;
  p.vs = v->scales;
  p.cu = cu;
  p.T = T;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.ndocs = ndocs;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.sm_scale = softmax_scale;
  p.ppw = short_ppw(T, ndocs);
  return p;
}

// CTAs of a short-document kernel.
inline unsigned short_grid(int ndocs, int H, int ppw) {
  const long long warps = (static_cast<long long>(ndocs) * H + ppw - 1) / ppw;
  return static_cast<unsigned>((warps + kShortWarps - 1) / kShortWarps);
}

}  // namespace

cudaError_t launch_fwd_short(const flamia_qtensor* q, const flamia_qtensor* k,
                             const flamia_qtensor* v, const int32_t* cu, int ndocs, int T, int H,
                             int Hkv, int d, float softmax_scale, bool nvfp4_qk, bool causal,
                             bool token, void* o, float* lse, cudaStream_t stream) {
  ShortParams p = make_params(q, k, v, cu, ndocs, T, H, Hkv, softmax_scale);
  p.causal = causal ? 1 : 0;
  p.token = token ? 1 : 0;  // (one-token documents: per-token scales are block scales)
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  const unsigned grid = short_grid(ndocs, H, p.ppw);
  if (!nvfp4_qk) {  // one-token documents: one thread per (document, head)
    const unsigned g1 = static_cast<unsigned>((static_cast<long long>(ndocs) * H + 255) / 256);
    if (d == 128)
      attn_fwd_single_kernel<128><<<g1, 256, 0, stream>>>(p);
    else
      attn_fwd_single_kernel<64><<<g1, 256, 0, stream>>>(p);
    count_launches(1);
    p.skip_single = 1;
  }
  if (nvfp4_qk)
    attn_fwd_short_kernel<64, true><<<grid, 32 * kShortWarps, 0, stream>>>(p);
  else if (d == 128)
    attn_fwd_short_kernel<128, false><<<grid, 32 * kShortWarps, 0, stream>>>(p);
  else
    attn_fwd_short_kernel<64, false><<<grid, 32 * kShortWarps, 0, stream>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_bwd_short(const flamia_qtensor* q, const flamia_qtensor* k,
                             const flamia_qtensor* v, const flamia_qtensor* dout, const float* D,
                             const float* lse, const int32_t* cu, int ndocs, int T, int H,
                             int Hkv, int d, float softmax_scale, bool nvfp4_qk, bool hadamard,
                             bool causal, bool ds_rows, bool token,
                             unsigned long long* ds_count, float* dq_acc,
                             const int8_t* dq_pre, void* dk, void* dv, cudaStream_t stream) {
  ShortParams p = make_params(q, k, v, cu, ndocs, T, H, Hkv, softmax_scale);
  p.hadamard = hadamard ? 1 : 0;
  p.causal = causal ? 1 : 0;
  p.doc_ = dout->codes;
  p.dos = dout->scales;
  p.lse_in = lse;
  p.D = D;
  p.dq_acc = dq_acc;
  p.dq_pre = dq_pre;
  p.ds_rows = ds_rows ? 1 : 0;
  p.token = token ? 1 : 0;
  p.ds_count = ds_count;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  if (Hkv == H && !nvfp4_qk && !hadamard) {  // one-token documents: one thread each
    const unsigned g1 = static_cast<unsigned>((static_cast<long long>(ndocs) * H + 255) / 256);
    if (d == 128)
      attn_bwd_single_kernel<128><<<g1, 256, 0, stream>>>(p);
    else
      attn_bwd_single_kernel<64><<<g1, 256, 0, stream>>>(p);
    count_launches(1);
    p.skip_single = 1;
  }
  if (Hkv == H) {
    const unsigned grid = short_grid(ndocs, H, p.ppw);
    if (nvfp4_qk)
      attn_bwd_short_kernel<64, true, false><<<grid, 32 * kShortWarps, 0, stream>>>(p);
    else if (d == 128)
      attn_bwd_short_kernel<128, false, false><<<grid, 32 * kShortWarps, 0, stream>>>(p);
    else
      attn_bwd_short_kernel<64, false, false><<<grid, 32 * kShortWarps, 0, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
  }
  // grouped query heads: one warp per (document, K / V head), dK / dV sums in
  // dynamic shared memory (2 x 32 rows x d floats per warp)
  const unsigned grid = short_grid(ndocs, Hkv, p.ppw);
  const size_t smem = static_cast<size_t>(kShortWarps) * 2 * kShortDoc * d * sizeof(float);
  cudaError_t err;
  if (nvfp4_qk) {
    err = cudaFuncSetAttribute(attn_bwd_short_kernel<64, true, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    attn_bwd_short_kernel<64, true, true><<<grid, 32 * kShortWarps, smem, stream>>>(p);
  } else if (d == 128) {
    err = cudaFuncSetAttribute(attn_bwd_short_kernel<128, false, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    attn_bwd_short_kernel<128, false, true><<<grid, 32 * kShortWarps, smem, stream>>>(p);
  } else {
    err = cudaFuncSetAttribute(attn_bwd_short_kernel<64, false, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    attn_bwd_short_kernel<64, false, true><<<grid, 32 * kShortWarps, smem, stream>>>(p);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace flamia
