// Causal forward over token-block MXFP8 operands (FLAMIA review page, sec.
// 1.2, 3.1, 3.4).
//
// One CTA = one work item (256 queries of one document = two 128-query
// tiles) x one head.  Warp roles:
//   warp 0      TMA producer: Q tiles once, then K/V tiles through a ring.
//   warp 1      tensor-memory owner and single-thread tcgen05 MMA issuer.
//   warps 4-7   softmax of query tile 0   (thread = query row = TMEM lane)
//   warps 8-11  softmax of query tile 1
// Per key tile j the MMA warp issues S_t = Q_t K_j^T (unscaled E4M3, f32 in
// TMEM) and, once the softmax group has written the E4M3 probability tile
// P^_t back into the consumed columns of S_t, O_t += P^_t V_j as a
// block-scaled MMA with A read from tensor memory and B = V_j (its per-32-key
// E8M0 scale).  The two query tiles ping-pong so the tensor core works on one
// while the other tile's softmax runs.
// The growth of the running maximum is not applied to O in tensor memory: the
// A scale of P^_t (one E8M0 per row) carries 2^(m - m_ref) instead, and the
// epilogue divides by 2^(m - m_ref) l.
//
// Tensor memory (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d),
// O_1 [256+d, 256+2d).  Head dim 128: after the softmax has read S_t, columns
// 0..7 of S_t take the scale factors of P^_t V_j and columns 8..39 the P^_t
// codes (four per column); the next S_t MMA is issued after P^_t V_j, and
// tcgen05 MMAs of one thread execute in order.  Head dim 64: P^_t has columns
// of its own, [400 + 40 t, 440 + 40 t) in the same arrangement, so the next
// S_t is issued as soon as the softmax holds the current one in registers and
// runs while the softmax turns it into P^_t (the pages' split of the next
// score product around the current P^V); the softmax writes P^_t once the
// previous P^_t V product has read it.
// Unmasked tiles take each 32-key chunk's maximum from the max-reducing
// tensor-memory load (tcgen05.ld.red) instead of 32 comparisons.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "short_docs.cuh"

namespace flamia {
namespace {

constexpr int kStages = 3;
// first column of P^_t inside S_t (columns 0..7 hold the scale factors of P^V)
constexpr uint32_t kColP = 8;
constexpr int kFwdThreads = 384;
constexpr float kLn2 = 0.69314718055994530942f;
// Largest exponent of the per-row block scale of P^ before O is rescaled: it
// bounds O's growth over the true scale to 2^32, far inside float32 range.
constexpr int kRefSpan = 32;
// head dim 64: first column of the P^_t region (scale factors, then codes)
constexpr uint32_t kColPR = 400, kPRStride = 40;

template <int DIM, bool NVF4, bool TOK>
struct FwdSmem {
  static constexpr int kTileBytes = kTile * DIM;
  static constexpr int kTile4Bytes = NVF4 ? kTile * DIM / 2 : 16;  // packed E2M1 tile
  alignas(1024) uint8_t q[2][kTileBytes];
  alignas(1024) uint8_t k[kStages][kTileBytes];
  alignas(1024) uint8_t v[kStages][kTileBytes];
  alignas(NVF4 ? 1024 : 16) uint8_t q4[2][kTile4Bytes];
  alignas(NVF4 ? 1024 : 16) uint8_t k4[kStages][kTile4Bytes];
  uint64_t bar_sf;
  uint64_t bar_q, bar_q_empty;
  uint64_t bar_o_empty[2];
  uint64_t bar_kv_full[kStages];
  uint64_t bar_kv_empty[kStages];
  uint64_t bar_s_full[2];
  uint64_t bar_p_full[2];
  uint64_t bar_o_full[2];
  uint64_t bar_s_read[2];   // head dim 64: the softmax holds S_t in registers
  uint64_t bar_pv_done[2];  // head dim 64: P^_t V_j has read P^_t
  uint64_t bar_k4;          // head dim 64, NVFP4: the next key tile's block scales written
  uint64_t bar_done;
  ItemRing<4> ring;  // claimed items, producer -> MMA issuer and softmax warps
  // per-token operand scales: per query tile and step parity, the key factors
  // 2^eK(j), V's folded factors 2^(eV(j) - EV(block)) and the block maxima
  // EV as E8M0 bytes
  alignas(16) float kf[TOK ? 2 : 1][2][TOK ? kTile : 4];
  alignas(16) float vf[TOK ? 2 : 1][2][TOK ? kTile : 4];
  int evb[2][2][4];
  uint32_t tmem_base;
  volatile int abort;
};

struct FwdParams {
  const uint8_t* q_scales;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  const uint32_t* q4_scales;  // NVFP4: 4 E4M3 scales per (token, head) as one word (d = 64)
  const uint32_t* k4_scales;
  const int32_t* cu;
  int* wl_header;  // list sizes, and the claim counters this kernel updates
  const int4* items;
  __nv_bfloat16* o;
  float* lse;
  int T, H, ndocs, cap;
  int Hkv, G;        // K / V heads; query head h reads K / V head h / G (G = H / Hkv)
  float scale_log2;  // softmax_scale * log2(e)
  int causal;        // 0: every query sees every key of its document
  int sched;         // kSchedDynamic / kSchedRule / kSchedStatic
  int* status;
};

template <int DIM>
__host__ __device__ constexpr uint32_t operand_layout() {
  return DIM == 128 ? kLayoutSW128 : kLayoutSW64;
}

__device__ __forceinline__ float pow2_or_zero(int k) {
  return k < -126 ? 0.f : exp2i(k);
}

// Maximum of the raw scores of a 32-column chunk; MASK keeps columns <= lim.
template <bool MASK>
__device__ __forceinline__ float chunk_max(const uint32_t (&v)[32], int lim) {
  float a = -INFINITY, b = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    float x0 = __uint_as_float(v[i]), x1 = __uint_as_float(v[i + 1]);
    float x2 = __uint_as_float(v[i + 2]), x3 = __uint_as_float(v[i + 3]);
    if (MASK) {
      if (i + 0 > lim) x0 = -INFINITY;
      if (i + 1 > lim) x1 = -INFINITY;
      if (i + 2 > lim) x2 = -INFINITY;
      if (i + 3 > lim) x3 = -INFINITY;
    }
    a = fmax3(x0, x1, a);
    b = fmax3(x2, x3, b);
  }
  return fmaxf(a, b);
}

// P8 = 2^8 exp2(x cf - m) of a 32-column chunk (masked columns give 0), their
// running sum, and the E4M3 codes packed four per word.
template <bool MASK>
__device__ __forceinline__ void chunk_probs(const uint32_t (&v)[32], float cf, float moff,
                                            int lim, float2& lsum, uint32_t (&w)[8]) {
  const float2 cf2 = make_float2(cf, cf), mo2 = make_float2(-moff, -moff);
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    float2 a = make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
    float2 b = make_float2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
    a = __ffma2_rn(a, cf2, mo2);
    b = __ffma2_rn(b, cf2, mo2);
    if (MASK) {  // after the product: cf is 0 for an all-zero key block
      if (i + 0 > lim) a.x = -INFINITY;
      if (i + 1 > lim) a.y = -INFINITY;
      if (i + 2 > lim) b.x = -INFINITY;
      if (i + 3 > lim) b.y = -INFINITY;
    }
    const float2 pa = make_float2(ex2_approx(a.x), ex2_approx(a.y));
    const float2 pb = make_float2(ex2_approx(b.x), ex2_approx(b.y));
    lsum = __fadd2_rn(lsum, pa);
    lsum = __fadd2_rn(lsum, pb);
    w[i / 4] = cvt_e4m3x4(pa.x, pa.y, pb.x, pb.y);
  }
}

// Per-token operand scales: P8 = 2^8 exp2(x cf - m) as in chunk_probs, with
// v = S 2^eK(j) already carrying the key factors, and the E4M3 operand
// P8 2^(eV(j) - EV) (vf, the chunk's folded V factors, times gmul for the
// diagonal block of a causal row, whose EV is the maximum over the keys the
// row sees).
template <bool MASK>
__device__ __forceinline__ void chunk_probs_tok(const uint32_t (&v)[32], float cf, float moff,
                                                int lim, float2& lsum, uint32_t (&w)[8],
                                                const float* vf, float gmul) {
  const float2 cf2 = make_float2(cf, cf), mo2 = make_float2(-moff, -moff);
  const float2 g2 = make_float2(gmul, gmul);
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    float2 a = make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
    float2 b = make_float2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
    a = __ffma2_rn(a, cf2, mo2);
    b = __ffma2_rn(b, cf2, mo2);
    if (MASK) {
      if (i + 0 > lim) a.x = -INFINITY;
      if (i + 1 > lim) a.y = -INFINITY;
      if (i + 2 > lim) b.x = -INFINITY;
      if (i + 3 > lim) b.y = -INFINITY;
    }
    const float2 pa = make_float2(ex2_approx(a.x), ex2_approx(a.y));
    const float2 pb = make_float2(ex2_approx(b.x), ex2_approx(b.y));
    lsum = __fadd2_rn(lsum, pa);
    lsum = __fadd2_rn(lsum, pb);
    const float4 f = *reinterpret_cast<const float4*>(vf + i);
    float2 fa = make_float2(f.x, f.y), fb = make_float2(f.z, f.w);
    if (MASK) {
      fa = __fmul2_rn(fa, g2);
      fb = __fmul2_rn(fb, g2);
    }
    const float2 qa = __fmul2_rn(pa, fa), qb = __fmul2_rn(pb, fb);
    w[i / 4] = cvt_e4m3x4(qa.x, qa.y, qb.x, qb.y);
  }
}

// NVFP4 score product (d = 64): tensor-memory columns of the block scales of
// Q_0, Q_1 (4 columns each) and of K_j (two 4-column buffers, by j parity).
constexpr uint32_t kSfQ4 = 384, kSfK4 = 392;

// One forward work item (256 queries of one document x one head), decoded
// identically by every role; false for items of short documents, which the
// CUDA-core kernel handles.
struct FwdItem {
  int h, hk, s, e, q0, q1, n0, n1, nkv;  // h: query head, hk: its K / V head
  bool valid1;
};

__device__ __forceinline__ bool decode_fwd_item(const FwdParams& prm, int n_items, int idx,
                                                FwdItem& it) {
  const int T = prm.T;
  it.h = idx / n_items;  // head-major: a wave of CTAs shares the K/V of few heads
  it.hk = it.h / prm.G;
  const int4 item = prm.items[idx % n_items];
  // clamped: a malformed work list or offsets cannot index outside [0, T)
  const int doc = min(max(item.x, 0), prm.ndocs - 1);
  it.s = min(max(prm.cu[doc], 0), T);
  it.e = min(max(prm.cu[doc + 1], it.s), T);
  if (it.e - it.s <= kShortDoc) return false;
  it.q0 = it.s + ((min(max(item.y, it.s), it.e) - it.s) & ~(kTile - 1));
  it.q1 = min(max(item.z, it.q0), it.e);
  it.valid1 = it.q1 > it.q0 + kTile;
  it.n0 = (it.q0 - it.s) / kTile + 1;      // key tiles of query tile 0
  it.n1 = it.valid1 ? it.n0 + 1 : 0;       // key tiles of query tile 1
  if (!prm.causal) {  // both tiles see every key tile of the document
    it.n0 = (it.e - it.s + kTile - 1) / kTile;
    it.n1 = it.valid1 ? it.n0 : 0;
  }
  it.nkv = it.valid1 ? it.n1 : it.n0;
  return true;
}

// Consumers of the item ring: the MMA issuer and the 8 softmax warps.
constexpr int kFwdRingConsumers = 1 + 8;

template <int DIM, bool NVF4, bool TOK>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v,
                    const __grid_constant__ CUtensorMap map_q4,
                    const __grid_constant__ CUtensorMap map_k4, const FwdParams prm) {
  static_assert(!NVF4 || DIM == 64, "the NVFP4 score product is built for head dim 64");
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<DIM, NVF4, TOK>& sm = *reinterpret_cast<FwdSmem<DIM, NVF4, TOK>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int H = prm.H, T = prm.T;
  const int n_items = min(prm.wl_header[kHdrTileFwd], prm.cap);
  const int total = n_items * H;
  if (static_cast<int>(blockIdx.x) >= total) {  // uniform over the CTA
    if (threadIdx.x == 0) finish_claims(prm.wl_header + kHdrFwdNext, prm.wl_header + kHdrFwdExit);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.bar_q), 1);
    mbar_init(smem_u32(&sm.bar_q_empty), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&sm.bar_kv_full[i]), 1);
      mbar_init(smem_u32(&sm.bar_kv_empty[i]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&sm.bar_s_full[t]), 1);
      mbar_init(smem_u32(&sm.bar_p_full[t]), kTile);
      mbar_init(smem_u32(&sm.bar_o_full[t]), 1);
      mbar_init(smem_u32(&sm.bar_o_empty[t]), kTile);
      mbar_init(smem_u32(&sm.bar_s_read[t]), kTile);
      mbar_init(smem_u32(&sm.bar_pv_done[t]), 1);
    }
    mbar_init(smem_u32(&sm.bar_done), 1);
    mbar_init(smem_u32(&sm.bar_sf), 2 * kTile);
    mbar_init(smem_u32(&sm.bar_k4), kTile);
    ring_init(sm.ring, kFwdRingConsumers);
    sm.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  constexpr uint32_t kTileBytes = FwdSmem<DIM, NVF4, TOK>::kTileBytes;
  constexpr uint32_t kQBytes = kTileBytes + (NVF4 ? FwdSmem<DIM, NVF4, TOK>::kTile4Bytes : 0);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      const uint32_t bq = smem_u32(&sm.bar_q);
      int nq_loaded = 0;  // items whose Q tiles were loaded
      int kvc = 0;        // key tiles loaded over all items
      bool ok = true;
      // items in head-major, longest-first order, claimed one at a time: a CTA
      // takes the next item when it has issued its current item's last load
      Claims claims{prm.wl_header + kHdrFwdNext,
                    static_schedule(prm.sched, prm.causal, prm.items, n_items, prm.T, prm.ndocs)};
      int idx = claims.next();
      for (int n = 0; ok; ++n) {
        const bool end = idx >= total;
        if (!ring_put(sm.ring, n, end ? total : idx) || sm.abort) {
          ok = false;
          break;
        }
        if (end) break;
        FwdItem it;
        if (!decode_fwd_item(prm, n_items, idx, it)) {
          idx = claims.next();
          continue;
        }
        // the previous item's Q tiles are free once its last score product is done
        if (nq_loaded > 0 && (!mbar_wait(smem_u32(&sm.bar_q_empty), (nq_loaded - 1) & 1) ||
                              sm.abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bq, (it.valid1 ? 2 : 1) * kQBytes);
        tma_load_3d(smem_u32(sm.q[0]), &map_q, bq, 0, it.h, it.q0);
        if (it.valid1) tma_load_3d(smem_u32(sm.q[1]), &map_q, bq, 0, it.h, it.q0 + kTile);
        if (NVF4) {
          tma_load_3d(smem_u32(sm.q4[0]), &map_q4, bq, 0, it.h, it.q0);
          if (it.valid1) tma_load_3d(smem_u32(sm.q4[1]), &map_q4, bq, 0, it.h, it.q0 + kTile);
        }
        ++nq_loaded;
        for (int j = 0; j < it.nkv; ++j, ++kvc) {
          const int st = kvc % kStages;
          if (kvc >= kStages &&
              (!mbar_wait(smem_u32(&sm.bar_kv_empty[st]), ((kvc / kStages) - 1) & 1) ||
               sm.abort)) {
            ok = false;
            break;
          }
          const uint32_t bf = smem_u32(&sm.bar_kv_full[st]);
          mbar_arrive_expect_tx(bf, kTileBytes + kQBytes);
          tma_load_3d(smem_u32(sm.k[st]), &map_k, bf, 0, it.hk, it.s + j * kTile);
          tma_load_3d(smem_u32(sm.v[st]), &map_v, bf, 0, it.hk, it.s + j * kTile);
          if (NVF4) tma_load_3d(smem_u32(sm.k4[st]), &map_k4, bf, 0, it.hk, it.s + j * kTile);
        }
        if (ok) idx = claims.next();
      }
      // Drain: every issued copy has landed before the CTA can exit.
      if (nq_loaded > 0) ok &= mbar_wait(bq, (nq_loaded - 1) & 1);
      for (int j = max(0, kvc - kStages); j < kvc; ++j)
        ok &= mbar_wait(smem_u32(&sm.bar_kv_full[j % kStages]), (j / kStages) & 1);
      if (!ok) sm.abort = 1;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this role on warp-uniform values; one elected lane
    // issues each tcgen05 instruction.
    {
      constexpr uint32_t lay = operand_layout<DIM>();
      constexpr uint32_t sbo = 8 * DIM;  // 8 rows of one swizzle atom
      const uint32_t id_qk = idesc_f8(kTile, kTile, 0, 0);
      // operand descriptors, built once: a K step, tile or ring stage moves only
      // the start address (bits 0..13, address / 16), which never carries out
      // of its field inside shared memory
      const uint64_t dq0 = smem_desc(smem_u32(sm.q[0]), 0, sbo, lay);
      const uint64_t dk0 = smem_desc(smem_u32(sm.k[0]), 0, sbo, lay);
      const uint64_t dv0 = smem_desc(smem_u32(sm.v[0]), 0, sbo, lay);
      constexpr uint32_t kStep = kTile * DIM / 16;  // one tile's bytes / 16
      // running counts of each barrier's completions (phase parity = count & 1)
      int nq_used = 0, kvc = 0, o_used[2] = {0, 0}, p_seen[2] = {0, 0};
      int s_issued[2] = {0, 0}, s_read_seen[2] = {0, 0};  // head dim 64
      int k4_seen = 0;  // head dim 64, NVFP4: key tiles whose block scales were written
      constexpr bool kSep = DIM == 64;
      bool ok = true;
      // head dim 64: S_t may be overwritten once the softmax has read every
      // S_t issued before (its s_read arrivals)
      auto wait_s_read = [&](int t) -> bool {
        while (s_read_seen[t] < s_issued[t]) {
          if (!mbar_wait_w_ab(smem_u32(&sm.bar_s_read[t]), s_read_seen[t] & 1, &sm.abort))
            return false;
          ++s_read_seen[t];
        }
        return true;
      };
      // S_t = Q_t K^T of the key tile with global index jk into columns [128 t, 128 t + 128)
      auto issue_qk = [&](int t, int jk) {
        const int st = jk % kStages;
        if (NVF4) {
          // packed E2M1 rows of 32 bytes, 32-byte swizzle, one K = 64 product
          mma_nvf4_w(tmem + t * kTile, smem_desc(smem_u32(sm.q4[t]), 0, 256, kLayoutSW32),
                   smem_desc(smem_u32(sm.k4[st]), 0, 256, kLayoutSW32), idesc_nvf4(kTile, kTile),
                   tmem + kSfQ4 + 4 * t, tmem + kSfK4 + 4 * (jk & 1), 0);
        } else {
          const uint64_t dq = dq0 + t * kStep, dk = dk0 + st * kStep;
#pragma unroll
          for (int ks = 0; ks < DIM / 32; ++ks)
            mma_f8_w(tmem + t * kTile, dq + 2 * ks, dk + 2 * ks, id_qk, ks > 0);
        }
        tc_commit_w(smem_u32(&sm.bar_s_full[t]));
        ++s_issued[t];
      };
      for (int n = 0; ok; ++n) {
        // every lane takes lane 0's copy; one arrive frees the slot
        const int idx = __shfl_sync(0xffffffffu, ring_get(sm.ring, n, false), 0);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.ring.empty[n % 4]));
        if (idx < 0) {
          ok = false;
          break;
        }
        if (idx >= total) break;
        FwdItem it;
        if (!decode_fwd_item(prm, n_items, idx, it)) continue;
        ok = mbar_wait_w(smem_u32(&sm.bar_q), nq_used & 1) &&
             mbar_wait_w(smem_u32(&sm.bar_kv_full[kvc % kStages]), (kvc / kStages) & 1);
        if (NVF4) ok = ok && mbar_wait_w(smem_u32(&sm.bar_sf), nq_used & 1);
        ++nq_used;
        if (!ok || __any_sync(0xffffffffu, sm.abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (kSep && (!wait_s_read(0) || (it.valid1 && !wait_s_read(1)))) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_qk(0, kvc);
        if (it.valid1) issue_qk(1, kvc);
        int kv_ready = kvc + 1;  // key tiles known loaded: global indices < kv_ready
        for (int j = 0; kSep && ok && j < it.nkv; ++j) {
          const int jk = kvc + j, st = jk % kStages;
          // NVFP4: the next key tile's block scales are written by group 0 (in
          // its step j, or in step n0 - 1 for tile 1's last key tile)
          if (NVF4 && j + 1 < it.nkv) {
            if (!mbar_wait_w(smem_u32(&sm.bar_k4), k4_seen & 1)) {
              ok = false;
              break;
            }
            ++k4_seen;
          }
          // the next S_t of both tiles, each once its softmax holds the current one
          for (int t = 0; t < 2 && ok; ++t) {
            const int nt = t == 0 ? it.n0 : it.n1;
            if (j + 1 >= nt) continue;
            if (kv_ready <= jk + 1) {
              if (!mbar_wait_w(smem_u32(&sm.bar_kv_full[(jk + 1) % kStages]),
                               ((jk + 1) / kStages) & 1)) {
                ok = false;
                break;
              }
              kv_ready = jk + 2;
            }
            if (!wait_s_read(t)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_qk(t, jk + 1);
          }
          for (int t = 0; t < 2 && ok; ++t) {
            const int nt = t == 0 ? it.n0 : it.n1;
            if (j >= nt) continue;
            if (!mbar_wait_w_ab(smem_u32(&sm.bar_p_full[t]), p_seen[t] & 1, &sm.abort)) {
              ok = false;
              break;
            }
            ++p_seen[t];
            if (j == 0 && o_used[t] > 0 &&
                !mbar_wait_w(smem_u32(&sm.bar_o_empty[t]), (o_used[t] - 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t dv = dv0 + st * kStep;
            const uint32_t sf = tmem + kColPR + kPRStride * t;
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)
              mma_mxf8_ts_w(tmem + 256 + t * DIM, sf + kColP + 8 * kb, dv + kb * (32 * DIM / 16),
                            idesc_mxf8(kTile, DIM, 0, 1, kb, kb), sf, sf + 4, (j > 0 || kb > 0));
            tc_commit_w(smem_u32(&sm.bar_pv_done[t]));
            if (j + 1 == nt) {
              tc_commit_w(smem_u32(&sm.bar_o_full[t]));
              ++o_used[t];
            }
          }
          if (ok) tc_commit_w(smem_u32(&sm.bar_kv_empty[st]));
        }
        for (int j = 0; !kSep && ok && j < it.nkv; ++j) {
          const int jk = kvc + j, st = jk % kStages;
          for (int t = 0; t < 2 && ok; ++t) {
            const int nt = t == 0 ? it.n0 : it.n1;
            if (j >= nt) continue;
            if (!mbar_wait_w_ab(smem_u32(&sm.bar_p_full[t]), p_seen[t] & 1, &sm.abort)) {
              ok = false;
              break;
            }
            ++p_seen[t];
            // the first P^V of an item overwrites O_t: the previous item's
            // epilogue must have read it
            if (j == 0 && o_used[t] > 0 &&
                !mbar_wait_w(smem_u32(&sm.bar_o_empty[t]), (o_used[t] - 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t dv = dv0 + st * kStep;
            // S_t columns 0..7 hold the scale factors, 8..39 the E4M3 P^_t (A
            // from tensor memory: 4 keys per column, 8 columns per 32-key step)
            const uint32_t sf = tmem + t * kTile;
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)
              mma_mxf8_ts_w(tmem + 256 + t * DIM, sf + kColP + 8 * kb, dv + kb * (32 * DIM / 16),
                          idesc_mxf8(kTile, DIM, 0, 1, kb, kb), sf, sf + 4, (j > 0 || kb > 0));
            if (j + 1 < nt) {
              if (kv_ready <= jk + 1) {
                if (!mbar_wait_w(smem_u32(&sm.bar_kv_full[(jk + 1) % kStages]),
                                 ((jk + 1) / kStages) & 1)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                kv_ready = jk + 2;
              }
              issue_qk(t, jk + 1);
            } else {
              tc_commit_w(smem_u32(&sm.bar_o_full[t]));
              ++o_used[t];
            }
          }
          if (ok) tc_commit_w(smem_u32(&sm.bar_kv_empty[st]));
        }
        kvc += it.nkv;
        // this item's Q tiles may be replaced once its products are done
        if (ok) tc_commit_w(smem_u32(&sm.bar_q_empty));
      }
      if (!ok) sm.abort = 1;
      // Drain: all MMAs of this thread complete before tensor memory is freed.
      tc_commit_w(smem_u32(&sm.bar_done));
      if (!mbar_wait_w(smem_u32(&sm.bar_done), 0)) sm.abort = 1;
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * kTile;
    const uint32_t tO = tmem + lane_off + 256 + t * DIM;
    int s_seen = 0, o_seen = 0;  // completions of s_full[t] and o_full[t] waited so far
    int pv_seen = 0;             // head dim 64: completions of pv_done[t] waited so far
    constexpr bool kSep = DIM == 64;
    const uint32_t tP = kSep ? tmem + lane_off + kColPR + kPRStride * t : tS;
    int kvc = 0;                 // global index of the current item's first key tile
    bool ok = true;
    for (int n = 0; ok; ++n) {
      // the whole warp takes lane 0's copy, so its lanes never disagree
      const int idx = __shfl_sync(0xffffffffu, ring_get(sm.ring, n, false), 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.ring.empty[n % 4]));
      if (idx < 0) {
        ok = false;
        break;
      }
      if (idx >= total) break;
      FwdItem it;
      if (!decode_fwd_item(prm, n_items, idx, it)) continue;
      const int h = it.h, s = it.s, e = it.e;
      const size_t hkT = static_cast<size_t>(it.hk) * T;  // K / V scale rows
      const int nt = t == 0 ? it.n0 : it.n1;
      const int kv0 = kvc;
      kvc += it.nkv;
      const int qa = it.q0 + t * kTile;
      const int qi = qa + r;
      const bool row_valid = qi < it.q1;
      const size_t hT = static_cast<size_t>(h) * T;
      const int eq = NVF4 ? 0 : static_cast<int>(prm.q_scales[hT + min(qi, T - 1)]) - 127;
      const float c_row = prm.scale_log2 * pow2_or_zero(eq);
      // m: running integer row maximum (log2 units); l8 = sum of 2^8 exp2(s - m);
      // m_ref: the maximum whose scale O_t is kept in (see the block scale of P^ below)
      float m = -INFINITY, l8 = 0.f, m_ref = 0.f;
      // NVFP4 score product: its block scales live in tensor memory, one 32-bit
      // word (4 E4M3 scales) per row; column c + i of this lane quadrant holds
      // row 32 i + lane (the same words in every quadrant).
      auto write_sf4 = [&](const uint32_t* words, int heads, int hh, int tok0, uint32_t col) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w[i] = words[static_cast<size_t>(min(tok0 + 32 * i + lane, T - 1)) * heads + hh];
        tmem_st4(tmem + lane_off + col, w);
      };
      if (NVF4) {
        // K scales go to the buffer of the key tile's global parity (it was
        // last read by the products of the key tile two before, complete once
        // this group saw the previous item's O_0)
        write_sf4(prm.q4_scales, H, h, qa, kSfQ4 + 4 * t);
        if (t == 0) write_sf4(prm.k4_scales, prm.Hkv, it.hk, s, kSfK4 + 4 * (kv0 & 1));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.bar_sf));
      }
      // E8M0 bytes of the 4 key blocks of key tile jj, fetched a step ahead:
      // lane kb loads K block kb's byte, lane 4 + kb V block kb's (the same
      // bytes serve every row, so one load per lane and the warp shares them)
      uint32_t sbyte = 127u;
      auto fetch_scales = [&](int jj) {
        const int kk = s + jj * kTile + 32 * (lane & 3);
        const bool in = lane < 8 && (lane >= 4 || !NVF4) && jj < nt && kk < e;
        sbyte = in ? (lane < 4 ? prm.k_scales : prm.v_scales)[hkT + kk] : 127u;
      };
      fetch_scales(0);
      // per-token operand scales: this thread's key r of key tile jj (its K and
      // V exponent bytes, 0 outside the document), fetched a step ahead
      int r_ek = 0, r_ev = 0;
      auto fetch_token_bytes = [&](int jj) {
        const int kk = s + jj * kTile + r;
        const bool in = jj < nt && kk < e;
        r_ek = in ? static_cast<int>(prm.k_scales[hkT + kk]) : 0;
        r_ev = in ? static_cast<int>(prm.v_scales[hkT + kk]) : 0;
      };
      if (TOK) fetch_token_bytes(0);
      for (int j = 0; j < nt; ++j) {
        const int k0 = s + j * kTile;
        // per-token operand scales: this step's key tables (buffer j & 1, last
        // read in step j - 2, before the group's barrier of step j - 1)
        int pm = 0, own_max = 0;  // the row's diagonal-block maxima (bytes)
        if constexpr (TOK) {
          const int kk = k0 + r;
          const bool kin = kk < e;
          own_max = __reduce_max_sync(0xffffffffu, r_ev);  // this warp's key block
          pm = r_ev;  // inclusive prefix maximum over lanes 0 .. lane
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, pm, off);
            if (lane >= off) pm = max(pm, y);
          }
          sm.kf[j & 1][t][r] = kin ? pow2_or_zero(r_ek - 127) : 0.f;
          sm.vf[j & 1][t][r] = kin ? pow2_or_zero(r_ev - own_max) : 0.f;
          if (lane == 0) sm.evb[j & 1][t][quad] = own_max;
          fetch_token_bytes(j + 1);
          named_barrier_sync(1 + t, kTile);
        }
        // lanes 0..3 gather the K word, lanes 4..7 the V word (byte kb = block kb)
        uint32_t sw = sbyte << (8 * (lane & 3));
        sw |= __shfl_xor_sync(0xffffffffu, sw, 1);
        sw |= __shfl_xor_sync(0xffffffffu, sw, 2);
        const uint32_t kword = __shfl_sync(0xffffffffu, sw, 0);
        const uint32_t sfb = __shfl_sync(0xffffffffu, sw, 4);
        float cf[4];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)  // c_row 2^(byte - 127); byte 0 gives 0
          cf[kb] = c_row * __int_as_float(((kword >> (8 * kb)) & 0xFFu) << 23);
        fetch_scales(j + 1);  // in flight while this tile is processed
        if (!mbar_wait_ab(smem_u32(&sm.bar_s_full[t]), s_seen & 1, &sm.abort)) {
          ok = false;
          break;
        }
        ++s_seen;
        tc_fence_after();
        // the last key tile holds the diagonal (causal) or the document end
        const bool diag = (j == nt - 1);
        const int lim = diag ? min(prm.causal ? r : kTile - 1, e - 1 - k0) : kTile - 1;
        // the whole 128-column row of S_t in registers: four loads, one wait;
        // unmasked tiles get each chunk's maximum with the load
        uint32_t sv[4][32];
        float cmx[4];
        if (diag || TOK) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, sv[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32_max(tS + 32 * c, sv[c], cmx[c]);
        }
        tmem_ld_wait();
        if (kSep) {
          // NVFP4: group 0 stages the block scales of the next key tile before
          // the next S products may be issued (their buffer was last read by
          // the score products of key tile j - 1, complete before S_0 of tile j)
          if (NVF4 && t == 0 && j + 1 < it.nkv) {
            write_sf4(prm.k4_scales, prm.Hkv, it.hk, k0 + kTile, kSfK4 + 4 * ((kv0 + j + 1) & 1));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&sm.bar_k4));
          }
          // S_t is in registers: the next S_t may be computed
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.bar_s_read[t]));
        }
        // pass 1: row maximum in the log2 domain
        float mx = -INFINITY;
        if constexpr (TOK) {
          // the key factors 2^eK(j) per column, then one row factor
          const float* kfp = sm.kf[j & 1][t];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 f = *reinterpret_cast<const float4*>(kfp + 32 * c + i);
              const float2 a = __fmul2_rn(
                  make_float2(__uint_as_float(sv[c][i]), __uint_as_float(sv[c][i + 1])),
                  make_float2(f.x, f.y));
              const float2 b = __fmul2_rn(
                  make_float2(__uint_as_float(sv[c][i + 2]), __uint_as_float(sv[c][i + 3])),
                  make_float2(f.z, f.w));
              sv[c][i] = __float_as_uint(a.x);
              sv[c][i + 1] = __float_as_uint(a.y);
              sv[c][i + 2] = __float_as_uint(b.x);
              sv[c][i + 3] = __float_as_uint(b.y);
            }
            const float cm = diag ? chunk_max<true>(sv[c], lim - 32 * c) : chunk_max<false>(sv[c], 0);
            mx = fmaxf(mx, cm * c_row);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float cm = diag ? chunk_max<true>(sv[c], lim - 32 * c) : cmx[c];
            mx = fmaxf(mx, cm * cf[c]);
          }
        }
        float m_new = (mx == -INFINITY) ? m : fmaxf(m, ceilf(mx));
        if (m_new == -INFINITY) m_new = 0.f;
        if (j == 0) m_ref = m_new;
        if (j > 0 && m_new > m) l8 *= pow2_or_zero(static_cast<int>(m - m_new));
        m = m_new;
        const float moff = m - 8.f;  // P8 = 2^8 exp2(s - m)
        // pass 2: probabilities, row sum, E4M3 operand (the codes stay in
        // registers until P^_t's columns are free)
        float2 lsum = make_float2(0.f, 0.f);
        // per-token operand scales, causal diagonal tile: the row's own key
        // block takes EV = the maximum over the keys it sees
        const bool tdiag = TOK && diag && prm.causal;
        const float gown = tdiag ? pow2_or_zero(own_max - pm) : 1.f;
        uint32_t pcode[4][8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if constexpr (TOK) {
            const float* vfp = sm.vf[j & 1][t] + 32 * c;
            if (diag)
              chunk_probs_tok<true>(sv[c], c_row, moff, lim - 32 * c, lsum, pcode[c], vfp,
                                    (tdiag && c == quad) ? gown : 1.f);
            else
              chunk_probs_tok<false>(sv[c], c_row, moff, 0, lsum, pcode[c], vfp, 1.f);
          } else if (diag) {
            chunk_probs<true>(sv[c], cf[c], moff, lim - 32 * c, lsum, pcode[c]);
          } else {
            chunk_probs<false>(sv[c], cf[c], moff, 0, lsum, pcode[c]);
          }
        }
        // head dim 64: P^_t's columns are free once the previous P^_t V has
        // read them (waited for only now, so the wait overlaps the exponentials)
        if (kSep && j > 0) {
          if (!mbar_wait_ab(smem_u32(&sm.bar_pv_done[t]), pv_seen & 1, &sm.abort)) {
            ok = false;
            break;
          }
          ++pv_seen;
          tc_fence_after();
        }
        // the 32 codes of each chunk: row r of P^_t, keys 32 c .. 32 c + 31, into
        // P^_t's columns (head dim 128: the consumed columns of S_t)
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_st8(tP + kColP + 8 * c, pcode[c]);
        l8 += lsum.x + lsum.y;
        // P^_t V_j enters O_t with the block scale 2^(m - m_ref) on P^'s row:
        // O_t stays in the scale of m_ref and needs no rescaling when the
        // maximum grows (powers of two: the same sums, exactly).  Only a growth
        // past kRefSpan moves m_ref, rescaling O_t once; the products into O_t
        // of key tile j - 1 completed before S_t of tile j.
        int dm = static_cast<int>(m - m_ref);
        if (__any_sync(0xffffffffu, dm > kRefSpan)) {
          const float c = pow2_or_zero(-dm);
          const float2 c2 = make_float2(c, c);
#pragma unroll 1
          for (int c0 = 0; c0 < DIM / 32; c0 += 2) {
            uint32_t a[32], b[32];
            tmem_ld32(tO + 32 * c0, a);
            tmem_ld32(tO + 32 * (c0 + 1), b);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float2 x = __fmul2_rn(make_float2(__uint_as_float(a[i]), __uint_as_float(a[i + 1])), c2);
              float2 y = __fmul2_rn(make_float2(__uint_as_float(b[i]), __uint_as_float(b[i + 1])), c2);
              a[i] = __float_as_uint(x.x);
              a[i + 1] = __float_as_uint(x.y);
              b[i] = __float_as_uint(y.x);
              b[i + 1] = __float_as_uint(y.y);
            }
            tmem_st32(tO + 32 * c0, a);
            tmem_st32(tO + 32 * (c0 + 1), b);
          }
          m_ref = m;
          dm = 0;
        }
        // scale factors of P^_t V_j: A (P^, this row) 2^dm for every K block
        // (each lane quadrant holds its own rows), B = V's block bytes
        uint32_t sa = static_cast<uint32_t>(127 + dm) * 0x01010101u, sb = sfb;
        if constexpr (TOK) {
          // A: 2^(dm + EV(block)) per key block (the V factors were folded into
          // P^ relative to EV); B: 2^0
          const int* evb = sm.evb[j & 1][t];
          sa = 0;
          bool bad = false;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int byte = dm + ((tdiag && b == quad) ? pm : evb[b]);
            bad |= byte > 254;
            sa |= static_cast<uint32_t>(min(byte, 254)) << (8 * b);
          }
          if (bad) report(prm.status, FLAMIA_DEV_RANGE);
          sb = 0x7F7F7F7Fu;
        }
        const uint32_t sfw[8] = {sa, sa, sa, sa, sb, sb, sb, sb};
        tmem_st8(tP, sfw);
        // NVFP4: group 0 stages the block scales of the next key tile (its
        // buffer was last read by the products of key tile j - 1, which
        // completed before S_0 of tile j)
        if (NVF4 && !kSep && t == 0 && j + 1 < it.nkv)
          write_sf4(prm.k4_scales, prm.Hkv, it.hk, k0 + kTile, kSfK4 + 4 * ((kv0 + j + 1) & 1));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.bar_p_full[t]));
      }
      if (nt > 0 && ok) {
        if (!mbar_wait_ab(smem_u32(&sm.bar_o_full[t]), o_seen & 1, &sm.abort)) ok = false;
        ++o_seen;
        // head dim 64: the item's last P^_t V (complete with O_t) consumes its phase
        if (kSep && ok) {
          if (!mbar_wait(smem_u32(&sm.bar_pv_done[t]), pv_seen & 1)) ok = false;
          ++pv_seen;
        }
      }
      if (nt > 0 && ok) {
        tc_fence_after();
        const float inv = pow2_or_zero(static_cast<int>(m_ref - m)) / l8;
        __nv_bfloat16* orow = prm.o + (static_cast<size_t>(qi) * H + h) * DIM;
#pragma unroll 1
        for (int c = 0; c < DIM / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tO + 32 * c, v);
          tmem_ld_wait();
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * inv,
                                                      __uint_as_float(v[2 * i + 1]) * inv);
            w[i] = *reinterpret_cast<uint32_t*>(&b2);
          }
          if (row_valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
            dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
          }
        }
        if (row_valid) prm.lse[hT + qi] = (m - 8.f + __log2f(l8)) * kLn2;
        // O_t may now be overwritten by the next item
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.bar_o_empty[t]));
      }
    }
    if (!ok) sm.abort = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (sm.abort) report(prm.status, FLAMIA_DEV_TIMEOUT);
    finish_claims(prm.wl_header + kHdrFwdNext, prm.wl_header + kHdrFwdExit);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DIM, bool NVF4, bool TOK>
flamia_status launch_fwd(const flamia_qtensor* q, const flamia_qtensor* k,
                         const flamia_qtensor* v, const int32_t* cu, int ndocs, int T, int H,
                         int Hkv, float softmax_scale, bool causal, int sched, void* wl, void* o,
                         float* lse, int* status, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mq4, mk4;
  const CUtensorMapSwizzle swz = swizzle_for_row_bytes(DIM);
  if (!make_token_map(&mq, q->codes, T, H, DIM, kTile, swz) ||
      !make_token_map(&mk, k->codes, T, Hkv, DIM, kTile, swz) ||
      !make_token_map(&mv, v->codes, T, Hkv, DIM, kTile, swz))
    return FLAMIA_ERR_CUDA;
  if (NVF4) {
    if (!make_token_map(&mq4, q->nvfp4_codes, T, H, DIM / 2, kTile, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_token_map(&mk4, k->nvfp4_codes, T, Hkv, DIM / 2, kTile, CU_TENSOR_MAP_SWIZZLE_32B))
      return FLAMIA_ERR_CUDA;
  } else {
    mq4 = mq;
    mk4 = mk;
  }
  const WorklistLayout L = worklist_layout(T, ndocs);
  FwdParams prm;
  prm.q_scales = q->scales;
  prm.k_scales = k->scales;
  prm.v_scales = v->scales;
  prm.q4_scales = reinterpret_cast<const uint32_t*>(q->nvfp4_scales);
  prm.k4_scales = reinterpret_cast<const uint32_t*>(k->nvfp4_scales);
  prm.cu = cu;
  prm.wl_header = static_cast<int*>(wl);
  prm.items = reinterpret_cast<const int4*>(static_cast<const char*>(wl) + L.off_tile_fwd);
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.T = T;
  prm.H = H;
  prm.Hkv = Hkv;
  prm.G = H / Hkv;
  prm.ndocs = ndocs;
  prm.cap = L.cap_fwd;
  prm.scale_log2 = softmax_scale * 1.4426950408889634f;
  prm.causal = causal ? 1 : 0;
  prm.sched = sched;
  prm.status = status;
  const size_t smem = sizeof(FwdSmem<DIM, NVF4, TOK>) + 1024;
  if (cudaFuncSetAttribute(attn_fwd_kernel<DIM, NVF4, TOK>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return FLAMIA_ERR_CUDA;
  // persistent: one CTA per SM (shared memory allows one), items claimed in list order
  const long long grid = std::min<long long>(static_cast<long long>(L.cap_fwd) * H, num_sms());
  attn_fwd_kernel<DIM, NVF4, TOK>
      <<<static_cast<unsigned>(grid), kFwdThreads, smem, stream>>>(mq, mk, mv, mq4, mk4, prm);
  if (cudaGetLastError() != cudaSuccess) return FLAMIA_ERR_CUDA;
  count_launches(1);
  return launch_fwd_short(q, k, v, cu, ndocs, T, H, Hkv, DIM, softmax_scale, NVF4, causal, TOK,
                          o, lse, stream) ==
                 cudaSuccess
             ? FLAMIA_OK
             : FLAMIA_ERR_CUDA;
}

}  // namespace
}  // namespace flamia

using namespace flamia;

extern "C" flamia_status flamia_attn_fwd_gqa(const flamia_qtensor* q, const flamia_qtensor* k,
                                             const flamia_qtensor* v, const int32_t* cu_seqlens,
                                             int ndocs, int T, int H, int H_kv, int d,
                                             float softmax_scale, int flags, void* wl,
                                             void* o_bf16, float* lse, int* dev_status,
                                             void* stream) {
  if (!supported_dim(d)) return FLAMIA_ERR_UNSUPPORTED;
  if (H_kv <= 0 || H <= 0 || H % H_kv != 0) return FLAMIA_ERR_INVALID_ARG;
  // the backward's dQ options are accepted and have nothing to do here (every
  // output row of the forward is written by one CTA)
  if ((flags & ~(FLAMIA_FLAG_NVFP4_QK | FLAMIA_FLAG_HADAMARD | FLAMIA_FLAG_NONCAUSAL |
                 FLAMIA_FLAG_DETERMINISTIC_DQ | FLAMIA_FLAG_DQ_FP16 |
                 FLAMIA_FLAG_DQ_CAUSAL_SCALE | FLAMIA_FLAG_SCHEDULE_STATIC |
                 FLAMIA_FLAG_SCHEDULE_RULE | FLAMIA_FLAG_DS_ROW_EXPONENTS |
                 FLAMIA_FLAG_TOKEN_SCALES | FLAMIA_FLAG_DS_ZERO_COUNT)) != 0)
    return FLAMIA_ERR_UNSUPPORTED;
  const int sched = schedule_of(flags);
  if (sched < 0) return FLAMIA_ERR_UNSUPPORTED;
  const bool nvf4 = (flags & FLAMIA_FLAG_NVFP4_QK) != 0;
  const bool tok = (flags & FLAMIA_FLAG_TOKEN_SCALES) != 0;
  if (tok && nvf4) return FLAMIA_ERR_UNSUPPORTED;
  const bool causal = (flags & FLAMIA_FLAG_NONCAUSAL) == 0;
  if ((nvf4 && d != 64) || (nvf4 && (flags & FLAMIA_FLAG_HADAMARD))) return FLAMIA_ERR_UNSUPPORTED;
  // rotated Q, K (FLAMIA_FLAG_HADAMARD): the same scores with softmax_scale / d
  // (exact: d = 2^k)
  if (flags & FLAMIA_FLAG_HADAMARD) softmax_scale /= static_cast<float>(d);
  if (!valid_sizes(T, H, d, ndocs) || q == nullptr || k == nullptr || v == nullptr ||
      cu_seqlens == nullptr || wl == nullptr || o_bf16 == nullptr || lse == nullptr ||
      !(softmax_scale > 0.f))
    return FLAMIA_ERR_INVALID_ARG;
  if (!q->codes || !q->scales || !k->codes || !k->scales || !v->codes || !v->scales)
    return FLAMIA_ERR_INVALID_ARG;
  if (!aligned(q->codes, 16) || !aligned(k->codes, 16) || !aligned(v->codes, 16) ||
      !aligned(o_bf16, 16) || !aligned(wl, 256))
    return FLAMIA_ERR_INVALID_ARG;
  if (nvf4 && (!q->nvfp4_codes || !q->nvfp4_scales || !k->nvfp4_codes || !k->nvfp4_scales ||
               !aligned(q->nvfp4_codes, 16) || !aligned(k->nvfp4_codes, 16) ||
               !aligned(q->nvfp4_scales, 4) || !aligned(k->nvfp4_scales, 4)))
    return FLAMIA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (nvf4)
    return launch_fwd<64, true, false>(q, k, v, cu_seqlens, ndocs, T, H, H_kv, softmax_scale,
                                       causal, sched, wl, o_bf16, lse, dev_status, s);
  if (tok)
    return d == 128 ? launch_fwd<128, false, true>(q, k, v, cu_seqlens, ndocs, T, H, H_kv,
                                                   softmax_scale, causal, sched, wl, o_bf16, lse,
                                                   dev_status, s)
                    : launch_fwd<64, false, true>(q, k, v, cu_seqlens, ndocs, T, H, H_kv,
                                                  softmax_scale, causal, sched, wl, o_bf16, lse,
                                                  dev_status, s);
  return d == 128 ? launch_fwd<128, false, false>(q, k, v, cu_seqlens, ndocs, T, H, H_kv,
                                                  softmax_scale, causal, sched, wl, o_bf16, lse,
                                                  dev_status, s)
                  : launch_fwd<64, false, false>(q, k, v, cu_seqlens, ndocs, T, H, H_kv,
                                                 softmax_scale, causal, sched, wl, o_bf16, lse,
                                                 dev_status, s);
}

// The forward keeps its running statistics and probabilities on chip: no
// workspace at any size.
extern "C" size_t flamia_fwd_workspace_bytes(int, int, int) { return 0; }

extern "C" flamia_status flamia_attn_fwd(const flamia_qtensor* q, const flamia_qtensor* k,
                                         const flamia_qtensor* v, const int32_t* cu_seqlens,
                                         int ndocs, int T, int H, int d, float softmax_scale,
                                         int flags, void* wl, void* o_bf16, float* lse,
                                         int* dev_status, void* stream) {
  return flamia_attn_fwd_gqa(q, k, v, cu_seqlens, ndocs, T, H, H, d, softmax_scale, flags, wl,
                             o_bf16, lse, dev_status, stream);
}
