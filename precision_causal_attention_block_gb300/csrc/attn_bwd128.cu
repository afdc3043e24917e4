// Causal backward for head dim 128 over token-block MXFP8 operands (FLAMIA
// review page, sec. 1.2, 3.1, 3.3, 3.4 "Backward pass"), pipelined so that
// the tensor core and the CUDA cores work at the same time.
//
// One work item = one 128-key tile of a document x one head (persistent CTAs
// claiming items as in the other kernels).  The item's queries are
// walked in 64-query tiles t from the diagonal to the document end; the two
// compute groups take alternate tiles, each with its own half of tensor memory:
//
//   TMEM columns  [64b, 64b+64)     S^T_t (keys x queries), then dQ^T_t
//                 [128+64b, +64)    dP^T_t, then the block scales of tile t
//                 [256, 384)        dV accumulator   [384, 512) dK accumulator
//   (b = t & 1 = the compute group of tile t)
//
// While group b turns S^T_t / dP^T_t into the dV operand RNE_E4M3(2^8 P) and
// the dS codes, the tensor core runs the products of the other group's tile;
// its S^T / dP^T for tile t+2 start as soon as dQ^T_t has been read out.
//   S^T_t = K Q_t^T, dP^T_t = V dO_t^T          (unscaled E4M3, M=128, N=64)
//   dV += P^b_t^T dO_t, dK += dS_t^T Q_t         (block-scaled, M=128, N=128, K=64)
//   dQ_t^T = K^T dS_t^T                          (block-scaled, M=128 dims, N=64)
// dQ_t^T is read with one thread per head-dim row, staged as [query][dim]
// float32 rows and added to the global accumulator by bulk tensor reduce-adds.
//
// Warp roles: warp 0 TMA producer (K, V per item; Q, dO 64-row tiles through a
// 4-stage ring), warp 1 tensor-memory owner and single-thread MMA issuer,
// warps 4-7 compute group 0, warps 8-11 compute group 1 (thread = key row for
// S^T / dP^T / dV / dK, head-dim row for dQ^T).
#include "bwd_common.cuh"

namespace flamia {
namespace {

constexpr int kQT = 64;          // queries per tile
constexpr int kRing = 4;         // Q / dO ring stages
constexpr int kThreads = 384;
constexpr int kGroupThreads = 128;
constexpr int kD = 128;          // head dim
constexpr uint32_t kColDV = 256, kColDK = 384;
// block-scale columns inside a dP^T half (written after dP^T is read)
constexpr uint32_t kSfDvA = 0, kSfDvB = 4, kSfDkA = 8, kSfDkB = 12, kSfDqA = 16, kSfDqB = 20;

__device__ __forceinline__ uint32_t col_s(int b) { return 64u * b; }
__device__ __forceinline__ uint32_t col_p(int b) { return 128u + 64u * b; }

template <bool TOKS>
struct Bwd128Smem {
  alignas(1024) uint8_t k[kTile * kD];             // [key][dim], 128B-swizzled rows
  alignas(1024) uint8_t v[kTile * kD];
  alignas(1024) uint8_t q[kRing][kQT * kD];        // [query][dim], 128B-swizzled rows
  alignas(1024) uint8_t dout[kRing][kQT * kD];
  alignas(1024) uint8_t pb[2][kTile * kQT];        // [key][query] E4M3, 64B-swizzled rows
  alignas(1024) uint8_t ds[2][kTile * kQT];
  alignas(1024) uint8_t ds2[2][kTile * kQT];      // query-row dS exponents: dQ's dS codes
  alignas(1024) float dqs[2][kD / 32][kQT * 32];   // per group: 4 boxes [query][32 dims]
  // per-query inputs of a group's tile, double-buffered by the group's tile count
  alignas(16) float nl[2][2][kQT];                 // 8 - lse2 (-inf outside the document)
  alignas(16) float dd[2][2][kQT];                 // D (0 outside)
  alignas(16) float pf[2][2][kQT];                 // FP16 dQ: prescale 2^p (0 outside)
  // per-token operand scales (query-row dS instances), per query of a group's
  // tile: 2^eQ, 2^eD (dO), 2^(eD - EdO) (dV's fold), 2^(eQ - EQ) (dK's fold)
  alignas(16) float tq[TOKS ? 4 : 1][2][2][TOKS ? kQT : 4];
  uint32_t qbyte[2][2][2], dobyte[2][2][2];        // [group][buffer][query block]
  uint32_t eds[2][2][4];                           // [group][query block][key block]
  uint8_t erow[2][2][4][32];  // query-row dS bytes [group][query block][key block][query]
  uint64_t bar_kv, bar_kv_free;
  uint64_t bar_qd_full[kRing], bar_qd_empty[kRing];
  uint64_t bar_s_full[2], bar_ds_full[2], bar_dq_full[2], bar_dq_read[2];
  uint64_t bar_acc_full, bar_acc_empty, bar_done;
  ItemRing<4> ring;   // claimed items: producer -> MMA issuer, group leaders
  int item_bc[2][2];  // [group][item parity]: the leader's copy for its group
  int pend[2];        // deterministic dQ: per group, the turn (index into the counters)
                      // its last reduce-adds pass on once complete, or -1
  unsigned long long dscnt[2];  // dS rounded-to-zero diagnostic of this CTA
  uint32_t tmem_base;
  volatile int abort;
};

__device__ __forceinline__ int n_tiles64(const BwdItem& it) { return (it.e - it.qs + kQT - 1) / kQT; }

// Tile v of an item walks the query heads of its K / V head in turn: head
// hk G + v / nt, queries qs + (v % nt) kQT (nt = 64-query tiles per head).
// (G == 1, multi-head attention, needs no division.)
__device__ __forceinline__ int tile_head(const BwdItem& it, int G, int nt, int v) {
  return G == 1 ? it.hk : it.hk * G + v / nt;
}
__device__ __forceinline__ int tile_u(int G, int nt, int v) { return G == 1 ? v : v % nt; }
__device__ __forceinline__ int tile_q0(const BwdItem& it, int G, int nt, int v) {
  return it.qs + tile_u(G, nt, v) * kQT;
}

// DET: the deterministic dQ mode (ordered reduce-adds through prm.dq_turns).
// F16: the prescaled FP16 dQ accumulator (prm.dq_pre), else float32.
// ROWDS: dQ^T's dS operand rounded with one exponent per (query, 32-key block),
// carried as the product's B scales (dK keeps the 32x32 block exponents).
// RD: 0 the 32x32 block dS exponents; 1 query-row exponents for dQ^T's
// operand (ROWDS); 2 per-token operand scales (TOK, with ROWDS).
// CNT: the dS rounded-to-zero diagnostic (prm.ds_count).
template <bool DET, bool F16, int RD, bool CNT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd128_kernel(const __grid_constant__ CUtensorMap map_q,
                       const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_v,
                       const __grid_constant__ CUtensorMap map_do,
                       const __grid_constant__ CUtensorMap map_dq, const BwdParams prm) {
  extern __shared__ uint8_t smem_raw[];
  constexpr bool ROWDS = RD >= 1, TOK = RD == 2;
  Bwd128Smem<TOK>& sm = *reinterpret_cast<Bwd128Smem<TOK>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int T = prm.T;
  const int n_items = min(prm.wl_header[kHdrTileBwd], prm.cap);
  const int total = n_items * prm.Hkv;  // (key tile, K / V head) items
  const int G = prm.G;
  if (static_cast<int>(blockIdx.x) >= total) {  // uniform over the CTA
    if (threadIdx.x == 0) finish_claims(prm.wl_header + kHdrBwdNext, prm.wl_header + kHdrBwdExit);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.bar_kv), 1);
    mbar_init(smem_u32(&sm.bar_kv_free), 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(smem_u32(&sm.bar_qd_full[i]), 1);
      mbar_init(smem_u32(&sm.bar_qd_empty[i]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.bar_s_full[b]), 1);
      mbar_init(smem_u32(&sm.bar_ds_full[b]), kGroupThreads);
      mbar_init(smem_u32(&sm.bar_dq_full[b]), 1);
      mbar_init(smem_u32(&sm.bar_dq_read[b]), kGroupThreads);
    }
    mbar_init(smem_u32(&sm.bar_acc_full), 1);
    mbar_init(smem_u32(&sm.bar_acc_empty), 2 * kGroupThreads);
    mbar_init(smem_u32(&sm.bar_done), 1);
    ring_init(sm.ring, 3);
    sm.abort = 0;
    sm.dscnt[0] = sm.dscnt[1] = 0ull;
    sm.pend[0] = sm.pend[1] = -1;
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
  constexpr uint32_t kKVBytes = 2 * kTile * kD;
  constexpr uint32_t kQDBytes = 2 * kQT * kD;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      prefetch_tensormap(&map_do);
      const uint32_t bkv = smem_u32(&sm.bar_kv);
      int nk = 0, uc = 0;  // items and query tiles loaded (tiles in the consumers' order)
      bool ok = true;
      auto load_qd = [&](int h, int q0) -> bool {
        const int st = uc % kRing;
        if (uc >= kRing &&
            (!mbar_wait(smem_u32(&sm.bar_qd_empty[st]), ((uc / kRing) - 1) & 1) || sm.abort))
          return false;
        const uint32_t bf = smem_u32(&sm.bar_qd_full[st]);
        mbar_arrive_expect_tx(bf, kQDBytes);
        tma_load_3d(smem_u32(sm.q[st]), &map_q, bf, 0, h, q0);
        tma_load_3d(smem_u32(sm.dout[st]), &map_do, bf, 0, h, q0);
        ++uc;
        return true;
      };
      // items in head-major, longest-first order, claimed one at a time: a CTA
      // takes the next item when it has issued its current item's last load
      Claims claims{prm.wl_header + kHdrBwdNext,
                    static_schedule(prm.sched, prm.causal, prm.items, n_items, T, prm.ndocs)};
      int idx = claims.next();
      for (int n = 0; ok; ++n) {
        const bool end = idx >= total;
        if (!ring_put(sm.ring, n, end ? total : idx) || sm.abort) {
          ok = false;
          break;
        }
        if (end) break;
        BwdItem it;
        if (!decode_bwd_item(prm, n_items, idx, it)) {
          idx = claims.next();
          continue;
        }
        const int nt = n_tiles64(it), nq = nt * G;
        const int pre = min(nq, 2);
        int u = 0;
        // the item's first query tiles do not depend on the previous K / V
        for (; u < pre && ok; ++u) ok = load_qd(tile_head(it, G, nt, u), tile_q0(it, G, nt, u));
        if (!ok) break;
        if (nk > 0 && (!mbar_wait(smem_u32(&sm.bar_kv_free), (nk - 1) & 1) || sm.abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bkv, kKVBytes);
        tma_load_3d(smem_u32(sm.k), &map_k, bkv, 0, it.hk, it.k0);
        tma_load_3d(smem_u32(sm.v), &map_v, bkv, 0, it.hk, it.k0);
        ++nk;
        for (; u < nq && ok; ++u) ok = load_qd(tile_head(it, G, nt, u), tile_q0(it, G, nt, u));
        if (ok) idx = claims.next();
      }
      // drain: every issued copy has landed before the CTA exits
      if (nk > 0) ok &= mbar_wait(bkv, (nk - 1) & 1);
      for (int t = max(0, uc - kRing); t < uc; ++t)
        ok &= mbar_wait(smem_u32(&sm.bar_qd_full[t % kRing]), (t / kRing) & 1);
      if (!ok) sm.abort = 1;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this role on warp-uniform values; one elected lane
    // issues each tcgen05 instruction.
    {
      constexpr uint32_t id_s = idesc_f8(kTile, kQT, 0, 0);
      // operand descriptors, built once: a K step or a ring stage moves only
      // the start address (bits 0..13, address / 16), which never carries out
      // of its field inside shared memory
      const uint64_t dk = smem_desc(smem_u32(sm.k), 0, 1024, kLayoutSW128);
      const uint64_t dv = smem_desc(smem_u32(sm.v), 0, 1024, kLayoutSW128);
      const uint64_t dq0 = smem_desc(smem_u32(sm.q[0]), 0, 1024, kLayoutSW128);
      const uint64_t ddo0 = smem_desc(smem_u32(sm.dout[0]), 0, 1024, kLayoutSW128);
      const uint64_t dpb0 = smem_desc(smem_u32(sm.pb[0]), 0, 512, kLayoutSW64);
      const uint64_t dds0 = smem_desc(smem_u32(sm.ds[0]), 0, 512, kLayoutSW64);
      const uint64_t dqs0 = smem_desc(smem_u32(ROWDS ? sm.ds2[0] : sm.ds[0]), 0, 512, kLayoutSW64);
      constexpr uint32_t kQStep = kQT * kD / 16, kPStep = kTile * kQT / 16;  // stage strides
      int nk = 0, ug = 0;
      bool ok = true;
      // S^T_t and dP^T_t into the tensor-memory half of tile t
      auto issue_sdp = [&](int t) -> bool {
        const int st = t % kRing, b = t & 1;
        if (!mbar_wait_w_ab(smem_u32(&sm.bar_qd_full[st]), (t / kRing) & 1, &sm.abort))
          return false;
        // the half's previous tile (t - 2) has had its dQ^T read out
        if (t >= 2 &&
            !mbar_wait_w_ab(smem_u32(&sm.bar_dq_read[b]), ((t >> 1) - 1) & 1, &sm.abort))
          return false;
        tc_fence_after();
        const uint64_t dq = dq0 + st * kQStep, ddo = ddo0 + st * kQStep;
#pragma unroll
        for (int ks = 0; ks < kD / 32; ++ks)
          mma_f8_w(tmem + col_s(b), dk + 2 * ks, dq + 2 * ks, id_s, ks > 0);
#pragma unroll
        for (int ks = 0; ks < kD / 32; ++ks)
          mma_f8_w(tmem + col_p(b), dv + 2 * ks, ddo + 2 * ks, id_s, ks > 0);
        tc_commit_w(smem_u32(&sm.bar_s_full[b]));
        return true;
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
        BwdItem it;
        if (!decode_bwd_item(prm, n_items, idx, it)) continue;
        const int nq = n_tiles64(it) * G;  // tiles over the item's query heads
        ok = mbar_wait_w(smem_u32(&sm.bar_kv), nk & 1) && (nq < 1 || issue_sdp(ug)) &&
             (nq < 2 || issue_sdp(ug + 1));
        for (int u = 0; ok && u < nq; ++u) {
          const int t = ug + u, b = t & 1, st = t % kRing;
          // dV / dK restart from zero on an item's first tile: the previous
          // item's epilogue must have read them
          if (!mbar_wait_w_ab(smem_u32(&sm.bar_ds_full[b]), (t >> 1) & 1, &sm.abort) ||
              (u == 0 && nk > 0 &&
               !mbar_wait_w_ab(smem_u32(&sm.bar_acc_empty), (nk - 1) & 1, &sm.abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dq = dq0 + st * kQStep, ddo = ddo0 + st * kQStep;
          const uint64_t dpb = dpb0 + b * kPStep, dds = dds0 + b * kPStep;
          const uint64_t ddq = dqs0 + b * kPStep;  // dQ^T's dS operand
          const uint32_t sf = tmem + col_p(b);
          // dQ^T_t = K^T dS^T : A = K read MN-major (M = dims), B = dS read MN-major
#pragma unroll
          for (int kb = 0; kb < kTile / 32; ++kb)
            mma_mxf8_w(tmem + col_s(b), dk + kb * (32 * kD / 16), ddq + kb * (32 * kQT / 16),
                     idesc_mxf8(kD, kQT, 1, 1, kb, kb), sf + kSfDqA, sf + kSfDqB, kb > 0);
          // dQ^T first: the group reads it out while dV / dK run
          tc_commit_w(smem_u32(&sm.bar_dq_full[b]));
          // dV += P^b^T dO_t : A [key][query] K-major (64-byte rows), B = dO_t MN-major
#pragma unroll
          for (int kb = 0; kb < kQT / 32; ++kb)
            mma_mxf8_w(tmem + kColDV, dpb + 2 * kb, ddo + kb * (32 * kD / 16),
                     idesc_mxf8(kTile, kD, 0, 1, kb, kb), sf + kSfDvA, sf + kSfDvB,
                     (u > 0 || kb > 0));
          // dK += dS^T Q_t
#pragma unroll
          for (int kb = 0; kb < kQT / 32; ++kb)
            mma_mxf8_w(tmem + kColDK, dds + 2 * kb, dq + kb * (32 * kD / 16),
                     idesc_mxf8(kTile, kD, 0, 1, kb, kb), sf + kSfDkA, sf + kSfDkB,
                     (u > 0 || kb > 0));
          tc_commit_w(smem_u32(&sm.bar_qd_empty[st]));
          if (u + 2 < nq && !issue_sdp(t + 2)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        tc_commit_w(smem_u32(&sm.bar_acc_full));
        tc_commit_w(smem_u32(&sm.bar_kv_free));
        ++nk;
        ug += nq;
      }
      if (!ok) sm.abort = 1;
      tc_commit_w(smem_u32(&sm.bar_done));
      if (!mbar_wait_w(smem_u32(&sm.bar_done), 0)) sm.abort = 1;
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute groups
    const int g = (warp - 4) >> 2;  // tiles t with t & 1 == g
    const int quad = warp & 3;
    const int j = quad * 32 + lane;  // key row (S^T, dP^T, dV, dK) / dim row (dQ^T)
    const bool issuer = (quad == 0 && lane == 0);
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t bar_id = 1 + g;
    const float LOG2E = 1.4426950408889634f;
    // Every thread of the group runs the same sequence of named barriers: a
    // wait that times out only clears `ok`, which skips work, never a barrier.
    bool ok = true;
    int ng = 0, ug = 0, nk = 0;  // this group's tiles, all tiles, items
    // per-query inputs of one tile: raw loads issued a tile ahead (from
    // clamped, always valid addresses) and only used when stored, so their
    // latency hides behind the tile's work
    float r_lse = 0.f, r_dd = 0.f;
    uint32_t r_qb = 127u, r_dob = 127u;
    int r_pre = 0;
    bool r_qv = false;
    constexpr bool tok = TOK;  // per-token operand scales
    uint32_t r_qt = 0u, r_dot = 0u;      // this query's own bytes (per-token scales)
    auto fetch_inputs = [&](size_t hT, int q0, int e) {
      if (quad < 2) {
        const int qi = q0 + j;
        r_qv = qi < e;
        const size_t at = hT + min(qi, T - 1);
        r_lse = prm.lse[at];
        r_dd = prm.D[at];
        if (F16) r_pre = prm.dq_pre[at];
        if (tok) {
          r_qt = prm.q_scales[at];
          r_dot = prm.do_scales[at];
        }
      } else if (lane == 0) {
        const int qi = q0 + 32 * (quad - 2);
        r_qv = qi < e;
        const size_t at = hT + min(qi, T - 1);
        r_qb = prm.q_scales[at];
        r_dob = prm.do_scales[at];
      }
    };
    auto store_inputs = [&](int buf) {
      if (quad < 2) {
        sm.nl[g][buf][j] = r_qv ? 8.f - r_lse * LOG2E : -INFINITY;
        sm.dd[g][buf][j] = r_qv ? r_dd : 0.f;
        if (F16) sm.pf[g][buf][j] = r_qv ? exp2i(r_pre) : 0.f;
        if constexpr (TOK) {
          {
            // this query's factors; its block's (this warp's 32 queries) largest
            // exponents are the B scales of dK and dV
            const int eqb = r_qv ? static_cast<int>(r_qt) : 0;
            const int edb = r_qv ? static_cast<int>(r_dot) : 0;
            const int EQ = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(eqb)));
            const int ED = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(edb)));
            sm.tq[0][g][buf][j] = r_qv ? pow2_or_zero(eqb - 127) : 0.f;
            sm.tq[1][g][buf][j] = r_qv ? pow2_or_zero(edb - 127) : 0.f;
            sm.tq[2][g][buf][j] = r_qv ? pow2_or_zero(edb - ED) : 0.f;
            sm.tq[3][g][buf][j] = r_qv ? pow2_or_zero(eqb - EQ) : 0.f;
            if (lane == 0) {
              sm.qbyte[g][buf][quad] = static_cast<uint32_t>(EQ);
              sm.dobyte[g][buf][quad] = static_cast<uint32_t>(ED);
            }
          }
        }
      } else if (lane == 0 && !tok) {
        sm.qbyte[g][buf][quad - 2] = r_qv ? r_qb : 127u;
        sm.dobyte[g][buf][quad - 2] = r_qv ? r_dob : 127u;
      }
    };
    for (int n = 0;; ++n) {
      if (issuer) sm.item_bc[g][n & 1] = ring_get(sm.ring, n, true);
      named_barrier_sync(bar_id, kGroupThreads);
      const int idx = sm.item_bc[g][n & 1];
      if (idx < 0) {
        ok = false;
        break;
      }
      if (idx >= total) break;
      BwdItem it;
      if (!decode_bwd_item(prm, n_items, idx, it)) continue;
      const int e = it.e, k0 = it.k0, nt = n_tiles64(it), nq = nt * G;
      const size_t hT = static_cast<size_t>(it.hk) * T;  // K / V scale rows
      auto tile_hT = [&](int v) { return static_cast<size_t>(tile_head(it, G, nt, v)) * T; };
      const int kj = k0 + j;
      const bool key_valid = kj < it.k1;
      const int ekj = key_valid ? static_cast<int>(prm.k_scales[hT + kj]) - 127 : 0;
      const int evj = key_valid ? static_cast<int>(prm.v_scales[hT + kj]) - 127 : 0;
      const float rowf = pow2_or_zero(ekj) * prm.scale_log2;
      const float rowg = pow2_or_zero(evj);
      // E8M0 bytes of the tile's 4 key blocks (A scale of dQ^T = K^T dS^T)
      uint32_t kword = 0;
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        const int kk = k0 + 32 * kb;
        kword |= (kk < e ? static_cast<uint32_t>(prm.k_scales[hT + kk]) : 127u) << (8 * kb);
      }
      int u = ((ug & 1) == g) ? 0 : 1;  // this group's first tile of the item
      if (u < nq) {
        fetch_inputs(tile_hT(u), tile_q0(it, G, nt, u), e);
        store_inputs(ng & 1);
      }
      named_barrier_sync(bar_id, kGroupThreads);
      for (; u < nq; u += 2, ++ng) {
        const int tu = tile_u(G, nt, u);  // the tile's place among its head's tiles
        const int q0 = it.qs + tu * kQT, h = tile_head(it, G, nt, u);
        const int buf = ng & 1;
        if (u + 2 < nq) fetch_inputs(tile_hT(u + 2), tile_q0(it, G, nt, u + 2), e);  // lands during this tile
        ok = ok && mbar_wait_ab(smem_u32(&sm.bar_s_full[g]), ng & 1, &sm.abort);
        tc_fence_after();
        uint8_t* pbrow = sm.pb[g] + j * kQT;
        uint8_t* dsrow = sm.ds[g] + j * kQT;
        const int sw = (j >> 1) & 3;  // 64-byte swizzle of row j
#pragma unroll 1
        for (int c = 0; c < 2 && ok; ++c) {
          const float fS = rowf * pow2_or_zero(static_cast<int>(sm.qbyte[g][buf][c]) - 127);
          const float fP = rowg * pow2_or_zero(static_cast<int>(sm.dobyte[g][buf][c]) - 127);
          uint32_t sv[32], dv[32];
          tmem_ld32(tmem + lane_off + col_s(g) + 32 * c, sv);
          tmem_ld32(tmem + lane_off + col_p(g) + 32 * c, dv);
          tmem_ld_wait();
          uint32_t pw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          float amax = 0.f;
          const float* nl = sm.nl[g][buf] + 32 * c;
          const float* dd = sm.dd[g][buf] + 32 * c;
          // per-token operand scales: dK's operand is dS 2^(eQ - EQ) per query
          const float* kq = sm.tq[TOK ? 3 : 0][g][buf] + 32 * c;
          if (!key_valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) dv[i] = 0u;
          } else if (tok) {
            const float* q0p = sm.tq[0][g][buf] + 32 * c;
            const float* d0p = sm.tq[TOK ? 1 : 0][g][buf] + 32 * c;
            const float* p0p = sm.tq[TOK ? 2 : 0][g][buf] + 32 * c;
            if (prm.causal && tu < 2)
              bwd_chunk_tok<true>(sv, dv, nl, dd, q0p, d0p, p0p, rowf, rowg, tu * kQT + 32 * c, j,
                                  pw);
            else
              bwd_chunk_tok<false>(sv, dv, nl, dd, q0p, d0p, p0p, rowf, rowg, 0, j, pw);
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(dv[i]) * kq[i]));
          } else if (prm.causal && tu < 2) {  // the tile crosses the diagonal
            amax = bwd_chunk<true>(sv, dv, nl, dd, fS, fP, tu * kQT + 32 * c, j, pw);
          } else {
            amax = bwd_chunk<false>(sv, dv, nl, dd, fS, fP, u * kQT + 32 * c, j, pw);
          }
          // one exponent per 32x32 block: this warp's 32 key rows x these 32 queries
          // (|dS| >= 0: the float order is the order of the bit patterns)
          amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
          const int eb = max(roundup_exponent(amax) - 8, -127);  // exponent of dS = 2^-8 dS8
          const float inv = exp2i(-(eb + 8));
          const float2 inv2 = make_float2(inv, inv);
          uint32_t dw[8];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float2 a = make_float2(__uint_as_float(dv[i]), __uint_as_float(dv[i + 1]));
            float2 bq = make_float2(__uint_as_float(dv[i + 2]), __uint_as_float(dv[i + 3]));
            if (tok) {
              a = __fmul2_rn(a, make_float2(kq[i], kq[i + 1]));
              bq = __fmul2_rn(bq, make_float2(kq[i + 2], kq[i + 3]));
            }
            a = __fmul2_rn(a, inv2);
            bq = __fmul2_rn(bq, inv2);
            dw[i / 4] = cvt_e4m3x4(a.x, a.y, bq.x, bq.y);
          }
          if (CNT) count_ds_zero(dv, dw, sm.dscnt, lane);
          const int ch0 = (2 * c) ^ sw, ch1 = (2 * c + 1) ^ sw;
          *reinterpret_cast<uint4*>(pbrow + 16 * ch0) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          *reinterpret_cast<uint4*>(pbrow + 16 * ch1) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
          *reinterpret_cast<uint4*>(dsrow + 16 * ch0) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
          *reinterpret_cast<uint4*>(dsrow + 16 * ch1) = make_uint4(dw[4], dw[5], dw[6], dw[7]);
          if (lane == 0) sm.eds[g][c][quad] = static_cast<uint32_t>(eb + 127);
          if (ROWDS) {
            // dQ's operand: per query column the maximum over this warp's 32
            // keys (one key block); lane q keeps query q's and its exponent.
            // Per-token operand scales: the operand is dS 2^eK(j) (K's factor
            // folded in, the key row's own)
            if (tok) {
              const float kf = pow2_or_zero(ekj);
#pragma unroll
              for (int q = 0; q < 32; ++q) dv[q] = __float_as_uint(__uint_as_float(dv[q]) * kf);
            }
            uint32_t mine = 0u;
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              const uint32_t m =
                  __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(__uint_as_float(dv[q]))));
              if (lane == q) mine = m;
            }
            const int er = max(roundup_exponent(__uint_as_float(mine)) - 8, -127);
            const float invr = exp2i(-(er + 8));
            sm.erow[g][c][quad][lane] = static_cast<uint8_t>(er + 127);
            uint32_t dr[8];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float i0 = __shfl_sync(0xffffffffu, invr, i);
              const float i1 = __shfl_sync(0xffffffffu, invr, i + 1);
              const float i2 = __shfl_sync(0xffffffffu, invr, i + 2);
              const float i3 = __shfl_sync(0xffffffffu, invr, i + 3);
              dr[i / 4] = cvt_e4m3x4(__uint_as_float(dv[i]) * i0, __uint_as_float(dv[i + 1]) * i1,
                                     __uint_as_float(dv[i + 2]) * i2,
                                     __uint_as_float(dv[i + 3]) * i3);
            }
            uint8_t* ds2row = sm.ds2[g] + j * kQT;
            *reinterpret_cast<uint4*>(ds2row + 16 * ch0) = make_uint4(dr[0], dr[1], dr[2], dr[3]);
            *reinterpret_cast<uint4*>(ds2row + 16 * ch1) = make_uint4(dr[4], dr[5], dr[6], dr[7]);
          }
        }
        // the group's previous reduce-add has read the staging buffer (and, in
        // the deterministic mode, completed: its turn is passed on)
        if (issuer) {
          if (!DET) {
            bulk_wait_group_read0();
          } else {
            bulk_wait_group0();
            if (sm.pend[g] >= 0) pass_turn(prm.dq_turns + sm.pend[g]);
            sm.pend[g] = -1;
          }
        }
        named_barrier_sync(bar_id, kGroupThreads);
        if (ok) {
          // block scales of the three products (the same words in every lane
          // quadrant: column base + i covers rows 32 i .. 32 i + 31)
          const uint32_t qw = sm.qbyte[g][buf][0] | (sm.qbyte[g][buf][1] << 8) | 0x7F7F0000u;
          const uint32_t dow =
              sm.dobyte[g][buf][0] | (sm.dobyte[g][buf][1] << 8) | 0x7F7F0000u;
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            w[i] = 0x7F7F7F7Fu;  // dV: A = P^b, scale 2^0
            w[4 + i] = dow;      // dV: B = dO_t, per query block
          }
          tmem_st8(tmem + lane_off + col_p(g) + kSfDvA, w);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // dK: A = dS^T, row block = key block i, K blocks = the 2 query blocks
            w[i] = sm.eds[g][0][i] | (sm.eds[g][1][i] << 8) | 0x7F7F0000u;
            w[4 + i] = qw;  // dK: B = Q_t, per query block
          }
          tmem_st8(tmem + lane_off + col_p(g) + kSfDkA, w);
#pragma unroll
          // dQ^T: A = K^T, per key block (2^0: per-token K factors are in dS)
          for (int i = 0; i < 4; ++i) w[i] = tok ? 0x7F7F7F7Fu : kword;
#pragma unroll
          for (int i = 0; i < 2; ++i) {  // dQ^T: B = dS^T, row block = query block i
            if (ROWDS)  // this lane's query 32 i + lane: one byte per key block
              w[4 + i] = static_cast<uint32_t>(sm.erow[g][i][0][lane]) |
                         (static_cast<uint32_t>(sm.erow[g][i][1][lane]) << 8) |
                         (static_cast<uint32_t>(sm.erow[g][i][2][lane]) << 16) |
                         (static_cast<uint32_t>(sm.erow[g][i][3][lane]) << 24);
            else
              w[4 + i] = sm.eds[g][i][0] | (sm.eds[g][i][1] << 8) | (sm.eds[g][i][2] << 16) |
                         (sm.eds[g][i][3] << 24);
          }
          w[6] = w[7] = 0x7F7F7F7Fu;
          tmem_st8(tmem + lane_off + col_p(g) + kSfDqA, w);
          tmem_st_wait();
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.bar_ds_full[g]));
        }
        // the next tile's inputs go to the other buffer (last read by the
        // group's previous tile, before its final barrier)
        if (u + 2 < nq) store_inputs(buf ^ 1);
        ok = ok && mbar_wait_ab(smem_u32(&sm.bar_dq_full[g]), ng & 1, &sm.abort);
        tc_fence_after();
        if (ok) {
          uint32_t v0[32], v1[32];
          tmem_ld32(tmem + lane_off + col_s(g), v0);
          tmem_ld32(tmem + lane_off + col_s(g) + 32, v1);
          tmem_ld_wait();
          // S^T / dP^T of the group's next tile may now be computed
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.bar_dq_read[g]));
          // raw sums of dS K (softmax_scale is applied in the BF16 conversion)
          const int nvalid = min(kQT, e - q0);  // queries of other documents add 0
          float* stg = sm.dqs[g][quad] + lane;  // row = query, element = this dim
          if (F16) {
            // x 2^p of the query (0 outside the document), rounded to FP16, in
            // two boxes [query][64 dims]
            const float4* pf4 = reinterpret_cast<const float4*>(sm.pf[g][buf]);
            __half* st16 = reinterpret_cast<__half*>(sm.dqs[g][0]) + (quad >> 1) * (kQT * 64) +
                           (quad & 1) * 32 + lane;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 fa = pf4[c4], fb = pf4[c4 + 8];  // queries 4 c4 + x, 32 + 4 c4 + x
              const float ma[4] = {fa.x, fa.y, fa.z, fa.w}, mb[4] = {fb.x, fb.y, fb.z, fb.w};
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                const int c = 4 * c4 + x;
                const __half2 h2 = __floats2half2_rn(__uint_as_float(v0[c]) * ma[x],
                                                     __uint_as_float(v1[c]) * mb[x]);
                st16[c * 64] = __low2half(h2);
                st16[(c + 32) * 64] = __high2half(h2);
              }
            }
          } else if (nvalid == kQT) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              stg[c * 32] = __uint_as_float(v0[c]);
              stg[(c + 32) * 32] = __uint_as_float(v1[c]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              stg[c * 32] = c < nvalid ? __uint_as_float(v0[c]) : 0.f;
              stg[(c + 32) * 32] = c + 32 < nvalid ? __uint_as_float(v1[c]) : 0.f;
            }
          }
          fence_proxy_async_smem();
        }
        if (!ok) sm.abort = 1;
        named_barrier_sync(bar_id, kGroupThreads);
        if (issuer && !sm.abort) {
          const int at = q0 * prm.H + h;
          if (DET && !wait_turn(prm.dq_turns + at, dq_turn(prm, it, q0))) {
            sm.abort = 1;
          } else {
            if (F16) {
              const __half* st16 = reinterpret_cast<const __half*>(sm.dqs[g][0]);
#pragma unroll
              for (int b = 0; b < kD / 64; ++b)
                tma_reduce_add_3d(&map_dq, smem_u32(st16 + b * (kQT * 64)), 64 * b, h, q0);
            } else {
#pragma unroll
              for (int c = 0; c < kD / 32; ++c)
                tma_reduce_add_3d(&map_dq, smem_u32(sm.dqs[g][c]), 32 * c, h, q0);
            }
            bulk_commit_group();
            if (DET) sm.pend[g] = at;
          }
        }
      }
      ug += nq;
      if (DET && issuer && sm.pend[g] >= 0) {  // the item's last turn
        bulk_wait_group0();
        pass_turn(prm.dq_turns + sm.pend[g]);
        sm.pend[g] = -1;
      }
      // dV = 2^-8 acc, dK = scale * acc; the groups split the head dimension
      ok = ok && !sm.abort && mbar_wait(smem_u32(&sm.bar_acc_full), nk & 1);
      tc_fence_after();
      if (ok && prm.hadamard) {
        // Q and K were rotated: group 0 writes whole rows of dK = dK_r H_d
        // (the butterflies need all 128 columns of a row), group 1 of dV
        __nv_bfloat16* out =
            (g == 0 ? prm.dk : prm.dv) + (static_cast<size_t>(kj) * prm.Hkv + it.hk) * kD;
        const float mul = g == 0 ? prm.sm_scale : (1.f / 256.f);
        uint32_t u[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + (g == 0 ? kColDK : kColDV) + 32 * c, u[c]);
        tmem_ld_wait();
        float x[kD];
#pragma unroll
        for (int i = 0; i < kD; ++i) x[i] = __uint_as_float(u[i / 32][i % 32]) * mul;
        if (g == 0) fwht_row<kD, 1>(x, 0);
        if (key_valid) {
#pragma unroll
          for (int i = 0; i < kD; i += 8) {
            uint32_t w[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(x[i + 2 * t], x[i + 2 * t + 1]);
              w[t] = *reinterpret_cast<uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(out + i) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.bar_acc_empty));
      } else if (ok) {
        __nv_bfloat16* dvrow = prm.dv + (static_cast<size_t>(kj) * prm.Hkv + it.hk) * kD;
        __nv_bfloat16* dkrow = prm.dk + (static_cast<size_t>(kj) * prm.Hkv + it.hk) * kD;
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const float mul = which == 0 ? (1.f / 256.f) : prm.sm_scale;
          __nv_bfloat16* row = which == 0 ? dvrow : dkrow;
          const uint32_t col = which == 0 ? kColDV : kColDK;
#pragma unroll 1
          for (int c = 2 * g; c < 2 * g + 2; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + col + 32 * c, v);
            tmem_ld_wait();
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * mul,
                                                        __uint_as_float(v[2 * i + 1]) * mul);
              w[i] = *reinterpret_cast<uint32_t*>(&b2);
            }
            if (key_valid) {
              uint4* dst = reinterpret_cast<uint4*>(row + 32 * c);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
              dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
              dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.bar_acc_empty));
      }
      ++nk;
    }
    if (issuer) bulk_wait_group0();
    if (!ok) sm.abort = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (sm.abort) report(prm.status, FLAMIA_DEV_TIMEOUT);
    if (CNT && prm.ds_count != nullptr) {
      atomicAdd(prm.ds_count, sm.dscnt[0]);
      atomicAdd(prm.ds_count + 1, sm.dscnt[1]);
    }
    finish_claims(prm.wl_header + kHdrBwdNext, prm.wl_header + kHdrBwdExit);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_bwd128_pipelined(const BwdParams& prm, const flamia_qtensor* q,
                                    const flamia_qtensor* k, const flamia_qtensor* v,
                                    const flamia_qtensor* dout, float* acc, unsigned grid,
                                    cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mdo, mdq;
  const int T = prm.T, H = prm.H;
  if (!make_token_map(&mq, q->codes, T, H, kD, kQT, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_token_map(&mk, k->codes, T, prm.Hkv, kD, kTile, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_token_map(&mv, v->codes, T, prm.Hkv, kD, kTile, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_token_map(&mdo, dout->codes, T, H, kD, kQT, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const bool f16 = prm.dq_pre != nullptr, det = prm.dq_turns != nullptr;
  if (f16 ? !make_f16_token_map(&mdq, acc, T, H, kD, kQT, CU_TENSOR_MAP_SWIZZLE_NONE)
          : !make_f32_token_map(&mdq, acc, T, H, kD, kQT, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const int rd = prm.token ? 2 : prm.ds_rows ? 1 : 0;
  const bool cnt = prm.ds_count != nullptr;
  const size_t smem = (rd == 2 ? sizeof(Bwd128Smem<true>) : sizeof(Bwd128Smem<false>)) + 1024;
  using Kernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                         const BwdParams);
  // [rd][f16][det]; the diagnostic count only with the float32, unordered dQ sum
  static const Kernel kernels[3][2][2] = {
      {{attn_bwd128_kernel<false, false, 0, false>, attn_bwd128_kernel<true, false, 0, false>},
       {attn_bwd128_kernel<false, true, 0, false>, attn_bwd128_kernel<true, true, 0, false>}},
      {{attn_bwd128_kernel<false, false, 1, false>, attn_bwd128_kernel<true, false, 1, false>},
       {attn_bwd128_kernel<false, true, 1, false>, attn_bwd128_kernel<true, true, 1, false>}},
      {{attn_bwd128_kernel<false, false, 2, false>, attn_bwd128_kernel<true, false, 2, false>},
       {attn_bwd128_kernel<false, true, 2, false>, attn_bwd128_kernel<true, true, 2, false>}}};
  static const Kernel counting[3] = {attn_bwd128_kernel<false, false, 0, true>,
                                     attn_bwd128_kernel<false, false, 1, true>,
                                     attn_bwd128_kernel<false, false, 2, true>};
  if (cnt && (det || f16)) return cudaErrorInvalidValue;
  const Kernel kernel = cnt ? counting[rd] : kernels[rd][f16 ? 1 : 0][det ? 1 : 0];
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  kernel<<<grid, kThreads, smem, stream>>>(mq, mk, mv, mdo, mdq, prm);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace flamia
