// Causal backward for head dim 128 on CTA pairs (FLAMIA review page, sec.
// 3.4 "Backward pass": the 2-CTA mode, a cluster of two CTAs that splits 256
// keys; the choice between it and the one-CTA kernel is a rule by shape).
//
// One work item = one 256-key tile of a document x one K / V head.  CTA r of
// the pair holds keys k0 + 128 r .. k0 + 128 r + 127; the pair walks the
// item's 64-query tiles from k0's diagonal together, and as in the one-CTA
// kernel the two compute groups of each CTA take alternate tiles with their
// own halves of tensor memory.  Every product is one product of the pair
// (tcgen05 .cta_group::2, issued by the even CTA): A and D are split by rows,
// each CTA holding its own 128; B is split by columns, each CTA supplying
// half of them from the same shared-memory address:
//
//   S^T_t = K Q_t^T, dP^T_t = V dO_t^T  M 256 (keys), N 64: CTA r supplies
//                                       the queries 32 r .. 32 r + 31
//   dV += P^b_t^T dO_t, dK += dS_t^T Q_t  M 256 (keys), N 128: CTA r supplies
//                                       the head dims 64 r .. 64 r + 63
//   dQ_t^T = K^T dS_t^T                 M 256, N 64, K = the pair's 256 keys
//
// In the dQ^T product each CTA's A is the K of both CTAs (its own keys
// first) and the B it supplies is dS^T of its 32 queries over the same 256
// keys in the same order (its own rows written by itself, the other CTA's
// rows copied there from the other CTA's shared memory); so the 32 columns a
// CTA supplied hold dQ^T of its queries over all 256 keys (the other 32
// columns mix the two orders and are never read).  Each CTA reads out and
// reduce-adds dQ of its own 32 queries: one reduce-add per element and pair
// tile where two one-CTA items would make two.
//
// Block scales live in each CTA's own tensor memory: A's for its own rows
// (column base + row / 32), B's for all N columns (each tensor core forms all
// N columns of its rows).  The 32 x 32 dS exponents of dQ^T's B come from
// both CTAs: each sends the other its exponents for the other's 32 queries.
// The other CTA's dS rows and exponents are written to a local staging buffer
// and sent with one bulk copy per tile, which completes on the receiving
// CTA's barrier: no generic-proxy writes cross the CTAs.
//
// Warp roles: warp 0 lane 0 the producer (the even CTA claims items and hands
// each to the odd CTA through a mailbox in the odd CTA's shared memory; each
// CTA loads its own halves of the operands); warp 1 the MMA issuer (even CTA)
// or the relay that reports the odd CTA's completed loads to it; warps 4-11
// the two compute groups (thread = key row of S^T / dP^T / dV / dK, head-dim
// row of dQ^T).
#include "bwd_common.cuh"

namespace flamia {
namespace {

constexpr int kQT = 64;          // queries per tile
constexpr int kQH = 32;          // queries per tile supplied (and reduced) by one CTA
constexpr int kRing = 4;         // Q / dO ring stages
constexpr int kThreads = 384;
constexpr int kGroupThreads = 128;
constexpr int kD = 128;          // head dim
constexpr uint32_t kColDV = 256, kColDK = 384;
// block-scale columns inside a dP^T half (written after dP^T is read):
// dV A / B, dK A / B (4 columns each), dQ^T A (two words x 4 columns), dQ^T B
// (two words x 2 columns)
constexpr uint32_t kSfDvA = 0, kSfDvB = 4, kSfDkA = 8, kSfDkB = 12, kSfDqA = 16, kSfDqB = 24;

__device__ __forceinline__ uint32_t col_s(int b) { return 64u * b; }
__device__ __forceinline__ uint32_t col_p(int b) { return 128u + 64u * b; }

struct PairSmem {
  alignas(1024) uint8_t k[2 * kTile * kD];         // [key][dim], own keys then the other CTA's
  alignas(1024) uint8_t v[kTile * kD];             // own keys
  alignas(1024) uint8_t qh[kRing][kQH * kD];       // this CTA's 32 queries [query][dim]
  alignas(1024) uint8_t doh[kRing][kQH * kD];
  alignas(1024) uint8_t qd[kRing][kQT * 64];       // all 64 queries x this CTA's 64 dims
  alignas(1024) uint8_t dod[kRing][kQT * 64];
  alignas(1024) uint8_t pb[2][kTile * kQT];        // [key][query] E4M3, 64B-swizzled rows
  alignas(1024) uint8_t ds[2][kTile * kQT];
  alignas(1024) uint8_t dsq[2][2 * kTile * kQH];   // [key][this CTA's 32 queries], 32B-swizzled,
                                                   // own keys then the other CTA's
  alignas(1024) float dqs[2][kD / 32][kQH * 32];   // per group: 4 boxes [query][32 dims]
  alignas(16) float nl[2][2][kQT];                 // 8 - lse2 (-inf outside the document)
  alignas(16) float dd[2][2][kQT];                 // D (0 outside)
  uint32_t qbyte[2][2][2], dobyte[2][2][2];        // [group][buffer][query block]
  uint32_t eds[2][2][4];                           // [group][query block][own key block]
  alignas(256) uint8_t xs[2][kTile * kQH];        // staging of the other CTA's rows (its layout)
  alignas(16) uint32_t xe[2][4];                   // staging of this CTA's exponents for its queries
  alignas(16) uint32_t eds_peer[2][4];  // [group][other CTA's key block]: its exponents, this CTA's queries
  uint64_t bar_kv, bar_kv_peer, bar_kv_free;
  uint64_t bar_qd_full[kRing], bar_qd_peer[kRing], bar_qd_empty[kRing];
  uint64_t bar_s_full[2], bar_ds_full[2], bar_dq_full[2], bar_dq_read[2], bar_eds[2];
  uint64_t bar_acc_full, bar_acc_empty, bar_done;
  uint64_t mbox_full[4], mbox_empty[4];
  int mbox[4];
  ItemRing<4> ring;   // claimed items: producer -> MMA issuer / relay, group leaders
  int item_bc[2][2];  // [group][item parity]: the leader's copy for its group
  uint32_t tmem_base;
  volatile int abort;
};

__device__ __forceinline__ int n_tiles64(const BwdItem& it) { return (it.e - it.qs + kQT - 1) / kQT; }
__device__ __forceinline__ int tile_head(const BwdItem& it, int G, int nt, int v) {
  return G == 1 ? it.hk : it.hk * G + v / nt;
}
__device__ __forceinline__ int tile_u(int G, int nt, int v) { return G == 1 ? v : v % nt; }
__device__ __forceinline__ int tile_q0(const BwdItem& it, int G, int nt, int v) {
  return it.qs + tile_u(G, nt, v) * kQT;
}
// Pair items are the list's key tiles at even positions of their document
// (the list is sorted by cost, so they stay sorted); short documents are the
// CUDA-core kernel's.
__device__ __forceinline__ bool pair_item(const BwdParams& prm, int n_items, int idx) {
  BwdItem it;
  return decode_bwd_item(prm, n_items, idx, it) && (((it.k0 - it.s) / kTile) & 1) == 0;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_bwd_pair_kernel(const __grid_constant__ CUtensorMap map_qh,
                         const __grid_constant__ CUtensorMap map_doh,
                         const __grid_constant__ CUtensorMap map_qd,
                         const __grid_constant__ CUtensorMap map_dod,
                         const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v,
                         const __grid_constant__ CUtensorMap map_dq, const BwdParams prm) {
  extern __shared__ uint8_t smem_raw[];
  PairSmem& sm = *reinterpret_cast<PairSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int T = prm.T;
  const int n_items = min(prm.wl_header[kHdrTileBwd], prm.cap);
  const int total = n_items * prm.Hkv;  // (key tile, K / V head) entries of the list
  const int G = prm.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.bar_kv), 1);
    mbar_init(smem_u32(&sm.bar_kv_peer), 1);
    mbar_init(smem_u32(&sm.bar_kv_free), 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(smem_u32(&sm.bar_qd_full[i]), 1);
      mbar_init(smem_u32(&sm.bar_qd_peer[i]), 1);
      mbar_init(smem_u32(&sm.bar_qd_empty[i]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.bar_s_full[b]), 1);
      mbar_init(smem_u32(&sm.bar_ds_full[b]), 8);  // 4 warps of each CTA's group
      mbar_init(smem_u32(&sm.bar_dq_full[b]), 1);
      mbar_init(smem_u32(&sm.bar_dq_read[b]), 8);
      mbar_init(smem_u32(&sm.bar_eds[b]), 1);      // own expect_tx + the other CTA's copy
    }
    mbar_init(smem_u32(&sm.bar_acc_full), 1);
    mbar_init(smem_u32(&sm.bar_acc_empty), 16);    // 8 compute warps of each CTA
    mbar_init(smem_u32(&sm.bar_done), 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(smem_u32(&sm.mbox_full[i]), 1);
      mbar_init(smem_u32(&sm.mbox_empty[i]), 1);
    }
    ring_init(sm.ring, 3);
    sm.abort = 0;
    fence_barrier_init();
  }
  cluster_sync_all();  // barriers initialised before the other CTA arrives on them
  if (warp == 1) {
    tmem_alloc2(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // the same location in the issuing (even) CTA, and in the other CTA
  auto at_leader = [&](const void* p) { return mapa_shared(smem_u32(p), 0); };
  auto at_peer = [&](const void* p) { return mapa_shared(smem_u32(p), peer); };
  // a failed wait stops both CTAs (their waits on each other then give up)
  auto abort_pair = [&]() {
    sm.abort = 1;
    st_cluster_u32(at_peer(const_cast<int*>(&sm.abort)), 1u);
  };
  constexpr uint32_t kKVBytes = 3 * kTile * kD;
  constexpr uint32_t kQDBytes = 2 * kQH * kD + 2 * kQT * 64;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&map_qh);
      prefetch_tensormap(&map_doh);
      prefetch_tensormap(&map_qd);
      prefetch_tensormap(&map_dod);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      const uint32_t bkv = smem_u32(&sm.bar_kv);
      int nk = 0, uc = 0;
      bool ok = true;
      auto load_qd = [&](int h, int q0) -> bool {
        const int st = uc % kRing;
        if (uc >= kRing &&
            (!mbar_wait(smem_u32(&sm.bar_qd_empty[st]), ((uc / kRing) - 1) & 1) || sm.abort))
          return false;
        const uint32_t bf = smem_u32(&sm.bar_qd_full[st]);
        mbar_arrive_expect_tx(bf, kQDBytes);
        tma_load_3d(smem_u32(sm.qh[st]), &map_qh, bf, 0, h, q0 + kQH * static_cast<int>(rank));
        tma_load_3d(smem_u32(sm.doh[st]), &map_doh, bf, 0, h, q0 + kQH * static_cast<int>(rank));
        tma_load_3d(smem_u32(sm.qd[st]), &map_qd, bf, 64 * static_cast<int>(rank), h, q0);
        tma_load_3d(smem_u32(sm.dod[st]), &map_dod, bf, 64 * static_cast<int>(rank), h, q0);
        ++uc;
        return true;
      };
      Claims claims{prm.wl_header + kHdrBwdNext, false};
      auto next_item = [&]() {
        int i = claims.next();
        while (i < total && !pair_item(prm, n_items, i)) i = claims.next();
        return i;
      };
      int idx = rank == 0 ? next_item() : 0;
      for (int n = 0; ok; ++n) {
        const int slot = n & 3;
        if (rank == 0) {
          // hand item n to the odd CTA
          if (n >= 4 && (!mbar_wait_cl(smem_u32(&sm.mbox_empty[slot]), ((n >> 2) - 1) & 1) ||
                         sm.abort)) {
            ok = false;
            break;
          }
          if (idx > total) idx = total;
          st_cluster_u32(at_peer(&sm.mbox[slot]), static_cast<uint32_t>(idx));
          mbar_arrive_cluster(at_peer(&sm.mbox_full[slot]));
        } else {
          if (!mbar_wait_cl(smem_u32(&sm.mbox_full[slot]), (n >> 2) & 1) || sm.abort) {
            ok = false;
            break;
          }
          idx = *reinterpret_cast<volatile int*>(&sm.mbox[slot]);
          mbar_arrive_cluster(at_leader(&sm.mbox_empty[slot]));
        }
        const bool end = idx >= total;
        if (!ring_put(sm.ring, n, end ? total : idx) || sm.abort) {
          ok = false;
          break;
        }
        if (end) break;
        BwdItem it;
        if (!decode_bwd_item(prm, n_items, idx, it)) {
          if (rank == 0) idx = next_item();
          continue;
        }
        const int nt = n_tiles64(it), nq = nt * G;
        const int pre = min(nq, 2);
        int u = 0;
        for (; u < pre && ok; ++u) ok = load_qd(tile_head(it, G, nt, u), tile_q0(it, G, nt, u));
        if (!ok) break;
        if (nk > 0 && (!mbar_wait(smem_u32(&sm.bar_kv_free), (nk - 1) & 1) || sm.abort)) {
          ok = false;
          break;
        }
        const int kown = it.k0 + kTile * static_cast<int>(rank);
        const int koth = it.k0 + kTile * static_cast<int>(peer);
        mbar_arrive_expect_tx(bkv, kKVBytes);
        tma_load_3d(smem_u32(sm.k), &map_k, bkv, 0, it.hk, kown);
        tma_load_3d(smem_u32(sm.k + kTile * kD), &map_k, bkv, 0, it.hk, koth);
        tma_load_3d(smem_u32(sm.v), &map_v, bkv, 0, it.hk, kown);
        ++nk;
        for (; u < nq && ok; ++u) ok = load_qd(tile_head(it, G, nt, u), tile_q0(it, G, nt, u));
        if (ok && rank == 0) idx = next_item();
      }
      // drain: every issued copy has landed before the CTA exits
      if (nk > 0) ok &= mbar_wait(bkv, (nk - 1) & 1);
      for (int t = max(0, uc - kRing); t < uc; ++t)
        ok &= mbar_wait(smem_u32(&sm.bar_qd_full[t % kRing]), (t / kRing) & 1);
      if (!ok) abort_pair();
    }
  } else if (warp == 1 && rank == 1) {
    // ------------------------------------------------------------ relay (odd CTA)
    // The even CTA's issuer may start a product only when this CTA's halves
    // of its operands have landed: report each completed load there.
    int nk = 0, ug = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
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
      const int nq = n_tiles64(it) * G;
      // in the order the issuer waits: the item's K / V, then its tiles
      ok = mbar_wait_w(smem_u32(&sm.bar_kv), nk & 1) && !__any_sync(0xffffffffu, sm.abort);
      if (ok && lane == 0) mbar_arrive_cluster(at_leader(&sm.bar_kv_peer));
      for (int u = 0; ok && u < nq; ++u) {
        const int t = ug + u, st = t % kRing;
        ok = mbar_wait_w(smem_u32(&sm.bar_qd_full[st]), (t / kRing) & 1) &&
             !__any_sync(0xffffffffu, sm.abort);
        if (ok && lane == 0) mbar_arrive_cluster(at_leader(&sm.bar_qd_peer[st]));
      }
      ++nk;
      ug += nq;
    }
    if (!ok && lane == 0) abort_pair();
    // every product of the pair has completed before the tensor memory is freed
    if (!mbar_wait_w(smem_u32(&sm.bar_done), 0) && lane == 0) abort_pair();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    {
      constexpr uint32_t id_s = idesc_f8(2 * kTile, kQT, 0, 0);
      const uint64_t dk = smem_desc(smem_u32(sm.k), 0, 1024, kLayoutSW128);
      const uint64_t dv = smem_desc(smem_u32(sm.v), 0, 1024, kLayoutSW128);
      const uint64_t dqh0 = smem_desc(smem_u32(sm.qh[0]), 0, 1024, kLayoutSW128);
      const uint64_t ddoh0 = smem_desc(smem_u32(sm.doh[0]), 0, 1024, kLayoutSW128);
      const uint64_t dqd0 = smem_desc(smem_u32(sm.qd[0]), 0, 512, kLayoutSW64);
      const uint64_t ddod0 = smem_desc(smem_u32(sm.dod[0]), 0, 512, kLayoutSW64);
      const uint64_t dpb0 = smem_desc(smem_u32(sm.pb[0]), 0, 512, kLayoutSW64);
      const uint64_t dds0 = smem_desc(smem_u32(sm.ds[0]), 0, 512, kLayoutSW64);
      const uint64_t ddsq0 = smem_desc(smem_u32(sm.dsq[0]), 0, 256, kLayoutSW32);
      constexpr uint32_t kHStep = kQH * kD / 16, kDStep = kQT * 64 / 16;  // ring stage strides
      constexpr uint32_t kPStep = kTile * kQT / 16, kSqStep = 2 * kTile * kQH / 16;
      int nk = 0, ug = 0;
      bool ok = true;
      // S^T_t and dP^T_t into the tensor-memory half of tile t, once both
      // CTAs' halves of Q_t / dO_t have landed (the odd CTA's phases, arrived
      // from there with cluster-scope release, are waited at cluster scope)
      auto issue_sdp = [&](int t) -> bool {
        const int st = t % kRing, b = t & 1;
        if (!mbar_wait_w(smem_u32(&sm.bar_qd_full[st]), (t / kRing) & 1) ||
            !mbar_wait_cl_w(smem_u32(&sm.bar_qd_peer[st]), (t / kRing) & 1))
          return false;
        // the half's previous tile (t - 2) has had its dQ^T read out in both CTAs
        if (t >= 2 && !mbar_wait_cl_w(smem_u32(&sm.bar_dq_read[b]), ((t >> 1) - 1) & 1))
          return false;
        if (__any_sync(0xffffffffu, sm.abort)) return false;
        tc_fence_after();
        const uint64_t dq = dqh0 + st * kHStep, ddo = ddoh0 + st * kHStep;
#pragma unroll
        for (int ks = 0; ks < kD / 32; ++ks)
          mma2_f8_w(tmem + col_s(b), dk + 2 * ks, dq + 2 * ks, id_s, ks > 0);
#pragma unroll
        for (int ks = 0; ks < kD / 32; ++ks)
          mma2_f8_w(tmem + col_p(b), dv + 2 * ks, ddo + 2 * ks, id_s, ks > 0);
        tc_commit2_w(smem_u32(&sm.bar_s_full[b]), 3);
        return true;
      };
      for (int n = 0; ok; ++n) {
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
        const int nq = n_tiles64(it) * G;
        ok = mbar_wait_w(smem_u32(&sm.bar_kv), nk & 1) &&
             mbar_wait_cl_w(smem_u32(&sm.bar_kv_peer), nk & 1) && (nq < 1 || issue_sdp(ug)) &&
             (nq < 2 || issue_sdp(ug + 1));
        for (int u = 0; ok && u < nq; ++u) {
          const int t = ug + u, b = t & 1, st = t % kRing;
          // dV / dK restart from zero on an item's first tile: the previous
          // item's epilogue (both CTAs) must have read them
          if (!mbar_wait_cl_w(smem_u32(&sm.bar_ds_full[b]), (t >> 1) & 1) ||
              (u == 0 && nk > 0 && !mbar_wait_cl_w(smem_u32(&sm.bar_acc_empty), (nk - 1) & 1)) ||
              __any_sync(0xffffffffu, sm.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dqd = dqd0 + st * kDStep, ddod = ddod0 + st * kDStep;
          const uint64_t dpb = dpb0 + b * kPStep, dds = dds0 + b * kPStep;
          const uint64_t dsq = ddsq0 + b * kSqStep;
          const uint32_t sf = tmem + col_p(b);
          // dQ^T_t = K^T dS^T over the pair's 256 keys: A = K read MN-major
          // (M = dims), B = dS^T of this CTA's queries read MN-major
#pragma unroll
          for (int kb = 0; kb < 2 * kTile / 32; ++kb)
            mma2_mxf8_w(tmem + col_s(b), dk + kb * (32 * kD / 16), dsq + kb * (32 * kQH / 16),
                        idesc_mxf8(2 * kTile, kQT, 1, 1, kb & 3, kb & 3),
                        sf + kSfDqA + 4 * (kb >> 2), sf + kSfDqB + 2 * (kb >> 2), kb > 0);
          tc_commit2_w(smem_u32(&sm.bar_dq_full[b]), 3);
          // dV += P^b^T dO_t : A [key][query] K-major, B = dO_t's dims MN-major
#pragma unroll
          for (int kb = 0; kb < kQT / 32; ++kb)
            mma2_mxf8_w(tmem + kColDV, dpb + 2 * kb, ddod + kb * (32 * 64 / 16),
                        idesc_mxf8(2 * kTile, kD, 0, 1, kb, kb), sf + kSfDvA, sf + kSfDvB,
                        (u > 0 || kb > 0));
          // dK += dS^T Q_t
#pragma unroll
          for (int kb = 0; kb < kQT / 32; ++kb)
            mma2_mxf8_w(tmem + kColDK, dds + 2 * kb, dqd + kb * (32 * 64 / 16),
                        idesc_mxf8(2 * kTile, kD, 0, 1, kb, kb), sf + kSfDkA, sf + kSfDkB,
                        (u > 0 || kb > 0));
          tc_commit2_w(smem_u32(&sm.bar_qd_empty[st]), 3);
          if (u + 2 < nq && !issue_sdp(t + 2)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        tc_commit2_w(smem_u32(&sm.bar_acc_full), 3);
        tc_commit2_w(smem_u32(&sm.bar_kv_free), 3);
        ++nk;
        ug += nq;
      }
      if (!ok && lane == 0) abort_pair();
      tc_commit2_w(smem_u32(&sm.bar_done), 3);
      if (!mbar_wait_w(smem_u32(&sm.bar_done), 0) && lane == 0) abort_pair();
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute groups
    const int g = (warp - 4) >> 2;  // tiles t with t & 1 == g
    const int quad = warp & 3;
    const int j = quad * 32 + lane;  // own key row (S^T, dP^T, dV, dK) / dim row (dQ^T)
    const bool issuer = (quad == 0 && lane == 0);
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t bar_id = 1 + g;
    const int r = static_cast<int>(rank);
    const float LOG2E = 1.4426950408889634f;
    bool ok = true;
    int ng = 0, ug = 0, nk = 0;
    float r_lse = 0.f, r_dd = 0.f;
    uint32_t r_qb = 127u, r_dob = 127u;
    bool r_qv = false;
    auto fetch_inputs = [&](size_t hT, int q0, int e) {
      if (quad < 2) {
        const int qi = q0 + j;
        r_qv = qi < e;
        const size_t at = hT + min(qi, T - 1);
        r_lse = prm.lse[at];
        r_dd = prm.D[at];
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
      } else if (lane == 0) {
        sm.qbyte[g][buf][quad - 2] = r_qv ? r_qb : 127u;
        sm.dobyte[g][buf][quad - 2] = r_qv ? r_dob : 127u;
      }
    };
    // one arrive per warp, on the even CTA's barrier, after the warp's writes
    // (cluster scope from the odd CTA only)
    auto warp_arrive_leader = [&](uint64_t* bar) {
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(smem_u32(bar));
        else mbar_arrive_cluster(at_leader(bar));
      }
    };
    // `ok` stays uniform over each warp (the tensor-memory accesses and the
    // arrives are warp-wide): every wait (which gives up once the abort flag
    // is set) is decided for the whole warp.  These phases are completed by the tensor core (pair
    // commits) or by the other CTA's bulk copy: CTA-scope waits
    auto wait_w = [&](uint64_t* bar, int parity) {
      ok = __all_sync(0xffffffffu, ok) && mbar_wait_w_ab(smem_u32(bar), parity, &sm.abort);
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
      const int e = it.e, nt = n_tiles64(it), nq = nt * G;
      const int k1 = min(it.k0 + 2 * kTile, e);  // the pair's keys end here
      const int kbase = it.k0 + kTile * r;        // this CTA's first key
      const size_t hT = static_cast<size_t>(it.hk) * T;
      auto tile_hT = [&](int v) { return static_cast<size_t>(tile_head(it, G, nt, v)) * T; };
      const int kj = kbase + j;
      const bool key_valid = kj < k1;
      const int ekj = key_valid ? static_cast<int>(prm.k_scales[hT + kj]) - 127 : 0;
      const int evj = key_valid ? static_cast<int>(prm.v_scales[hT + kj]) - 127 : 0;
      const float rowf = pow2_or_zero(ekj) * prm.scale_log2;
      const float rowg = pow2_or_zero(evj);
      // E8M0 bytes of the key blocks (dQ^T's A scales): own blocks, then the other CTA's
      uint32_t kword[2] = {0u, 0u};
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          const int kk = it.k0 + kTile * (h == 0 ? r : 1 - r) + 32 * kb;
          kword[h] |= (kk < k1 ? static_cast<uint32_t>(prm.k_scales[hT + kk]) : 127u) << (8 * kb);
        }
      int u = ((ug & 1) == g) ? 0 : 1;  // this group's first tile of the item
      if (u < nq) {
        fetch_inputs(tile_hT(u), tile_q0(it, G, nt, u), e);
        store_inputs(ng & 1);
      }
      named_barrier_sync(bar_id, kGroupThreads);
      for (; u < nq; u += 2, ++ng) {
        const int tu = tile_u(G, nt, u);
        const int q0 = it.qs + tu * kQT, h = tile_head(it, G, nt, u);
        const int buf = ng & 1;
        if (u + 2 < nq) fetch_inputs(tile_hT(u + 2), tile_q0(it, G, nt, u + 2), e);
        // this tile's rows and exponents from the other CTA arrive as one copy
        if (issuer) mbar_arrive_expect_tx(smem_u32(&sm.bar_eds[g]), kTile * kQH + 16);
        wait_w(&sm.bar_s_full[g], ng & 1);
        tc_fence_after();
        uint8_t* pbrow = sm.pb[g] + j * kQT;
        uint8_t* dsrow = sm.ds[g] + j * kQT;
        const int sw = (j >> 1) & 3;  // 64-byte swizzle of row j
        // the tile crosses or lies below this CTA's diagonal (keys 128 r + j)
        const bool masked = prm.causal && tu < 2 + 2 * r;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          // the other CTA's query block first: its rows and exponents travel
          // while this CTA computes its own block
          const int c = cc ^ (1 - r);
          if (ok) {
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
          if (!key_valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) dv[i] = 0u;
          } else if (masked) {
            amax = bwd_chunk<true>(sv, dv, nl, dd, fS, fP, tu * kQT + 32 * c, kTile * r + j, pw);
          } else {
            amax = bwd_chunk<false>(sv, dv, nl, dd, fS, fP, 0, 0, pw);
          }
          amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
          const int eb = max(roundup_exponent(amax) - 8, -127);
          const float inv = exp2i(-(eb + 8));
          const float2 inv2 = make_float2(inv, inv);
          uint32_t dw[8];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float2 a = __fmul2_rn(make_float2(__uint_as_float(dv[i]), __uint_as_float(dv[i + 1])), inv2);
            const float2 bq =
                __fmul2_rn(make_float2(__uint_as_float(dv[i + 2]), __uint_as_float(dv[i + 3])), inv2);
            dw[i / 4] = cvt_e4m3x4(a.x, a.y, bq.x, bq.y);
          }
          const int ch0 = (2 * c) ^ sw, ch1 = (2 * c + 1) ^ sw;
          *reinterpret_cast<uint4*>(pbrow + 16 * ch0) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          *reinterpret_cast<uint4*>(pbrow + 16 * ch1) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
          *reinterpret_cast<uint4*>(dsrow + 16 * ch0) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
          *reinterpret_cast<uint4*>(dsrow + 16 * ch1) = make_uint4(dw[4], dw[5], dw[6], dw[7]);
          // dQ^T's operand: the same codes in query block c's CTA, row j there
          // for its own keys, 128 + j for the other's (32-byte swizzle; the
          // staging buffer holds the other CTA's rows 128 .. 255 in its layout)
          const int s32 = (j >> 2) & 1;
          uint8_t* qrow = c == r ? sm.dsq[g] + j * kQH : sm.xs[g] + j * kQH;
          *reinterpret_cast<uint4*>(qrow + 16 * s32) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
          *reinterpret_cast<uint4*>(qrow + 16 * (1 ^ s32)) = make_uint4(dw[4], dw[5], dw[6], dw[7]);
          if (lane == 0) {
            sm.eds[g][c][quad] = static_cast<uint32_t>(eb + 127);
            if (c != r) sm.xe[g][quad] = static_cast<uint32_t>(eb + 127);
          }
          }
          if (cc == 0) {
            // the other CTA's rows 128 .. 255 of its dQ^T operand and the
            // exponents of its query block are staged: one copy sends them
            fence_proxy_async_smem();
            named_barrier_sync(bar_id, kGroupThreads);
            if (issuer && ok) {
              bulk_copy_to_cluster(at_peer(sm.dsq[g] + kTile * kQH), smem_u32(sm.xs[g]),
                                   kTile * kQH, at_peer(&sm.bar_eds[g]));
              bulk_copy_to_cluster(at_peer(sm.eds_peer[g]), smem_u32(sm.xe[g]), 16,
                                   at_peer(&sm.bar_eds[g]));
            }
          }
        }
        fence_proxy_async_smem();
        // the group's previous reduce-add has read the staging buffer
        if (issuer) bulk_wait_group_read0();
        named_barrier_sync(bar_id, kGroupThreads);
        // the other CTA's copy to this one
        wait_w(&sm.bar_eds[g], ng & 1);
        if (ok) {
          const uint32_t qw = sm.qbyte[g][buf][0] | (sm.qbyte[g][buf][1] << 8) | 0x7F7F0000u;
          const uint32_t dow =
              sm.dobyte[g][buf][0] | (sm.dobyte[g][buf][1] << 8) | 0x7F7F0000u;
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            w[i] = 0x7F7F7F7Fu;  // dV: A = P^b, scale 2^0
            w[4 + i] = dow;      // dV: B = dO_t, per query block, every column
          }
          tmem_st8(tmem + lane_off + col_p(g) + kSfDvA, w);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // dK: A = dS^T, row block = own key block i, K blocks = the 2 query blocks
            w[i] = sm.eds[g][0][i] | (sm.eds[g][1][i] << 8) | 0x7F7F0000u;
            w[4 + i] = qw;
          }
          tmem_st8(tmem + lane_off + col_p(g) + kSfDkA, w);
          // dQ^T: A = K^T per key block (own four, then the other CTA's), every
          // row; B = dS^T of this CTA's query block per key block, every column
          const uint32_t bw0 = sm.eds[g][r][0] | (sm.eds[g][r][1] << 8) |
                               (sm.eds[g][r][2] << 16) | (sm.eds[g][r][3] << 24);
          const uint32_t bw1 = sm.eds_peer[g][0] | (sm.eds_peer[g][1] << 8) |
                               (sm.eds_peer[g][2] << 16) | (sm.eds_peer[g][3] << 24);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            w[i] = kword[0];
            w[4 + i] = kword[1];
          }
          tmem_st8(tmem + lane_off + col_p(g) + kSfDqA, w);
          uint32_t w4[4] = {bw0, bw0, bw1, bw1};
          tmem_st4(tmem + lane_off + col_p(g) + kSfDqB, w4);
          tmem_st_wait();
        }
        tc_fence_before();
        if (ok) warp_arrive_leader(&sm.bar_ds_full[g]);
        if (u + 2 < nq) store_inputs(buf ^ 1);
        wait_w(&sm.bar_dq_full[g], ng & 1);
        tc_fence_after();
        if (ok) {
          uint32_t v0[32];
          tmem_ld32(tmem + lane_off + col_s(g) + kQH * r, v0);
          tmem_ld_wait();
          tc_fence_before();
          warp_arrive_leader(&sm.bar_dq_read[g]);
          // raw sums of dS K over the pair's keys for this CTA's 32 queries
          const int qh0 = q0 + kQH * r;
          const int nvalid = min(kQH, e - qh0);
          float* stg = sm.dqs[g][quad] + lane;  // row = query, element = this dim
          if (nvalid == kQH) {
#pragma unroll
            for (int c = 0; c < 32; ++c) stg[c * 32] = __uint_as_float(v0[c]);
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) stg[c * 32] = c < nvalid ? __uint_as_float(v0[c]) : 0.f;
          }
          fence_proxy_async_smem();
        }
        if (!ok) abort_pair();
        named_barrier_sync(bar_id, kGroupThreads);
        if (issuer && !sm.abort && q0 + kQH * r < e) {
#pragma unroll
          for (int c = 0; c < kD / 32; ++c)
            tma_reduce_add_3d(&map_dq, smem_u32(sm.dqs[g][c]), 32 * c, h, q0 + kQH * r);
          bulk_commit_group();
        }
      }
      ug += nq;
      // dV = 2^-8 acc, dK = scale * acc for this CTA's keys; the groups split
      // the head dimension
      wait_w(&sm.bar_acc_full, nk & 1);
      tc_fence_after();
      if (ok && prm.hadamard) {
        __nv_bfloat16* out =
            (g == 0 ? prm.dk : prm.dv) + (static_cast<size_t>(kj) * prm.Hkv + it.hk) * kD;
        const float mul = g == 0 ? prm.sm_scale : (1.f / 256.f);
        uint32_t uu[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tmem + lane_off + (g == 0 ? kColDK : kColDV) + 32 * c, uu[c]);
        tmem_ld_wait();
        float x[kD];
#pragma unroll
        for (int i = 0; i < kD; ++i) x[i] = __uint_as_float(uu[i / 32][i % 32]) * mul;
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
        warp_arrive_leader(&sm.bar_acc_empty);
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
        warp_arrive_leader(&sm.bar_acc_empty);
      }
      ++nk;
    }
    if (issuer) bulk_wait_group0();
    if (!ok) abort_pair();
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (sm.abort) report(prm.status, FLAMIA_DEV_TIMEOUT);
    finish_claims(prm.wl_header + kHdrBwdNext, prm.wl_header + kHdrBwdExit);
  }
  // neither CTA frees its tensor memory or exits while the other may still
  // write its shared memory or arrive on its barriers
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem, 512);
  }
}

}  // namespace

// Pair items exist only where the one-CTA kernel's modes are the defaults:
// float32 unordered dQ, 32 x 32 dS exponents, MXFP8, dynamic claims.
bool bwd_pair_supported(const BwdParams& prm) {
  return prm.dq_turns == nullptr && prm.dq_pre == nullptr && !prm.ds_rows && !prm.token &&
         prm.ds_count == nullptr && prm.sched != kSchedStatic &&
         (prm.causal || prm.sched == kSchedDynamic);
}

cudaError_t launch_bwd128_pair(const BwdParams& prm, const flamia_qtensor* q,
                               const flamia_qtensor* k, const flamia_qtensor* v,
                               const flamia_qtensor* dout, float* acc, cudaStream_t stream) {
  if (!bwd_pair_supported(prm)) return cudaErrorInvalidValue;
  CUtensorMap mqh, mdoh, mqd, mdod, mk, mv, mdq;
  const int T = prm.T, H = prm.H;
  if (!make_token_map(&mqh, q->codes, T, H, kD, kQH, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_token_map(&mdoh, dout->codes, T, H, kD, kQH, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_token_slice_map(&mqd, q->codes, T, H, kD, 64, kQT, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_token_slice_map(&mdod, dout->codes, T, H, kD, 64, kQT, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_token_map(&mk, k->codes, T, prm.Hkv, kD, kTile, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_token_map(&mv, v->codes, T, prm.Hkv, kD, kTile, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_f32_token_map(&mdq, acc, T, H, kD, kQH, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(PairSmem) + 1024;
  cudaError_t err = cudaFuncSetAttribute(attn_bwd_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  // persistent: as many pairs as can be resident at once (the kernel's
  // cluster shape is fixed at compile time)
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.gridDim = dim3(2);
  int clusters = 0;
  err = cudaOccupancyMaxActiveClusters(&clusters, attn_bwd_pair_kernel, &cfg);
  if (err != cudaSuccess) return err;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const long long pairs = std::min<long long>(clusters, (static_cast<long long>(prm.cap) * prm.Hkv + 1) / 2);
  attn_bwd_pair_kernel<<<static_cast<unsigned>(2 * std::max<long long>(pairs, 1)), kThreads, smem,
                         stream>>>(mqh, mdoh, mqd, mdod, mk, mv, mdq, prm);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace flamia
