// Causal backward over token-block MXFP8 operands (FLAMIA review page, sec.
// 1.2, 3.1, 3.3, 3.4 "Backward pass"): the entry point, and the kernel for
// head dim 64 (MXFP8 or the mixed NVFP4 score product); head dim 128 runs the
// pipelined kernel of attn_bwd128.cu.
//
// One work item = one 128-key tile of a document x one head; it walks the
// 128-query tiles of the same document from the diagonal to the document end.
// Items are ordered head-major (all key tiles of a head, longest first, then
// the next head), so the Q / dO tiles and the dQ rows a wave of CTAs touches
// belong to few heads and stay in L2.  Warp roles:
//   warp 0       TMA producer: K, V per item; Q, dO tiles through a 3-stage ring.
//   warp 1       tensor-memory owner and single-thread tcgen05 MMA issuer.
//   warps 4-7    compute group 0: query columns 0..63 of every tile
//   warps 8-11   compute group 1: query columns 64..127
//   (thread = key row of S^T / dP^T; for the dQ partial thread = query row,
//   the two groups splitting the head dimension).
// Per query tile t:
//   S^T = K Q^T and dP^T = V dO^T (unscaled E4M3, f32 in TMEM);
//   the compute groups recompute P = exp2(s - lse2) with the forward's
//   factors and masks, write the dV operand RNE_E4M3(2^8 P) and the dS codes
//   (one round-up exponent per document-aligned 32x32 block) to shared
//   memory, and the block scales of the three products to TMEM;
//   dV += P^b^T dO, dK += dS^T Q (both stay in TMEM over all t) and
//   dQ_t = dS K are block-scaled MMAs;
//   dQ_t is staged in shared memory and added in float32 to the global
//   accumulator by bulk tensor reduce-adds.
// The tensor core and the compute groups overlap in both directions: the
// groups signal as soon as they have loaded the last S^T / dP^T columns of
// tile t into registers, and S^T / dP^T of tile t+1 are issued then, while
// the groups still turn tile t into P^b and dS; the products of tile t run
// while the groups compute tile t+1, which reads dQ_t out after its own
// recompute (the P^b / dS payloads and the block scales are double-buffered
// by tile parity).
// Tensor memory (512 columns): S^T [0,128), dP^T [128,256), dV [256,320),
// dK [320,384), the NVFP4 score scales [384,396), the block scales of the
// products of even / odd tiles [400,424) / [424,448), dQ_t [448,512).
#include <cuda_bf16.h>

#include "bwd_common.cuh"

namespace flamia {
namespace {

constexpr int kBStages = 3;
constexpr int kBwdThreads = 384;
constexpr int kComputeThreads = 256;
constexpr uint32_t kColSP = 0, kColDP = 128, kColDV = 256, kColDQ = 448;
// block-scale columns of a tile's products, by tile parity
constexpr uint32_t kColSf = 400;
constexpr uint32_t kSfDvA = 0, kSfDvB = 4, kSfDkA = 8, kSfDkB = 12, kSfDqA = 16, kSfDqB = 20;
__device__ __forceinline__ uint32_t col_sf(int t) { return kColSf + 24u * static_cast<uint32_t>(t & 1); }

template <int DIM, bool NVF4, bool OPT>
struct BwdSmem {
  static constexpr int kTileBytes = kTile * DIM;
  static constexpr int kTile4Bytes = NVF4 ? kTile * DIM / 2 : 16;  // packed E2M1 tile
  alignas(1024) uint8_t k[kTileBytes];
  alignas(1024) uint8_t v[kTileBytes];
  alignas(1024) uint8_t q[kBStages][kTileBytes];
  alignas(1024) uint8_t dout[kBStages][kTileBytes];
  // [key][query] E4M3, 128B-swizzled rows, by tile parity
  alignas(1024) uint8_t pb[2][kTile * kTile];
  alignas(1024) uint8_t ds[2][kTile * kTile];
  // query-row dS exponents (optional-mode instances only): dQ's dS codes
  alignas(1024) uint8_t ds2[OPT ? 2 : 1][OPT ? kTile * kTile : 1024];
  // dQ_t staging: DIM/32 boxes of [128 query rows][32 floats], 128B-swizzled
  alignas(1024) float dqs[DIM / 32][kTile * 32];
  alignas(NVF4 ? 1024 : 16) uint8_t k4[kTile4Bytes];
  alignas(NVF4 ? 1024 : 16) uint8_t q4[kBStages][kTile4Bytes];
  // per-query-tile inputs, double-buffered by tile parity (the next tile's are
  // loaded while the current one is processed)
  alignas(16) float nl[2][kTile];  // 8 - lse2 of each query column (-inf outside the document)
  alignas(16) float dd[2][kTile];  // D of each query column (0 outside)
  // FP16 dQ: prescale 2^p of each query (0 outside); four buffers: written a
  // tile ahead, and a tile's dQ is staged during the next tile, after the
  // compute threads' arrival on bar_tile of that tile
  alignas(16) float pf[4][kTile];
  // per-token operand scales, per query and tile parity: 2^eQ, 2^eD (dO),
  // 2^(eD - EdO) (dV's fold), 2^(eQ - EQ) (dK's fold); EQ, EdO the query
  // block's largest exponents
  alignas(16) float tq[OPT && !NVF4 ? 4 : 1][2][OPT && !NVF4 ? kTile : 4];
  // E8M0 bytes of the 4 query blocks of Q and dO, three buffers (written a
  // tile ahead; read for the block scales after the wait on bar_tile)
  uint32_t qbyte[3][4], dobyte[3][4];
  // by tile parity (a fast warp may start the next tile's recompute while a
  // slow one still reads this tile's to write the block scales)
  uint32_t eds[2][4][4];         // dS block bytes [query block][key block]
  uint8_t erow[2][4][4][32];     // query-row dS bytes [query block][key block][query]
  uint64_t bar_kv;
  uint64_t bar_qd_full[kBStages];
  uint64_t bar_qd_empty[kBStages];
  uint64_t bar_s_full, bar_sdp_read, bar_ds_full, bar_dq_full, bar_dq_read, bar_done, bar_sf;
  uint64_t bar_staged, bar_stage_free;  // dQ staging: compute groups <-> reducer warp
  uint64_t bar_kv_free, bar_acc_full, bar_acc_empty;
  // once per query tile: every compute thread has written its dS block bytes
  // and the next tile's per-query inputs
  uint64_t bar_tile;
  ItemRing<4> ring;  // claimed items: producer -> MMA issuer, compute leader
  int item_bc[2];    // the compute leader's copy for the compute groups
  unsigned long long dscnt[2];  // dS rounded-to-zero diagnostic of this CTA
  uint32_t tmem_base;
  volatile int abort;
};

// one CTA per SM: the largest instance fits the 227 KB a CTA may take (with
// the 1 KB alignment slack of the launch)
static_assert(sizeof(BwdSmem<64, true, true>) + 1024 <= 232448, "backward shared memory");
static_assert(sizeof(BwdSmem<64, false, true>) + 1024 <= 232448, "backward shared memory");

template <int DIM>
__host__ __device__ constexpr uint32_t operand_layout() {
  return DIM == 128 ? kLayoutSW128 : kLayoutSW64;
}

// NVFP4 score product (d = 64): tensor-memory columns of the block scales of
// K (4 columns) and of Q_t (two 4-column buffers, by t parity).
constexpr uint32_t kSfK4 = 384, kSfQ4 = 388;

// OPT: the deterministic dQ mode, the FP16 accumulator or the query-row dS
// exponents are on (their code is compiled only into these instances).
template <int DIM, bool NVF4, bool OPT>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v,
                    const __grid_constant__ CUtensorMap map_do,
                    const __grid_constant__ CUtensorMap map_dq,
                    const __grid_constant__ CUtensorMap map_q4,
                    const __grid_constant__ CUtensorMap map_k4, const BwdParams prm) {
  static_assert(DIM == 64, "head dim 128 runs attn_bwd128_kernel (tensor-memory plan for 64)");
  static_assert(!NVF4 || DIM == 64, "the NVFP4 score product is built for head dim 64");
  using Smem = BwdSmem<DIM, NVF4, OPT>;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int H = prm.H, T = prm.T;
  const int n_items = min(prm.wl_header[kHdrTileBwd], prm.cap);
  const int total = n_items * prm.Hkv;  // (key tile, K / V head) items
  const int G = prm.G;
  // tile v of an item walks the query heads of its K / V head in turn: head
  // hk G + v / nq, queries qs + (v % nq) kTile
  auto tile_head = [&](const BwdItem& it, int v) { return G == 1 ? it.hk : it.hk * G + v / it.nq; };
  auto tile_q0 = [&](const BwdItem& it, int v) {
    return it.qs + (G == 1 ? v : v % it.nq) * kTile;
  };
  if (static_cast<int>(blockIdx.x) >= total) {  // uniform over the CTA
    if (threadIdx.x == 0) finish_claims(prm.wl_header + kHdrBwdNext, prm.wl_header + kHdrBwdExit);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.bar_kv), 1);
    mbar_init(smem_u32(&sm.bar_kv_free), 1);
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(smem_u32(&sm.bar_qd_full[i]), 1);
      mbar_init(smem_u32(&sm.bar_qd_empty[i]), 1);
    }
    mbar_init(smem_u32(&sm.bar_s_full), 1);
    mbar_init(smem_u32(&sm.bar_sdp_read), kComputeThreads);
    mbar_init(smem_u32(&sm.bar_ds_full), kComputeThreads);
    mbar_init(smem_u32(&sm.bar_dq_full), 1);
    mbar_init(smem_u32(&sm.bar_dq_read), kComputeThreads);
    mbar_init(smem_u32(&sm.bar_staged), kComputeThreads);
    mbar_init(smem_u32(&sm.bar_stage_free), 1);
    mbar_init(smem_u32(&sm.bar_acc_full), 1);
    mbar_init(smem_u32(&sm.bar_acc_empty), kComputeThreads);
    mbar_init(smem_u32(&sm.bar_tile), kComputeThreads);
    mbar_init(smem_u32(&sm.bar_done), 1);
    mbar_init(smem_u32(&sm.bar_sf), kTile);
    ring_init(sm.ring, 3);  // the MMA issuer, the compute leader, the dQ reducer
    sm.abort = 0;
    sm.dscnt[0] = sm.dscnt[1] = 0ull;
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
  constexpr uint32_t kTileBytes = Smem::kTileBytes;
  constexpr uint32_t kPairBytes = 2 * kTileBytes + (NVF4 ? Smem::kTile4Bytes : 0);
  constexpr uint32_t lay = operand_layout<DIM>();
  constexpr uint32_t sbo = 8 * DIM;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      prefetch_tensormap(&map_k);
      prefetch_tensormap(&map_v);
      prefetch_tensormap(&map_do);
      const uint32_t bkv = smem_u32(&sm.bar_kv);
      int nk = 0;  // items whose K / V were loaded
      int uc = 0;  // query tiles loaded over all items
      bool ok = true;
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
        // the previous item's K / V are free once its last products are done
        if (nk > 0 && (!mbar_wait(smem_u32(&sm.bar_kv_free), (nk - 1) & 1) || sm.abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bkv, kPairBytes);
        tma_load_3d(smem_u32(sm.k), &map_k, bkv, 0, it.hk, it.k0);
        tma_load_3d(smem_u32(sm.v), &map_v, bkv, 0, it.hk, it.k0);
        if (NVF4) tma_load_3d(smem_u32(sm.k4), &map_k4, bkv, 0, it.hk, it.k0);
        ++nk;
        for (int u = 0; u < it.nq * G; ++u, ++uc) {
          const int st = uc % kBStages;
          if (uc >= kBStages &&
              (!mbar_wait(smem_u32(&sm.bar_qd_empty[st]), ((uc / kBStages) - 1) & 1) ||
               sm.abort)) {
            ok = false;
            break;
          }
          const uint32_t bf = smem_u32(&sm.bar_qd_full[st]);
          mbar_arrive_expect_tx(bf, kPairBytes);
          const int th = tile_head(it, u), tq0 = tile_q0(it, u);
          tma_load_3d(smem_u32(sm.q[st]), &map_q, bf, 0, th, tq0);
          tma_load_3d(smem_u32(sm.dout[st]), &map_do, bf, 0, th, tq0);
          if (NVF4) tma_load_3d(smem_u32(sm.q4[st]), &map_q4, bf, 0, th, tq0);
        }
        if (ok) idx = claims.next();
      }
      if (nk > 0) ok &= mbar_wait(bkv, (nk - 1) & 1);
      for (int u = max(0, uc - kBStages); u < uc; ++u)
        ok &= mbar_wait(smem_u32(&sm.bar_qd_full[u % kBStages]), (u / kBStages) & 1);
      if (!ok) sm.abort = 1;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this role on warp-uniform values; one elected lane
    // issues each tcgen05 instruction.  Order per tile t: S^T / dP^T of tile
    // t+1 (once the groups hold tile t's in registers), then dV_t, dK_t and
    // dQ_t (once tile t's dS is written and dQ_{t-1} has been read out).  Each
    // barrier phase is waited for before the next one can complete.
    {
      const uint32_t id_s = idesc_f8(kTile, kTile, 0, 0);
      // operand descriptors, built once: a K step, a ring stage or a payload
      // buffer moves only the start address (bits 0..13, address / 16), which
      // never carries out of its field inside shared memory
      const uint64_t dk = smem_desc(smem_u32(sm.k), 0, sbo, lay);
      const uint64_t dv = smem_desc(smem_u32(sm.v), 0, sbo, lay);
      const uint64_t dq0 = smem_desc(smem_u32(sm.q[0]), 0, sbo, lay);
      const uint64_t ddo0 = smem_desc(smem_u32(sm.dout[0]), 0, sbo, lay);
      const uint64_t dpb0 = smem_desc(smem_u32(sm.pb[0]), 0, 1024, kLayoutSW128);
      const uint64_t dds0 = smem_desc(smem_u32(sm.ds[0]), 0, 1024, kLayoutSW128);
      // dQ's dS operand: the query-row-exponent copy when asked for
      const uint64_t ddq0 =
          smem_desc(smem_u32(OPT && prm.ds_rows ? sm.ds2[0] : sm.ds[0]), 0, 1024, kLayoutSW128);
      constexpr uint32_t kStep = kTileBytes / 16;         // one ring stage
      constexpr uint32_t kPStep = kTile * kTile / 16;     // one payload buffer
      int nk = 0, uc = 0;  // items and query tiles consumed so far
      bool ok = true;
      // S^T_t and dP^T_t: tile t's Q / dO have landed and the groups have read
      // tile t-1's S^T / dP^T columns
      auto issue_sdp = [&](int t) -> bool {
        const int st = t % kBStages;
        if (!mbar_wait_w_ab(smem_u32(&sm.bar_qd_full[st]), (t / kBStages) & 1, &sm.abort) ||
            (t > 0 && !mbar_wait_w_ab(smem_u32(&sm.bar_sdp_read), (t - 1) & 1, &sm.abort)))
          return false;
        tc_fence_after();
        const uint64_t dq = dq0 + st * kStep, ddo = ddo0 + st * kStep;
        if (NVF4) {
          // S^T from the NVFP4 copies: packed E2M1 rows of 32 bytes, one K = 64 product
          mma_nvf4_w(tmem + kColSP, smem_desc(smem_u32(sm.k4), 0, 256, kLayoutSW32),
                     smem_desc(smem_u32(sm.q4[st]), 0, 256, kLayoutSW32),
                     idesc_nvf4(kTile, kTile), tmem + kSfK4, tmem + kSfQ4 + 4 * (t & 1), 0);
        } else {
#pragma unroll
          for (int ks = 0; ks < DIM / 32; ++ks)
            mma_f8_w(tmem + kColSP, dk + 2 * ks, dq + 2 * ks, id_s, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < DIM / 32; ++ks)
          mma_f8_w(tmem + kColDP, dv + 2 * ks, ddo + 2 * ks, id_s, ks > 0);
        tc_commit_w(smem_u32(&sm.bar_s_full));
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
        ok = mbar_wait_w(smem_u32(&sm.bar_kv), nk & 1);
        if (NVF4) ok = ok && mbar_wait_w(smem_u32(&sm.bar_sf), nk & 1);
        ++nk;
        const int ntot = it.nq * G;  // tiles over the item's query heads
        if (ntot > 0) ok = ok && issue_sdp(uc);
        for (int u = 0; ok && u < ntot; ++u, ++uc) {
          const int st = uc % kBStages, b = uc & 1;
          const uint64_t dq = dq0 + st * kStep, ddo = ddo0 + st * kStep;
          const uint64_t dpb = dpb0 + b * kPStep, dds = dds0 + b * kPStep;
          const uint64_t ddq = ddq0 + b * kPStep;
          const uint32_t sf = tmem + col_sf(uc);
          // the next tile's S^T / dP^T as soon as this tile's are in registers
          if (u + 1 < ntot && !issue_sdp(uc + 1)) {
            ok = false;
            break;
          }
          // dV / dK restart from zero on an item's first tile: the previous
          // item's epilogue must have read them
          if (!mbar_wait_w_ab(smem_u32(&sm.bar_ds_full), uc & 1, &sm.abort) ||
              (u == 0 && nk > 1 &&
               !mbar_wait_w_ab(smem_u32(&sm.bar_acc_empty), (nk - 2) & 1, &sm.abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dV += P^b^T dO : A [key][query] K-major, B = dO tile read MN-major
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            mma_mxf8_w(tmem + kColDV, dpb + 2 * kb, ddo + kb * (32 * DIM / 16),
                       idesc_mxf8(kTile, DIM, 0, 1, kb, kb), sf + kSfDvA, sf + kSfDvB,
                       (u > 0 || kb > 0));
          // dK += dS^T Q : A [key][query] K-major, B = Q tile read MN-major
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            mma_mxf8_w(tmem + kColDV + DIM, dds + 2 * kb, dq + kb * (32 * DIM / 16),
                       idesc_mxf8(kTile, DIM, 0, 1, kb, kb), sf + kSfDkA, sf + kSfDkB,
                       (u > 0 || kb > 0));
          tc_commit_w(smem_u32(&sm.bar_qd_empty[st]));
          // dQ_t = dS K into its own columns, once the groups have read dQ_{t-1}:
          // A = the same dS bytes read MN-major (M = queries), B = K MN-major
          if (uc > 0 && !mbar_wait_w_ab(smem_u32(&sm.bar_dq_read), (uc - 1) & 1, &sm.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            mma_mxf8_w(tmem + kColDQ, ddq + kb * (32 * kTile / 16), dk + kb * (32 * DIM / 16),
                       idesc_mxf8(kTile, DIM, 1, 1, kb, kb), sf + kSfDqA, sf + kSfDqB, kb > 0);
          tc_commit_w(smem_u32(&sm.bar_dq_full));
        }
        // dV / dK of the item are complete, and its K / V may be replaced
        if (ok) {
          tc_commit_w(smem_u32(&sm.bar_acc_full));
          tc_commit_w(smem_u32(&sm.bar_kv_free));
        }
      }
      if (!ok) sm.abort = 1;
      tc_commit_w(smem_u32(&sm.bar_done));
      if (!mbar_wait_w(smem_u32(&sm.bar_done), 0)) sm.abort = 1;
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ dQ reducer
    // One thread reduce-adds each tile's staged dQ into the global float32 (or
    // FP16) accumulator, so no compute warp waits for the bulk copies: it
    // follows the items in claim order, waits for a tile's staging, issues the
    // reduce-adds and frees the staging buffer once they have read it (in the
    // deterministic mode: once they are complete, passing the tile's turn on).
    if (lane == 0) {
      bool ok = true;
      int tg = 0;  // query tiles over all items
      for (int n = 0; ok; ++n) {
        const int idx = ring_get(sm.ring, n, true);
        if (idx < 0) {
          ok = false;
          break;
        }
        if (idx >= total) break;
        BwdItem it;
        if (!decode_bwd_item(prm, n_items, idx, it)) continue;
        for (int u = 0; u < it.nq * G; ++u, ++tg) {
          if (!mbar_wait(smem_u32(&sm.bar_staged), tg & 1) || sm.abort) {
            ok = false;
            break;
          }
          const int q0 = tile_q0(it, u), h = tile_head(it, u);
          int* turn = !OPT || prm.dq_turns == nullptr
                          ? nullptr
                          : prm.dq_turns + static_cast<size_t>(q0) * prm.H + h;
          if (turn != nullptr && !wait_turn(turn, dq_turn(prm, it, q0))) {
            ok = false;
            break;
          }
          if (OPT && prm.dq_pre != nullptr) {
            const __half* box0 = reinterpret_cast<const __half*>(sm.dqs[0]);
#pragma unroll
            for (int b = 0; b < DIM / 64; ++b)
              tma_reduce_add_3d(&map_dq, smem_u32(box0 + b * (kTile * 64)), 64 * b, h, q0);
          } else {
#pragma unroll
            for (int c = 0; c < DIM / 32; ++c)
              tma_reduce_add_3d(&map_dq, smem_u32(sm.dqs[c]), 32 * c, h, q0);
          }
          bulk_commit_group();
          if (turn != nullptr) {
            bulk_wait_group0();
            pass_turn(turn);
          } else {
            bulk_wait_group_read0();
          }
          mbar_arrive(smem_u32(&sm.bar_stage_free));
        }
      }
      bulk_wait_group0();
      if (!ok) sm.abort = 1;
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute groups
    const int g = (warp - 4) >> 2;   // 0: query columns 0..63, 1: 64..127
    const int quad = warp & 3;
    const int j = quad * 32 + lane;  // key row (S^T, dP^T, dV, dK) / query row (dQ_t)
    const bool issuer = (warp == 4 && lane == 0);
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float LOG2E = 1.4426950408889634f;
    // Every compute thread runs the same sequence of named barriers whatever
    // happens: a wait that times out only clears `ok`, which skips the work
    // (never a barrier), so no thread can be left waiting at bar.sync.
    bool ok = true;
    int uc = 0;  // query tiles processed over all items (phase and buffer parity)
    int nk = 0;  // items processed
    // dQ_t (tile t = ut of the item, global index tg) from tensor memory to the
    // staging buffer, for the reducer warp; every compute thread calls it (it
    // arrives on dq_read, then on staged).  The buffer is free once the
    // reducer's bulk copies of the previous tile have read it.
    auto read_dq = [&](const BwdItem& it, int ut, int tg) {
      ok = ok && mbar_wait_ab(smem_u32(&sm.bar_dq_full), tg & 1, &sm.abort) &&
           (tg == 0 || mbar_wait_ab(smem_u32(&sm.bar_stage_free), (tg - 1) & 1, &sm.abort));
      tc_fence_after();
      if (!ok) return;
      const bool qv = tile_q0(it, ut) + j < it.e;  // TMEM lane j of dQ_t is query row j
      constexpr int kCh = DIM / 64;  // 32-column chunks of dQ_t per group
      uint32_t v[kCh][32];
#pragma unroll
      for (int cc = 0; cc < kCh; ++cc)
        tmem_ld32(tmem + lane_off + kColDQ + 32 * (g * kCh + cc), v[cc]);
      tmem_ld_wait();
      // dQ of the next tile may now be written
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.bar_dq_read));
      if (OPT && prm.dq_pre != nullptr) {
        // x 2^p of the query row (0 outside the document), rounded to FP16,
        // in DIM / 64 boxes [128 query rows][64 halves], 128B-swizzled
        const float pf = sm.pf[tg & 3][j];
        __half* box0 = reinterpret_cast<__half*>(sm.dqs[0]);
#pragma unroll
        for (int t = 0; t < 4 * kCh; ++t) {  // 8-dim chunk t of this group's dims
          const int dim0 = g * 32 * kCh + 8 * t;
          const int b = dim0 / 64, ch = (dim0 % 64) / 8;
          uint32_t w[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const __half2 h2 = __floats2half2_rn(
                __uint_as_float(v[t / 4][8 * (t % 4) + 2 * x]) * pf,
                __uint_as_float(v[t / 4][8 * (t % 4) + 2 * x + 1]) * pf);
            w[x] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(box0 + b * (kTile * 64) + j * 64 + 8 * (ch ^ (j & 7))) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < kCh; ++cc) {
          float* row = sm.dqs[g * kCh + cc] + j * 32;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            // softmax_scale is applied once, in the float32 -> BF16 conversion
            float4 f = make_float4(__uint_as_float(v[cc][4 * i]), __uint_as_float(v[cc][4 * i + 1]),
                                   __uint_as_float(v[cc][4 * i + 2]),
                                   __uint_as_float(v[cc][4 * i + 3]));
            if (!qv) f = make_float4(0.f, 0.f, 0.f, 0.f);  // rows of other documents add 0
            *reinterpret_cast<float4*>(row + 4 * (i ^ (j & 7))) = f;
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&sm.bar_staged));
    };
    for (int n = 0;; ++n) {
      if (issuer) sm.item_bc[n & 1] = ring_get(sm.ring, n, true);
      named_barrier_sync(1, kComputeThreads);
      const int idx = sm.item_bc[n & 1];
      if (idx < 0) {
        ok = false;
        break;
      }
      if (idx >= total) break;
      BwdItem it;
      if (!decode_bwd_item(prm, n_items, idx, it)) continue;
      const int e = it.e, k0 = it.k0, nt = it.nq, nq = nt * G;
      const int kj = k0 + j;
      const bool key_valid = kj < it.k1;
      const size_t hT = static_cast<size_t>(it.hk) * T;  // K / V scale rows
      const int ekj = (key_valid && !NVF4) ? static_cast<int>(prm.k_scales[hT + kj]) - 127 : 0;
      const int evj = key_valid ? static_cast<int>(prm.v_scales[hT + kj]) - 127 : 0;
      const float rowf = pow2_or_zero(ekj) * prm.scale_log2;
      const float rowg = pow2_or_zero(evj);
      // E8M0 bytes of this key tile's 4 key blocks (B scale of dQ_t = dS K)
      uint32_t kword = 0;
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        const int kk = k0 + 32 * kb;
        kword |= (kk < e ? static_cast<uint32_t>(prm.k_scales[hT + kk]) : 127u) << (8 * kb);
      }
      // NVFP4 score product: block scales in tensor memory, one 32-bit word (4
      // E4M3 scales) per row; column c + i of a lane quadrant holds row 32 i +
      // lane (the same words in every quadrant).  Group 0 writes them.
      auto write_sf4 = [&](const uint32_t* words, int heads, int hh, int tok0, uint32_t col) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w[i] = words[static_cast<size_t>(min(tok0 + 32 * i + lane, T - 1)) * heads + hh];
        tmem_st4(tmem + lane_off + col, w);
      };
      if (NVF4 && g == 0) {
        // the previous item's score products completed before its last tile
        // was computed
        write_sf4(prm.k4_scales, prm.Hkv, it.hk, k0, kSfK4);
        write_sf4(prm.q4_scales, H, tile_head(it, 0), tile_q0(it, 0), kSfQ4 + 4 * (uc & 1));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.bar_sf));
      }
      // the per-query inputs of tile u: raw loads from clamped (always valid)
      // addresses, issued a tile ahead and only used when stored (group 0)
      float r_lse = 0.f, r_dd = 0.f;
      uint32_t r_qb = 127u, r_dob = 127u;
      int r_pre = 0;
      bool r_qv = false;
      auto fetch_query_inputs = [&](int u) {
        const int qi = tile_q0(it, u) + j;
        r_qv = qi < e;
        const size_t at = static_cast<size_t>(tile_head(it, u)) * T + min(qi, T - 1);
        r_lse = prm.lse[at];
        r_dd = prm.D[at];
        if (OPT && prm.dq_pre != nullptr) r_pre = prm.dq_pre[at];
        if (lane == 0 || (OPT && !NVF4 && prm.token)) {
          r_qb = prm.q_scales[at];
          r_dob = prm.do_scales[at];
        }
      };
      auto store_query_inputs = [&](int tg) {
        const int b = tg & 1, b3 = tg % 3;
        sm.nl[b][j] = r_qv ? 8.f - r_lse * LOG2E : -INFINITY;
        sm.dd[b][j] = r_qv ? r_dd : 0.f;
        if (OPT) sm.pf[tg & 3][j] = r_qv ? exp2i(r_pre) : 0.f;
        if constexpr (OPT && !NVF4) {
          if (prm.token) {
            // per-token operand scales: this query's factors and its block's
            // largest exponents (the B scales of dK and dV)
            const int eqb = r_qv ? static_cast<int>(r_qb) : 0;
            const int edb = r_qv ? static_cast<int>(r_dob) : 0;
            const int EQ = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(eqb)));
            const int ED = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(edb)));
            sm.tq[0][b][j] = r_qv ? pow2_or_zero(eqb - 127) : 0.f;
            sm.tq[1][b][j] = r_qv ? pow2_or_zero(edb - 127) : 0.f;
            sm.tq[2][b][j] = r_qv ? pow2_or_zero(edb - ED) : 0.f;
            sm.tq[3][b][j] = r_qv ? pow2_or_zero(eqb - EQ) : 0.f;
            if (lane == 0) {
              sm.qbyte[b3][quad] = static_cast<uint32_t>(EQ);
              sm.dobyte[b3][quad] = static_cast<uint32_t>(ED);
            }
            return;
          }
        }
        if (lane == 0) {
          sm.qbyte[b3][quad] = r_qv ? r_qb : 127u;
          sm.dobyte[b3][quad] = r_qv ? r_dob : 127u;
        }
      };
      if (g == 0) {
        fetch_query_inputs(0);
        store_query_inputs(uc);
      }
      named_barrier_sync(1, kComputeThreads);
      for (int u = 0; u < nq; ++u, ++uc) {
        const int ub = uc & 1, ub3 = uc % 3;
        if (g == 0 && u + 1 < nq) fetch_query_inputs(u + 1);  // lands during this tile
        ok = ok && mbar_wait_ab(smem_u32(&sm.bar_s_full), uc & 1, &sm.abort);
        tc_fence_after();
        uint8_t* pbrow = sm.pb[ub] + j * kTile;
        uint8_t* dsrow = sm.ds[ub] + j * kTile;
#pragma unroll 1
        for (int cc = 0; cc < 2 && ok; ++cc) {
          const int c = 2 * g + cc;  // 32-query block of this chunk
          const float fS =
              NVF4 ? rowf : rowf * pow2_or_zero(static_cast<int>(sm.qbyte[ub3][c]) - 127);
          const float fP = rowg * pow2_or_zero(static_cast<int>(sm.dobyte[ub3][c]) - 127);
          uint32_t sv[32], dv[32];
          tmem_ld32(tmem + lane_off + kColSP + 32 * c, sv);
          tmem_ld32(tmem + lane_off + kColDP + 32 * c, dv);
          tmem_ld_wait();
          if (cc == 1) {
            // every S^T / dP^T column this thread needs is in registers: the
            // next tile's may be computed (its NVFP4 Q scales first)
            if (NVF4 && g == 0 && u + 1 < nq) {
              write_sf4(prm.q4_scales, H, tile_head(it, u + 1), tile_q0(it, u + 1),
                        kSfQ4 + 4 * ((uc + 1) & 1));
              tmem_st_wait();
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&sm.bar_sdp_read));
          }
          uint32_t pw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          float amax = 0.f;
          const bool tok = OPT && !NVF4 && prm.token;
          // per-token operand scales: dK's operand is dS 2^(eQ - EQ) per query
          const float* kq = sm.tq[OPT && !NVF4 ? 3 : 0][ub] + 32 * c;
          if (!key_valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) dv[i] = 0u;
          } else if (tok) {
            const float* q0p = sm.tq[0][ub] + 32 * c;
            const float* d0p = sm.tq[OPT && !NVF4 ? 1 : 0][ub] + 32 * c;
            const float* p0p = sm.tq[OPT && !NVF4 ? 2 : 0][ub] + 32 * c;
            if (prm.causal && (G == 1 ? u : u % nt) == 0)
              bwd_chunk_tok<true>(sv, dv, sm.nl[ub] + 32 * c, sm.dd[ub] + 32 * c, q0p, d0p, p0p,
                                  rowf, rowg, 32 * c, j, pw);
            else
              bwd_chunk_tok<false>(sv, dv, sm.nl[ub] + 32 * c, sm.dd[ub] + 32 * c, q0p, d0p, p0p,
                                   rowf, rowg, 32 * c, j, pw);
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(dv[i]) * kq[i]));
          } else if (prm.causal && (G == 1 ? u : u % nt) == 0) {
            amax = bwd_chunk<true>(sv, dv, sm.nl[ub] + 32 * c, sm.dd[ub] + 32 * c, fS, fP,
                                   32 * c, j, pw);
          } else {
            amax = bwd_chunk<false>(sv, dv, sm.nl[ub] + 32 * c, sm.dd[ub] + 32 * c, fS, fP,
                                    32 * c, j, pw);
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
            float2 b = make_float2(__uint_as_float(dv[i + 2]), __uint_as_float(dv[i + 3]));
            if (tok) {
              a = __fmul2_rn(a, make_float2(kq[i], kq[i + 1]));
              b = __fmul2_rn(b, make_float2(kq[i + 2], kq[i + 3]));
            }
            a = __fmul2_rn(a, inv2);
            b = __fmul2_rn(b, inv2);
            dw[i / 4] = cvt_e4m3x4(a.x, a.y, b.x, b.y);
          }
          if (OPT && prm.ds_count != nullptr) count_ds_zero(dv, dw, sm.dscnt, lane);
          const int ch0 = (2 * c) ^ (j & 7), ch1 = (2 * c + 1) ^ (j & 7);
          *reinterpret_cast<uint4*>(pbrow + 16 * ch0) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          *reinterpret_cast<uint4*>(pbrow + 16 * ch1) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
          *reinterpret_cast<uint4*>(dsrow + 16 * ch0) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
          *reinterpret_cast<uint4*>(dsrow + 16 * ch1) = make_uint4(dw[4], dw[5], dw[6], dw[7]);
          if (lane == 0) sm.eds[ub][c][quad] = static_cast<uint32_t>(eb + 127);
          if (OPT && prm.ds_rows) {
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
            sm.erow[ub][c][quad][lane] = static_cast<uint8_t>(er + 127);
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
            uint8_t* ds2row = sm.ds2[OPT ? ub : 0] + j * kTile;
            *reinterpret_cast<uint4*>(ds2row + 16 * ch0) = make_uint4(dr[0], dr[1], dr[2], dr[3]);
            *reinterpret_cast<uint4*>(ds2row + 16 * ch1) = make_uint4(dr[4], dr[5], dr[6], dr[7]);
          }
        }
        // the next tile's per-query inputs (their nl / dd buffer was last read
        // by tile t-1's recompute, the byte buffer by tile t-2's block scales,
        // the prescale buffer by tile t-3's staging), visible after the wait on
        // bar_tile, which also completes the dS block exponents.  Split
        // arrive / wait: the previous tile's dQ is read out in between, so a
        // fast warp does that instead of waiting for the slowest one.  Every
        // compute thread arrives once per tile, whatever happened.
        if (g == 0 && u + 1 < nq) store_query_inputs(uc + 1);
        mbar_arrive(smem_u32(&sm.bar_tile));
        // dQ of the previous tile, computed while this tile was recomputed
        if (u > 0) read_dq(it, u - 1, uc - 1);
        ok = ok && mbar_wait_ab(smem_u32(&sm.bar_tile), uc & 1, &sm.abort);
        if (ok) {
          // block scales of the three products (this tile's parity buffer,
          // last read by the products of tile t-2, complete before tile t's
          // S^T); every lane quadrant holds the same words: column (base +
          // m/32) of an A scale holds the 4 K-block bytes of rows m/32*32 .. +31
          const uint32_t sfc = col_sf(uc);
          uint32_t w[8];
          if (g == 0) {
            const uint32_t* db = sm.dobyte[ub3];
            const uint32_t* qb = sm.qbyte[ub3];
            const uint32_t dow = db[0] | (db[1] << 8) | (db[2] << 16) | (db[3] << 24);
            const uint32_t qw = qb[0] | (qb[1] << 8) | (qb[2] << 16) | (qb[3] << 24);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              w[i] = 0x7F7F7F7Fu;  // dV: A = P^b, scale 2^0
              w[4 + i] = dow;      // dV: B = dO, per query block
            }
            tmem_st8(tmem + lane_off + sfc + kSfDvA, w);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              // dK: A = dS^T, row block = key block i, K blocks = query blocks
              w[i] = sm.eds[ub][0][i] | (sm.eds[ub][1][i] << 8) | (sm.eds[ub][2][i] << 16) |
                     (sm.eds[ub][3][i] << 24);
              w[4 + i] = qw;  // dK: B = Q, per query block
            }
            tmem_st8(tmem + lane_off + sfc + kSfDkA, w);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              // dQ: A = dS, row block = query block i, K blocks = key blocks
              if (OPT && prm.ds_rows)  // this lane's query 32 i + lane
                w[i] = static_cast<uint32_t>(sm.erow[ub][i][0][lane]) |
                       (static_cast<uint32_t>(sm.erow[ub][i][1][lane]) << 8) |
                       (static_cast<uint32_t>(sm.erow[ub][i][2][lane]) << 16) |
                       (static_cast<uint32_t>(sm.erow[ub][i][3][lane]) << 24);
              else
                w[i] = sm.eds[ub][i][0] | (sm.eds[ub][i][1] << 8) | (sm.eds[ub][i][2] << 16) |
                       (sm.eds[ub][i][3] << 24);
              // dQ: B = K, per key block (2^0: per-token K factors are in dS)
              w[4 + i] = (OPT && !NVF4 && prm.token) ? 0x7F7F7F7Fu : kword;
            }
            tmem_st8(tmem + lane_off + sfc + kSfDqA, w);
          }
        }
        if (ok) {
          tmem_st_wait();
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.bar_ds_full));
        }
        if (!ok) sm.abort = 1;
      }
      // the item's last dQ
      if (nq > 0) read_dq(it, nq - 1, uc - 1);
      if (!ok) sm.abort = 1;
      // every product of the item is complete
      ok = ok && !sm.abort && mbar_wait(smem_u32(&sm.bar_acc_full), nk & 1);
      tc_fence_after();
      ++nk;
      if (ok && prm.hadamard) {
        // Q and K were rotated: group 0 writes whole rows of dK = dK_r H_d
        // (the butterflies need all DIM columns of a row), group 1 of dV
        __nv_bfloat16* out =
            (g == 0 ? prm.dk : prm.dv) + (static_cast<size_t>(kj) * prm.Hkv + it.hk) * DIM;
        const float mul = g == 0 ? prm.sm_scale : (1.f / 256.f);
        uint32_t u[DIM / 32][32];
#pragma unroll
        for (int c = 0; c < DIM / 32; ++c)
          tmem_ld32(tmem + lane_off + kColDV + (g == 0 ? DIM : 0) + 32 * c, u[c]);
        tmem_ld_wait();
        float x[DIM];
#pragma unroll
        for (int i = 0; i < DIM; ++i) x[i] = __uint_as_float(u[i / 32][i % 32]) * mul;
        if (g == 0) fwht_row<DIM, 1>(x, 0);
        if (key_valid) {
#pragma unroll
          for (int i = 0; i < DIM; i += 8) {
            uint32_t w[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(x[i + 2 * t], x[i + 2 * t + 1]);
              w[t] = *reinterpret_cast<uint32_t*>(&b2);
            }
            *reinterpret_cast<uint4*>(out + i) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        // dV / dK columns may now be restarted by the next item
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.bar_acc_empty));
      } else if (ok) {
        // dV = 2^-8 acc, dK = scale * acc, written to the packed buffers; the
        // groups split the head dimension
        __nv_bfloat16* dvrow = prm.dv + (static_cast<size_t>(kj) * prm.Hkv + it.hk) * DIM;
        __nv_bfloat16* dkrow = prm.dk + (static_cast<size_t>(kj) * prm.Hkv + it.hk) * DIM;
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
          const float mul = which == 0 ? (1.f / 256.f) : prm.sm_scale;
          __nv_bfloat16* row = which == 0 ? dvrow : dkrow;
#pragma unroll 1
          for (int c = g * (DIM / 64); c < (g + 1) * (DIM / 64); ++c) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + kColDV + which * DIM + 32 * c, v);
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
        // dV / dK columns may now be restarted by the next item
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.bar_acc_empty));
      }
    }
    if (!ok) sm.abort = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (sm.abort) report(prm.status, FLAMIA_DEV_TIMEOUT);
    if (OPT && prm.ds_count != nullptr) {
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

// ------------------------------------------------- FP16 dQ accumulator prescale
// Review page, sec. 3.2 "accumulator leakage", sec. 3.5.3 "Backward pass": the
// key tiles' dQ partials are reduce-added in FP16 after multiplication by
// 2^p(i).  Every element of a 32-token block satisfies |x| <= 448 2^e (its
// E8M0 exponent), which bounds the raw sum: |sum_j dS^_ij K^_jk| <=
// 16 d 448^3 2^E with E = e_dO(i) + max e_V + max e_K, so
//   p(i) = 15 - ceil(log2(16 d 448^3)) - E   (clamped to [-126, 126])
// keeps |2^p acc| <= 2^15.  The maxima run over the head's whole sequence
// (FLAMIA_FLAG_DQ_FP16) or, with causal dQ scaling, over the keys the row sees.
__host__ __device__ constexpr int dq16_bound_log2(int d) { return d == 128 ? 38 : 37; }

__device__ __forceinline__ int8_t dq16_prescale(int e_sum_bytes, int cbound) {
  const int E = e_sum_bytes - 3 * 127;  // three E8M0 bytes
  return static_cast<int8_t>(min(max(15 - cbound - E, -126), 126));
}

// Per row of the E8M0 tables, the largest byte: rows 0 .. H-1 dO (query
// heads), H .. H+Hkv-1 V, H+Hkv .. H+2Hkv-1 K; maxb zeroed by the caller.
__global__ void scale_max_kernel(const uint8_t* __restrict__ dos, const uint8_t* __restrict__ vs,
                                 const uint8_t* __restrict__ ks, int T, int H, int Hkv,
                                 int* __restrict__ maxb) {
  const int r = blockIdx.y;
  const uint8_t* row = r < H ? dos + static_cast<size_t>(r) * T
                       : r < H + Hkv ? vs + static_cast<size_t>(r - H) * T
                                     : ks + static_cast<size_t>(r - H - Hkv) * T;
  int m = 0;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T; i += gridDim.x * blockDim.x)
    m = max(m, static_cast<int>(row[i]));
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && m > 0) atomicMax(maxb + r, m);
}

// Sequence-wide prescale: one value per query head, written for every token.
__global__ void dq_prescale_seq_kernel(const int* __restrict__ maxb, int T, int H, int Hkv,
                                       int cbound, int8_t* __restrict__ pre) {
  const int G = H / Hkv;
  const size_t n = static_cast<size_t>(T) * H;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int h = static_cast<int>(i / T), hk = h / G;
    pre[i] = dq16_prescale(maxb[h] + maxb[H + hk] + maxb[H + Hkv + hk], cbound);
  }
}

// Causal dQ scaling: one warp per (document, query head) walks the
// document's 32-token blocks 32 at a time (lane = block): running maxima of
// the V and K bytes (inclusive prefix over the lanes, plus the carry of the
// earlier blocks), or the document maxima in a non-causal call, then writes
// the block's prescale to its tokens.
__global__ void dq_prescale_causal_kernel(const uint8_t* __restrict__ dos,
                                          const uint8_t* __restrict__ vs,
                                          const uint8_t* __restrict__ ks,
                                          const int32_t* __restrict__ cu, int ndocs, int T, int H,
                                          int Hkv, int cbound, int causal,
                                          int8_t* __restrict__ pre) {
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5);
       w < static_cast<long long>(ndocs) * H; w += warps) {
    const int doc = static_cast<int>(w / H), h = static_cast<int>(w % H), hk = h / (H / Hkv);
    const int s = min(max(cu[doc], 0), T), e = min(max(cu[doc + 1], s), T);
    const int nb = (e - s + 31) / 32;
    const uint8_t* dr = dos + static_cast<size_t>(h) * T;
    const uint8_t* vr = vs + static_cast<size_t>(hk) * T;
    const uint8_t* kr = ks + static_cast<size_t>(hk) * T;
    int mv = 0, mk = 0;  // carries (E8M0 bytes are >= 0)
    if (!causal) {
      for (int b = lane; b < nb; b += 32) {
        mv = max(mv, static_cast<int>(vr[s + 32 * b]));
        mk = max(mk, static_cast<int>(kr[s + 32 * b]));
      }
      mv = __reduce_max_sync(0xffffffffu, mv);
      mk = __reduce_max_sync(0xffffffffu, mk);
    }
    for (int b0 = 0; b0 < nb; b0 += 32) {
      const int b = b0 + lane;
      int ev = 0, ek = 0, ed = 0;
      if (b < nb) {
        ev = vr[s + 32 * b];
        ek = kr[s + 32 * b];
        ed = dr[s + 32 * b];
      }
      if (causal) {
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int yv = __shfl_up_sync(0xffffffffu, ev, off);
          const int yk = __shfl_up_sync(0xffffffffu, ek, off);
          if (lane >= off) {
            ev = max(ev, yv);
            ek = max(ek, yk);
          }
        }
        ev = max(ev, mv);
        ek = max(ek, mk);
        mv = __shfl_sync(0xffffffffu, ev, 31);
        mk = __shfl_sync(0xffffffffu, ek, 31);
      } else {
        ev = mv;
        ek = mk;
      }
      const int p = dq16_prescale(ed + ev + ek, cbound);
      const int nblk = min(32, nb - b0);
      for (int t = 0; t < nblk; ++t) {
        const int pt = __shfl_sync(0xffffffffu, p, t);
        const int tok = s + 32 * (b0 + t) + lane;
        if (tok < e) pre[static_cast<size_t>(h) * T + tok] = static_cast<int8_t>(pt);
      }
    }
  }
}

// dQ accumulator -> BF16 dQ = softmax_scale * acc (float32), or
// softmax_scale * 2^-p * acc (FP16, p of the row).
// dQ = (sm_scale acc) H_d, one warp per (token, head) row: lane l holds the
// DIM/32 consecutive elements [DIM/32 l, DIM/32 (l + 1)).
template <int DIM>
__global__ void dq_convert_rotate_kernel(const float* __restrict__ acc,
                                         __nv_bfloat16* __restrict__ out, size_t rows,
                                         float sm_scale, const int8_t* __restrict__ pre, int T,
                                         int H) {
  constexpr int N = DIM / 32;
  const int lane = threadIdx.x & 31;
  const size_t warps = static_cast<size_t>(gridDim.x) * (blockDim.x >> 5);
  for (size_t r = blockIdx.x * static_cast<size_t>(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    float v[N];
    if (pre == nullptr) {
      const float* src = acc + r * DIM + N * lane;
#pragma unroll
      for (int i = 0; i < N; ++i) v[i] = src[i] * sm_scale;
    } else {
      const __half* src = reinterpret_cast<const __half*>(acc) + r * DIM + N * lane;
      const float f = exp2i(-pre[(r % H) * T + r / H]);
#pragma unroll
      for (int i = 0; i < N; ++i) v[i] = (__half2float(src[i]) * f) * sm_scale;
    }
    fwht_row<N, 32>(v, lane);
    __nv_bfloat16* dst = out + r * DIM + N * lane;
#pragma unroll
    for (int i = 0; i < N; i += 2)
      *reinterpret_cast<__nv_bfloat162*>(dst + i) = __floats2bfloat162_rn(v[i], v[i + 1]);
  }
}

// FP16 accumulator: 8 elements of one row per thread.
__global__ void dq16_convert_kernel(const uint4* __restrict__ acc, uint4* __restrict__ out,
                                    size_t n8, int d, int T, int H, float sm_scale,
                                    const int8_t* __restrict__ pre) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t r = i * 8 / d;  // (token, head) row
    const float f = exp2i(-pre[(r % H) * T + r / H]);
    const uint4 a = acc[i];
    const uint32_t in[4] = {a.x, a.y, a.z, a.w};
    uint32_t o[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&in[x]));
      const __nv_bfloat162 b2 = __floats2bfloat162_rn((v.x * f) * sm_scale, (v.y * f) * sm_scale);
      o[x] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ out,
                                  size_t n4, float sm_scale) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 a = acc[i];
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * sm_scale, a.y * sm_scale),
                   hi = __floats2bfloat162_rn(a.z * sm_scale, a.w * sm_scale);
    out[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
}

// Backward workspace: float32 [T, H, d] dQ accumulator (the FP16 one uses its
// first half), int32 [T, H] turn counters, int8 [H, T] prescale table, the
// per-row byte maxima (H + 2 H_kv <= 3 H ints); each part 256-byte aligned.
struct BwdWorkspace {
  size_t off_turns, off_pre, off_max, off_count, total;
};
inline BwdWorkspace bwd_workspace(int T, int H, int d) {
  const size_t th = static_cast<size_t>(T) * H;
  BwdWorkspace w;
  w.off_turns = align_up(th * d * sizeof(float), 256);
  w.off_pre = w.off_turns + align_up(th * sizeof(int), 256);
  w.off_max = w.off_pre + align_up(th, 256);
  w.off_count = w.off_max + align_up(3ull * H * sizeof(int), 256);
  w.total = w.off_count + 256;
  return w;
}

template <int DIM, bool NVF4>
flamia_status launch_bwd(const flamia_qtensor* q, const flamia_qtensor* k,
                         const flamia_qtensor* v, const flamia_qtensor* dout, const float* D,
                         const float* lse, const int32_t* cu, int ndocs, int T, int H,
                         int Hkv, float softmax_scale, bool had, bool causal, bool det, int dq16,
                         int sched, bool ds_rows, bool tok, bool dscount, int ctas, void* wl,
                         void* dq, void* dk, void* dv, void* ws, int* status,
                         cudaStream_t stream) {
  ds_rows = ds_rows || tok;  // per-token operand scales take query-row dS exponents
  // (head dim 128 builds its own maps in launch_bwd128_pipelined)
  CUtensorMap mq{}, mk{}, mv{}, mdo{}, mdq{}, mq4{}, mk4{};
  const CUtensorMapSwizzle swz = swizzle_for_row_bytes(DIM);
  const BwdWorkspace W = bwd_workspace(T, H, DIM);
  float* acc = static_cast<float*>(ws);
  if (DIM == 64 && (!make_token_map(&mq, q->codes, T, H, DIM, kTile, swz) ||
      !make_token_map(&mk, k->codes, T, Hkv, DIM, kTile, swz) ||
      !make_token_map(&mv, v->codes, T, Hkv, DIM, kTile, swz) ||
      !make_token_map(&mdo, dout->codes, T, H, DIM, kTile, swz) ||
      !(dq16 ? make_f16_token_map(&mdq, acc, T, H, DIM, kTile, CU_TENSOR_MAP_SWIZZLE_128B)
             : make_f32_token_map(&mdq, acc, T, H, DIM, kTile))))
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
  BwdParams prm;
  prm.q_scales = q->scales;
  prm.k_scales = k->scales;
  prm.v_scales = v->scales;
  prm.do_scales = dout->scales;
  prm.q4_scales = reinterpret_cast<const uint32_t*>(q->nvfp4_scales);
  prm.k4_scales = reinterpret_cast<const uint32_t*>(k->nvfp4_scales);
  prm.D = D;
  prm.lse = lse;
  prm.cu = cu;
  prm.wl_header = static_cast<int*>(wl);
  prm.items = reinterpret_cast<const int4*>(static_cast<const char*>(wl) + L.off_tile_bwd);
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);
  prm.T = T;
  prm.H = H;
  prm.Hkv = Hkv;
  prm.G = H / Hkv;
  prm.ndocs = ndocs;
  prm.cap = L.cap_bwd;
  prm.scale_log2 = softmax_scale * 1.4426950408889634f;
  prm.sm_scale = softmax_scale;
  prm.hadamard = had ? 1 : 0;
  prm.causal = causal ? 1 : 0;
  prm.status = status;
  const size_t n = static_cast<size_t>(T) * H * DIM;
  char* wsb = static_cast<char*>(ws);
  prm.dq_turns = det ? reinterpret_cast<int*>(wsb + W.off_turns) : nullptr;
  int8_t* pre = dq16 ? reinterpret_cast<int8_t*>(wsb + W.off_pre) : nullptr;
  prm.dq_pre = pre;
  // the deterministic mode needs the claims in list order (a turn only waits
  // for an item claimed before it)
  prm.sched = det ? kSchedDynamic : sched;
  prm.ds_rows = ds_rows ? 1 : 0;
  prm.token = tok ? 1 : 0;
  prm.ds_count = dscount ? reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) +
                                                                 W.off_count)
                         : nullptr;
  // the accumulator (float32 or FP16) and, in the deterministic mode, the
  // turn counters behind it
  if (cudaMemsetAsync(acc, 0, n * (dq16 ? 2 : 4), stream) != cudaSuccess ||
      (det && cudaMemsetAsync(wsb + W.off_turns, 0, static_cast<size_t>(T) * H * sizeof(int),
                              stream) != cudaSuccess))
    return FLAMIA_ERR_CUDA;
  if (dscount && cudaMemsetAsync(prm.ds_count, 0, 2 * sizeof(unsigned long long), stream) !=
                     cudaSuccess)
    return FLAMIA_ERR_CUDA;
  if (dq16) {  // the prescale table
    const int cb = dq16_bound_log2(DIM);
    if (dq16 == 1) {
      int* maxb = reinterpret_cast<int*>(wsb + W.off_max);
      if (cudaMemsetAsync(maxb, 0, sizeof(int) * (H + 2 * Hkv), stream) != cudaSuccess)
        return FLAMIA_ERR_CUDA;
      const dim3 g(static_cast<unsigned>(std::min(64, (T + 255) / 256)), H + 2 * Hkv);
      scale_max_kernel<<<g, 256, 0, stream>>>(dout->scales, v->scales, k->scales, T, H, Hkv, maxb);
      const size_t nb = static_cast<size_t>(T) * H;
      const int blocks = static_cast<int>(std::min<size_t>((nb + 255) / 256, 152 * 8));
      dq_prescale_seq_kernel<<<blocks, 256, 0, stream>>>(maxb, T, H, Hkv, cb, pre);
    } else {
      const long long pairs = static_cast<long long>(ndocs) * H;
      const int blocks = static_cast<int>(std::min<long long>((pairs + 7) / 8, 152 * 8));
      dq_prescale_causal_kernel<<<blocks, 256, 0, stream>>>(dout->scales, v->scales, k->scales,
                                                             cu, ndocs, T, H, Hkv, cb,
                                                             causal ? 1 : 0, pre);
    }
    if (cudaGetLastError() != cudaSuccess) return FLAMIA_ERR_CUDA;
    count_launches(dq16 == 1 ? 2 : 1);
  }
  // persistent: one CTA per SM (shared memory allows one), items claimed in list order
  const long long grid = std::min<long long>(static_cast<long long>(L.cap_bwd) * Hkv, num_sms());
  if constexpr (DIM == 128 && !NVF4) {
    // two-CTA items when the caller asks for them; the rule by shape picks
    // one-CTA items for every call (the pair measured about 1.5x slower on
    // every shape, 4 x 4096 and the variable-length 65,536 packing: each
    // 64-query tile hands its products, dS and dQ read-out between the two
    // SMs four times, about 540 cycles a hop)
    const bool pair = ctas == 2 && bwd_pair_supported(prm);
    const cudaError_t e =
        pair ? launch_bwd128_pair(prm, q, k, v, dout, acc, stream)
             : launch_bwd128_pipelined(prm, q, k, v, dout, acc, static_cast<unsigned>(grid), stream);
    if (e != cudaSuccess) return FLAMIA_ERR_CUDA;
  } else {
    const bool opt = det || dq16 || ds_rows || dscount;
    const size_t smem =
        (opt ? sizeof(BwdSmem<DIM, NVF4, true>) : sizeof(BwdSmem<DIM, NVF4, false>)) + 1024;
    auto kernel = opt ? attn_bwd_kernel<DIM, NVF4, true> : attn_bwd_kernel<DIM, NVF4, false>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return FLAMIA_ERR_CUDA;
    kernel<<<static_cast<unsigned>(grid), kBwdThreads, smem, stream>>>(
        mq, mk, mv, mdo, mdq, mq4, mk4, prm);
    if (cudaGetLastError() != cudaSuccess) return FLAMIA_ERR_CUDA;
    count_launches(1);
  }
  if (launch_bwd_short(q, k, v, dout, D, lse, cu, ndocs, T, H, Hkv, DIM, softmax_scale, NVF4, had,
                       causal, ds_rows, tok, prm.ds_count, acc, pre, dk, dv, stream) !=
      cudaSuccess)
    return FLAMIA_ERR_CUDA;
  if (had) {
    const size_t rows = static_cast<size_t>(T) * H;
    const int blocks = static_cast<int>(std::min<size_t>((rows + 7) / 8, 152 * 16));
    dq_convert_rotate_kernel<DIM><<<blocks, 256, 0, stream>>>(
        acc, static_cast<__nv_bfloat16*>(dq), rows, softmax_scale, pre, T, H);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
  }
  if (dq16) {
    const size_t n8 = n / 8;
    const int blocks = static_cast<int>(std::min<size_t>((n8 + 255) / 256, 152 * 16));
    dq16_convert_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const uint4*>(acc),
                                                    static_cast<uint4*>(dq), n8, DIM, T, H,
                                                    softmax_scale, pre);
    count_launches(1);
    return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
  }
  const size_t n4 = n / 4;
  const int blocks = static_cast<int>(std::min<size_t>((n4 + 255) / 256, 152 * 16));
  dq_convert_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(acc),
                                                static_cast<uint2*>(dq), n4, softmax_scale);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

}  // namespace
}  // namespace flamia

using namespace flamia;

extern "C" size_t flamia_bwd_ds_counts_offset(int T, int H, int d) {
  if (T <= 0 || H <= 0 || !supported_dim(d)) return 0;
  return bwd_workspace(T, H, d).off_count;
}

extern "C" size_t flamia_bwd_workspace_bytes(int T, int H, int d) {
  if (T <= 0 || H <= 0 || !supported_dim(d)) return 0;
  return bwd_workspace(T, H, d).total;
}

extern "C" flamia_status flamia_attn_bwd_gqa(const flamia_qtensor* q, const flamia_qtensor* k,
                                             const flamia_qtensor* v, const flamia_qtensor* dout,
                                             const float* D, const float* lse,
                                             const int32_t* cu_seqlens, int ndocs, int T, int H,
                                             int H_kv, int d, float softmax_scale, int flags,
                                             void* wl, void* dq_bf16, void* dk_bf16,
                                             void* dv_bf16, void* ws, size_t ws_bytes,
                                             int* dev_status, void* stream) {
  if (!supported_dim(d)) return FLAMIA_ERR_UNSUPPORTED;
  if (H_kv <= 0 || H <= 0 || H % H_kv != 0) return FLAMIA_ERR_INVALID_ARG;
  if ((flags & ~(FLAMIA_FLAG_NVFP4_QK | FLAMIA_FLAG_HADAMARD | FLAMIA_FLAG_NONCAUSAL |
                 FLAMIA_FLAG_DETERMINISTIC_DQ | FLAMIA_FLAG_DQ_FP16 |
                 FLAMIA_FLAG_DQ_CAUSAL_SCALE | FLAMIA_FLAG_SCHEDULE_STATIC |
                 FLAMIA_FLAG_SCHEDULE_RULE | FLAMIA_FLAG_DS_ROW_EXPONENTS |
                 FLAMIA_FLAG_TOKEN_SCALES | FLAMIA_FLAG_DS_ZERO_COUNT |
                 FLAMIA_FLAG_BWD_CTA_PAIR | FLAMIA_FLAG_BWD_ONE_CTA)) != 0)
    return FLAMIA_ERR_UNSUPPORTED;
  const int ctas = (flags & FLAMIA_FLAG_BWD_CTA_PAIR) ? 2 : (flags & FLAMIA_FLAG_BWD_ONE_CTA) ? 1 : 0;
  if ((flags & FLAMIA_FLAG_BWD_CTA_PAIR) && (flags & FLAMIA_FLAG_BWD_ONE_CTA))
    return FLAMIA_ERR_UNSUPPORTED;
  // the 2-CTA mode runs the default numerics only (head dim 128, MXFP8, float32
  // unordered dQ, 32 x 32 dS exponents, dynamic claims)
  if (ctas == 2 && (d != 128 || (flags & (FLAMIA_FLAG_NVFP4_QK | FLAMIA_FLAG_DETERMINISTIC_DQ |
                                          FLAMIA_FLAG_DQ_FP16 | FLAMIA_FLAG_DS_ROW_EXPONENTS |
                                          FLAMIA_FLAG_TOKEN_SCALES | FLAMIA_FLAG_DS_ZERO_COUNT |
                                          FLAMIA_FLAG_SCHEDULE_STATIC)) ||
                    ((flags & FLAMIA_FLAG_SCHEDULE_RULE) && (flags & FLAMIA_FLAG_NONCAUSAL))))
    return FLAMIA_ERR_UNSUPPORTED;
  const bool ds_rows = (flags & FLAMIA_FLAG_DS_ROW_EXPONENTS) != 0;
  const bool tok = (flags & FLAMIA_FLAG_TOKEN_SCALES) != 0;
  const bool dscount = (flags & FLAMIA_FLAG_DS_ZERO_COUNT) != 0;
  // the diagnostic count runs with the float32, unordered dQ sum
  if (dscount && (flags & (FLAMIA_FLAG_DETERMINISTIC_DQ | FLAMIA_FLAG_DQ_FP16)))
    return FLAMIA_ERR_UNSUPPORTED;
  const int sched = schedule_of(flags);
  if (sched < 0) return FLAMIA_ERR_UNSUPPORTED;
  if ((flags & FLAMIA_FLAG_DETERMINISTIC_DQ) && sched == kSchedStatic) return FLAMIA_ERR_UNSUPPORTED;
  if ((flags & FLAMIA_FLAG_DQ_CAUSAL_SCALE) && !(flags & FLAMIA_FLAG_DQ_FP16))
    return FLAMIA_ERR_UNSUPPORTED;
  const bool nvf4 = (flags & FLAMIA_FLAG_NVFP4_QK) != 0;
  const bool det = (flags & FLAMIA_FLAG_DETERMINISTIC_DQ) != 0;
  const int dq16 = !(flags & FLAMIA_FLAG_DQ_FP16) ? 0
                   : (flags & FLAMIA_FLAG_DQ_CAUSAL_SCALE) ? 2 : 1;
  const bool had = (flags & FLAMIA_FLAG_HADAMARD) != 0;
  const bool causal = (flags & FLAMIA_FLAG_NONCAUSAL) == 0;
  if ((nvf4 && d != 64) || (nvf4 && had) || (nvf4 && tok)) return FLAMIA_ERR_UNSUPPORTED;
  if (!valid_sizes(T, H, d, ndocs) || !q || !k || !v || !dout || !D || !lse || !cu_seqlens ||
      !wl || !dq_bf16 || !dk_bf16 || !dv_bf16 || !ws || !(softmax_scale > 0.f))
    return FLAMIA_ERR_INVALID_ARG;
  if (!q->codes || !q->scales || !k->codes || !k->scales || !v->codes || !v->scales ||
      !dout->codes || !dout->scales)
    return FLAMIA_ERR_INVALID_ARG;
  if (!aligned(q->codes, 16) || !aligned(k->codes, 16) || !aligned(v->codes, 16) ||
      !aligned(dout->codes, 16) || !aligned(dq_bf16, 16) || !aligned(dk_bf16, 16) ||
      !aligned(dv_bf16, 16) || !aligned(ws, 256) || !aligned(wl, 256))
    return FLAMIA_ERR_INVALID_ARG;
  if (ws_bytes < flamia_bwd_workspace_bytes(T, H, d)) return FLAMIA_ERR_WORKSPACE;
  if (nvf4 && (!q->nvfp4_codes || !q->nvfp4_scales || !k->nvfp4_codes || !k->nvfp4_scales ||
               !aligned(q->nvfp4_codes, 16) || !aligned(k->nvfp4_codes, 16) ||
               !aligned(q->nvfp4_scales, 4) || !aligned(k->nvfp4_scales, 4)))
    return FLAMIA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // rotated Q, K: the same scores with softmax_scale / d (exact: d = 2^k)
  const float sc = had ? softmax_scale / static_cast<float>(d) : softmax_scale;
  if (nvf4)
    return launch_bwd<64, true>(q, k, v, dout, D, lse, cu_seqlens, ndocs, T, H, H_kv, sc,
                                false, causal, det, dq16, sched, ds_rows, false, dscount, ctas, wl, dq_bf16,
                                dk_bf16, dv_bf16, ws, dev_status, s);
  return d == 128 ? launch_bwd<128, false>(q, k, v, dout, D, lse, cu_seqlens, ndocs, T, H, H_kv,
                                           sc, had, causal, det, dq16, sched, ds_rows, tok, dscount, ctas, wl,
                                           dq_bf16, dk_bf16, dv_bf16, ws, dev_status, s)
                  : launch_bwd<64, false>(q, k, v, dout, D, lse, cu_seqlens, ndocs, T, H, H_kv,
                                          sc, had, causal, det, dq16, sched, ds_rows, tok, dscount, ctas, wl,
                                          dq_bf16, dk_bf16, dv_bf16, ws, dev_status, s);
}

extern "C" flamia_status flamia_attn_bwd(const flamia_qtensor* q, const flamia_qtensor* k,
                                         const flamia_qtensor* v, const flamia_qtensor* dout,
                                         const float* D, const float* lse,
                                         const int32_t* cu_seqlens, int ndocs, int T, int H,
                                         int d, float softmax_scale, int flags, void* wl,
                                         void* dq_bf16, void* dk_bf16, void* dv_bf16, void* ws,
                                         size_t ws_bytes, int* dev_status, void* stream) {
  return flamia_attn_bwd_gqa(q, k, v, dout, D, lse, cu_seqlens, ndocs, T, H, H, d, softmax_scale,
                             flags, wl, dq_bf16, dk_bf16, dv_bf16, ws, ws_bytes, dev_status,
                             stream);
}
