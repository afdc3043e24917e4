// Single-tile tensor-core product used by the tests to check operand
// descriptors and scale-factor placement (declared in flamia_debug.h).
#include "../../include/flamia_debug.h"
#include "common.cuh"
#include "ptx.cuh"

namespace flamia {
namespace {

struct ProbeSmem {
  alignas(1024) uint8_t a[128 * 128];
  alignas(1024) uint8_t b[128 * 128];
  uint64_t bar_load, bar_mma;
  uint32_t tmem_base;
};

struct ProbeArgs {
  int mode, N, a_mn, b_mn, variant;  // modes 3 / 4: modes 1 / 0 with A from tensor memory
  const uint8_t* a_g;                 // A in global memory ([128][128] K-major, mode 3)
  int a_bytes, b_bytes;
  uint32_t a_rowb, b_rowb;  // bytes per shared-memory row of each operand
  const uint8_t* sfa;
  const uint8_t* sfb;
  float* d;
  int* status;
};

__device__ __forceinline__ uint32_t layout_for(uint32_t rowb) {
  return rowb == 128 ? kLayoutSW128 : rowb == 64 ? kLayoutSW64 : kLayoutSW32;
}

__global__ void __launch_bounds__(128, 1)
    probe_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                 const ProbeArgs g) {
  extern __shared__ uint8_t smem_raw[];
  ProbeSmem& sm = *reinterpret_cast<ProbeSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.bar_load), 1);
    mbar_init(smem_u32(&sm.bar_mma), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_base), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  bool ok = true;
  if (threadIdx.x == 0) {
    const uint32_t bl = smem_u32(&sm.bar_load);
    mbar_arrive_expect_tx(bl, g.a_bytes + g.b_bytes);
    tma_load_2d(smem_u32(sm.a), &map_a, bl, 0, 0);
    tma_load_2d(smem_u32(sm.b), &map_b, bl, 0, 0);
  }
  // scale factors into tensor memory (columns 128.. for A, 132.. for B)
  if (g.mode == 1 || g.mode == 2 || g.mode == 3) {
    const int variant = (g.variant >> 1) & 3;
    uint32_t w[8];
    for (int c = 0; c < 4; ++c) {
      int ma, nb;
      if (variant == 1) {
        ma = 32 * warp + lane;
        nb = 32 * warp + lane;
      } else {  // 0: every lane quadrant holds all rows; 2: only the rows of this warp
        ma = 32 * c + lane;
        nb = 32 * c + lane;
      }
      uint32_t wa = 0, wb = 0;
      for (int kb = 0; kb < 4; ++kb) {
        wa |= static_cast<uint32_t>(g.sfa[ma * 4 + kb]) << (8 * kb);
        const uint32_t bb = nb < g.N ? g.sfb[nb * 4 + kb] : ((g.mode == 1 || g.mode == 3) ? 127u : 0x38u);
        wb |= bb << (8 * kb);
      }
      // placement 2: A's columns of other warps' rows hold 0 (2^-127), which
      // a product reading them would show; B stays replicated
      w[c] = (variant != 2 || c == warp) ? wa : 0u;
      w[4 + c] = wb;
    }
    tmem_st8(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 128, w);
    tmem_st_wait();
  }
  if (g.mode >= 3) {
    // A row (warp * 32 + lane) into columns 160..191: 4 K elements per column
    uint32_t r[32];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(g.a_g) + (warp * 32 + lane) * 32;
    for (int i = 0; i < 32; ++i) r[i] = src[i];
    tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 160, r);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    ok = mbar_wait(smem_u32(&sm.bar_load), 0);
    tc_fence_after();
    if (ok) {
      const uint32_t aa = smem_u32(sm.a), ba = smem_u32(sm.b);
      const bool swap = g.variant & 1;
      auto kdesc = [&](uint32_t base, uint32_t rowb, int ks) {  // K-major, ks-th 32-byte slice
        return smem_desc(base + 32 * ks, 0, 8 * rowb, layout_for(rowb));
      };
      auto mdesc = [&](uint32_t base, uint32_t rowb, int ks) {  // MN-major, ks-th 32-row slice
        const uint32_t off = 8 * rowb;
        return smem_desc(base + ks * 32 * rowb, swap ? off : 0, swap ? 0 : off, layout_for(rowb));
      };
      if (g.mode >= 3) {
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bd = g.b_mn ? mdesc(ba, g.b_rowb, ks) : kdesc(ba, g.b_rowb, ks);
          if (g.mode == 3)
            mma_mxf8_ts(tmem, tmem + 160 + 8 * ks, bd, idesc_mxf8(128, g.N, 0, g.b_mn, ks, ks),
                        tmem + 128, tmem + 132, ks > 0);
          else
            mma_f8_ts(tmem, tmem + 160 + 8 * ks, bd, idesc_f8(128, g.N, 0, g.b_mn), ks > 0);
        }
      } else if (g.mode == 0 || g.mode == 1) {
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = g.a_mn ? mdesc(aa, g.a_rowb, ks) : kdesc(aa, g.a_rowb, ks);
          const uint64_t bd = g.b_mn ? mdesc(ba, g.b_rowb, ks) : kdesc(ba, g.b_rowb, ks);
          if (g.mode == 0)
            mma_f8(tmem, ad, bd, idesc_f8(128, g.N, g.a_mn, g.b_mn), ks > 0);
          else
            mma_mxf8(tmem, ad, bd, idesc_mxf8(128, g.N, g.a_mn, g.b_mn, ks, ks), tmem + 128,
                     tmem + 132, ks > 0);
        }
      } else {
        mma_nvf4(tmem, smem_desc(aa, 0, 8 * g.a_rowb, layout_for(g.a_rowb)),
                 smem_desc(ba, 0, 8 * g.b_rowb, layout_for(g.b_rowb)), idesc_nvf4(128, g.N),
                 tmem + 128, tmem + 132, 0);
      }
    }
    tc_commit(smem_u32(&sm.bar_mma));
    if (!mbar_wait(smem_u32(&sm.bar_mma), 0)) ok = false;
    if (!ok) report(g.status, FLAMIA_DEV_TIMEOUT);
  }
  __syncthreads();
  tc_fence_after();
  const int row = warp * 32 + lane;
  for (int c = 0; c < g.N / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 32 * c, v);
    tmem_ld_wait();
    for (int i = 0; i < 32; ++i) g.d[row * g.N + 32 * c + i] = __uint_as_float(v[i]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace
}  // namespace flamia

using namespace flamia;

namespace flamia {
namespace {

// tcgen05.ld.red: 128 threads store rows of 32 floats to tensor memory and
// read them back with the max-reducing load.
__global__ void ldred_kernel(const float* in, float* vals, float* mx) {
  __shared__ uint32_t base;
  const int warp = threadIdx.x >> 5, r = threadIdx.x;
  if (warp == 0) {
    tmem_alloc(smem_u32(&base), 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t t = base + (static_cast<uint32_t>(warp * 32) << 16);
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(in[r * 32 + i]);
  tmem_st32(t, w);
  tmem_st_wait();
  uint32_t v[32];
  float m;
  tmem_ld32_max(t, v, m);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) vals[r * 32 + i] = __uint_as_float(v[i]);
  mx[r] = m;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(base, 32);
  }
}

__global__ void bounded_waits_kernel(int* turn, int* status) {
  __shared__ alignas(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  fence_barrier_init();
  if (!mbar_wait(smem_u32(&bar), 0)) report(status, FLAMIA_DEV_TIMEOUT);  // nobody arrives
  if (!wait_turn(turn, 1)) report(status, FLAMIA_DEV_TIMEOUT);           // nobody passes
}

}  // namespace
}  // namespace flamia

extern "C" flamia_status flamia_debug_bounded_waits(int* turn, int* dev_status, void* stream) {
  if (turn == nullptr || dev_status == nullptr) return FLAMIA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(turn, 0, sizeof(int), s) != cudaSuccess) return FLAMIA_ERR_CUDA;
  flamia::bounded_waits_kernel<<<1, 32, 0, s>>>(turn, dev_status);
  flamia::count_launches(1);
  return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

extern "C" flamia_status flamia_debug_mma_tile(int mode, int N, int a_mn_major, int b_mn_major,
                                               int variant, const uint8_t* a, const uint8_t* b,
                                               const uint8_t* sfa, const uint8_t* sfb,
                                               float* d_out, int* dev_status, void* stream) {
  if (mode < 0 || mode > 4 || (N != 32 && N != 64 && N != 128) || variant < 0 || variant > 5)
    return FLAMIA_ERR_UNSUPPORTED;
  if (!a || !b || !d_out || ((mode == 1 || mode == 2 || mode == 3) && (!sfa || !sfb)))
    return FLAMIA_ERR_INVALID_ARG;
  if (mode == 2 && (a_mn_major || b_mn_major)) return FLAMIA_ERR_UNSUPPORTED;
  if (mode >= 3 && a_mn_major) return FLAMIA_ERR_UNSUPPORTED;
  if (!aligned(a, 16) || !aligned(b, 16)) return FLAMIA_ERR_INVALID_ARG;
  const int kbytes = mode == 2 ? 32 : 128;  // K = 128 E4M3 or 64 packed E2M1
  ProbeArgs g;
  g.mode = mode;
  g.N = N;
  g.a_mn = a_mn_major;
  g.b_mn = b_mn_major;
  g.variant = variant;
  g.a_g = a;
  int a_rows, b_rows;
  if (a_mn_major) { a_rows = 128; g.a_rowb = 128; }   // [K][M]
  else { a_rows = 128; g.a_rowb = kbytes; }            // [M][K]
  if (b_mn_major) { b_rows = 128; g.b_rowb = N; }      // [K][N]
  else { b_rows = N; g.b_rowb = kbytes; }              // [N][K]
  g.a_bytes = a_rows * g.a_rowb;
  g.b_bytes = b_rows * g.b_rowb;
  g.sfa = sfa;
  g.sfb = sfb;
  g.d = d_out;
  g.status = dev_status;
  CUtensorMap ma, mb;
  if (!make_matrix_map(&ma, a, a_rows, g.a_rowb, a_rows, swizzle_for_row_bytes(g.a_rowb)) ||
      !make_matrix_map(&mb, b, b_rows, g.b_rowb, b_rows, swizzle_for_row_bytes(g.b_rowb)))
    return FLAMIA_ERR_CUDA;
  const size_t smem = sizeof(ProbeSmem) + 1024;
  if (cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return FLAMIA_ERR_CUDA;
  probe_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(ma, mb, g);
  flamia::count_launches(1);
  return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

namespace flamia {
namespace {

// One product of a CTA pair (tcgen05 .cta_group::2) in each of the three
// shapes the pair backward uses; each CTA loads its own half of the operands
// from global memory and reads its own 128 rows of the result back.
struct PairSmem {
  alignas(1024) uint8_t a[256 * 128];
  alignas(1024) uint8_t b[256 * 32];
  uint64_t bar_load, bar_peer, bar_mma;
  uint32_t tmem_base;
};

struct PairArgs {
  int shape, variant, N;
  int a_bytes, b_bytes;
  const uint8_t* sfa;
  const uint8_t* sfb;
  float* d;
  uint32_t* cols;
  int* status;
};

constexpr uint32_t kPairSfA = 128, kPairSfB = 144;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    pair_probe_kernel(const __grid_constant__ CUtensorMap map_a,
                      const __grid_constant__ CUtensorMap map_b, const PairArgs g) {
  extern __shared__ uint8_t smem_raw[];
  PairSmem& sm = *reinterpret_cast<PairSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.bar_load), 1);
    mbar_init(smem_u32(&sm.bar_peer), 1);
    mbar_init(smem_u32(&sm.bar_mma), 1);
    fence_barrier_init();
  }
  cluster_sync_all();  // barriers initialised before the other CTA arrives on them
  if (warp == 0) {
    tmem_alloc2(smem_u32(&sm.tmem_base), 256);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (threadIdx.x == 0) {
    g.cols[rank] = tmem;
    const uint32_t bl = smem_u32(&sm.bar_load);
    mbar_arrive_expect_tx(bl, g.a_bytes + g.b_bytes);
    const int a_rows = g.shape == 2 ? 256 : 128;
    const int b_rows = g.shape == 0 ? 32 : g.shape == 1 ? 64 : 256;
    tma_load_2d(smem_u32(sm.a), &map_a, bl, 0, static_cast<int>(rank) * a_rows);
    tma_load_2d(smem_u32(sm.b), &map_b, bl, 0, static_cast<int>(rank) * b_rows);
  }
  // scale factors of this CTA's rows (A) and of B, in its own tensor memory
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  if (g.shape == 1) {
    // A: row m's word in lane m, column + m / 32, and (unless variant bit 0)
    // again at column + 4 + m / 32; B: one word (per K block) in every column
    const int m = warp * 32 + lane;
    const uint32_t wa = g.sfa[(rank * 128 + m) * 2] | (static_cast<uint32_t>(g.sfa[(rank * 128 + m) * 2 + 1]) << 8) |
                        0x7F7F0000u;
    const uint32_t wb = g.sfb[0] | (static_cast<uint32_t>(g.sfb[1]) << 8) | 0x7F7F0000u;
    uint32_t w[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) w[c] = (c == warp || (c == 4 + warp && !(g.variant & 1))) ? wa : 0u;
    tmem_st8(tmem + lane_off + kPairSfA, w);
#pragma unroll
    for (int c = 0; c < 8; ++c) w[c] = (!(g.variant & 2) || c < 2) ? wb : 0u;
    tmem_st8(tmem + lane_off + kPairSfB, w);
    tmem_st_wait();
  } else if (g.shape == 2) {
    // A and B: per K block only (8 blocks: two words), in every lane and column
    uint32_t wa[2], wb[2];
    for (int h = 0; h < 2; ++h) {
      wa[h] = wb[h] = 0u;
      for (int i = 0; i < 4; ++i) {
        wa[h] |= static_cast<uint32_t>(g.sfa[rank * 8 + 4 * h + i]) << (8 * i);
        wb[h] |= static_cast<uint32_t>(g.sfb[rank * 8 + 4 * h + i]) << (8 * i);
      }
    }
    uint32_t w[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) w[c] = c < 4 ? wa[0] : wa[1];
    tmem_st8(tmem + lane_off + kPairSfA, w);
#pragma unroll
    for (int c = 0; c < 8; ++c) w[c] = c < 4 ? wb[0] : wb[1];
    tmem_st8(tmem + lane_off + kPairSfB, w);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  bool ok = true;
  if (warp == 0) {
    ok = mbar_wait_w(smem_u32(&sm.bar_load), 0);
    if (rank == 1) {
      // this CTA's operands and scales are in place: tell the issuing CTA
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sm.bar_peer), 0));
    } else {
      ok = mbar_wait_cl_w(smem_u32(&sm.bar_peer), 0) && ok;
      tc_fence_after();
      if (ok) {
        const uint32_t aa = smem_u32(sm.a), ba = smem_u32(sm.b);
        if (g.shape == 0) {
          // S^T-like: A [128][128] K-major, B half [32][128] K-major
          for (int ks = 0; ks < 4; ++ks)
            mma2_f8_w(tmem, smem_desc(aa + 32 * ks, 0, 1024, kLayoutSW128),
                      smem_desc(ba + 32 * ks, 0, 1024, kLayoutSW128), idesc_f8(256, 64, 0, 0),
                      ks > 0);
        } else if (g.shape == 1) {
          // dV-like: A [128][64] K-major, B half [64 K][64 N] MN-major
          for (int ks = 0; ks < 2; ++ks)
            mma2_mxf8_w(tmem, smem_desc(aa + 32 * ks, 0, 512, kLayoutSW64),
                        smem_desc(ba + ks * 32 * 64, 0, 512, kLayoutSW64),
                        idesc_mxf8(256, 128, 0, 1, ks, ks), tmem + kPairSfA, tmem + kPairSfB,
                        ks > 0);
        } else {
          // dQ^T-like: A [256 K][128 M] MN-major, B half [256 K][32 N] MN-major
          for (int ks = 0; ks < 8; ++ks)
            mma2_mxf8_w(tmem, smem_desc(aa + ks * 32 * 128, 0, 1024, kLayoutSW128),
                        smem_desc(ba + ks * 32 * 32, 0, 256, kLayoutSW32),
                        idesc_mxf8(256, 64, 1, 1, ks & 3, ks & 3), tmem + kPairSfA + 4 * (ks >> 2),
                        tmem + kPairSfB + 4 * (ks >> 2), ks > 0);
        }
      }
      tc_commit2_w(smem_u32(&sm.bar_mma), 3);
    }
  }
  if (warp == 0) {
    ok = mbar_wait_cl_w(smem_u32(&sm.bar_mma), 0) && ok;
    if (!ok && lane == 0) report(g.status, FLAMIA_DEV_TIMEOUT);
  }
  __syncthreads();
  tc_fence_after();
  const int row = warp * 32 + lane;
  float* out = g.d + (static_cast<size_t>(rank) * 128 + row) * g.N;
  for (int c = 0; c < g.N / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(tmem + lane_off + 32 * c, v);
    tmem_ld_wait();
    for (int i = 0; i < 32; ++i) out[32 * c + i] = __uint_as_float(v[i]);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA frees or exits while the pair may still touch it
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc2(tmem, 256);
  }
}

}  // namespace
}  // namespace flamia

extern "C" flamia_status flamia_debug_pair_mma(int shape, int variant, const uint8_t* a,
                                               const uint8_t* b, const uint8_t* sfa,
                                               const uint8_t* sfb, float* d_out,
                                               uint32_t* tmem_cols, int* dev_status,
                                               void* stream) {
  using namespace flamia;
  if (shape < 0 || shape > 2 || variant < 0 || variant > 3) return FLAMIA_ERR_UNSUPPORTED;
  if (!a || !b || !d_out || !tmem_cols || !dev_status || (shape > 0 && (!sfa || !sfb)))
    return FLAMIA_ERR_INVALID_ARG;
  if (!aligned(a, 16) || !aligned(b, 16)) return FLAMIA_ERR_INVALID_ARG;
  // per CTA: A rows x bytes, B rows x bytes (the global arrays hold both CTAs' halves)
  const int a_rows = shape == 2 ? 256 : 128, a_rowb = shape == 1 ? 64 : 128;
  const int b_rows = shape == 0 ? 32 : shape == 1 ? 64 : 256, b_rowb = shape == 0 ? 128 : shape == 1 ? 64 : 32;
  PairArgs g;
  g.shape = shape;
  g.variant = variant;
  g.N = shape == 1 ? 128 : 64;
  g.a_bytes = a_rows * a_rowb;
  g.b_bytes = b_rows * b_rowb;
  g.sfa = sfa;
  g.sfb = sfb;
  g.d = d_out;
  g.cols = tmem_cols;
  g.status = dev_status;
  CUtensorMap ma, mb;
  if (!make_matrix_map(&ma, a, 2 * a_rows, a_rowb, a_rows, swizzle_for_row_bytes(a_rowb)) ||
      !make_matrix_map(&mb, b, 2 * b_rows, b_rowb, b_rows, swizzle_for_row_bytes(b_rowb)))
    return FLAMIA_ERR_CUDA;
  const size_t smem = sizeof(PairSmem) + 1024;
  if (cudaFuncSetAttribute(pair_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return FLAMIA_ERR_CUDA;
  pair_probe_kernel<<<2, 128, smem, static_cast<cudaStream_t>(stream)>>>(ma, mb, g);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

extern "C" flamia_status flamia_debug_tmem_ldred(const float* in, float* vals, float* mx,
                                                 void* stream) {
  if (in == nullptr || vals == nullptr || mx == nullptr) return FLAMIA_ERR_INVALID_ARG;
  flamia::ldred_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(in, vals, mx);
  flamia::count_launches(1);
  return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}
