// Fused token-block quantiser (FLAMIA review page, sec. 3.1, 3.2 and 3.4
// "Quantization fusion" / "Packed documents").
//
// One CTA owns the 32-token blocks whose first token lies in a 128-token
// segment of one head.  The rows of those blocks (at most 128 + 31) are read
// once from HBM by one TMA box into shared memory, reduced to per-block
// maxima, and written back as E4M3 codes plus the per-token E8M0 scale table,
// optionally with the NVFP4 copy and with D = dO . O fused in, or with the
// rows rotated by the Sylvester-Hadamard matrix first (review page, sec. 3.4
// "Hadamard rotation"; float32 butterflies across the lanes that hold a row,
// redone where the rows are read, so nothing extra goes through memory).
// HBM-bound: 2 bytes read + 1 byte written per element.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace flamia {
namespace {

constexpr int kSeg = 128;             // tokens per CTA segment
constexpr int kQThreads = kSeg + 32;  // one thread per token of [seg0, seg0 + 160)

__device__ __forceinline__ int doc_of(const int32_t* __restrict__ cu, int ndocs, int t) {
  int lo = 0, hi = ndocs;  // cu[lo] <= t < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid;
    else hi = mid;
  }
  return lo;
}

// The same document index found by a whole warp: each step the 32 lanes probe
// 32 points inside [lo, hi) and keep the interval between the last probe
// with cu <= t and the next, so a search over any number of documents takes
// about four dependent loads (log_33).  Every step shrinks the interval, so
// it ends on malformed offsets too (which the callers flag and clamp).
__device__ __forceinline__ int warp_doc_of(const int32_t* __restrict__ cu, int ndocs, int t,
                                           int lane) {
  int lo = 0, hi = ndocs;
  while (hi - lo > 1) {
    const int span = hi - lo;
    const int p = span <= 33 ? lo + 1 + lane : lo + ((lane + 1) * span) / 33;
    const bool in = span <= 33 ? p < hi : true;
    const unsigned below = __ballot_sync(0xffffffffu, in && __ldg(cu + p) <= t);
    const int k = __popc(below);
    const int last = k == 0 ? lo : __shfl_sync(0xffffffffu, p, k - 1);
    const int next = __shfl_sync(0xffffffffu, p, min(k, 31));
    hi = (k == 32 || (span <= 33 && k >= span - 1)) ? hi : next;
    lo = last;
  }
  return lo;
}

// Offsets of the documents a CTA's staged rows can belong to, cached in
// shared memory (one-token documents: about 160 of them), when the call has
// more than kFewDocs documents.
constexpr int kCuCache = 192;
constexpr int kFewDocs = 64;

// 2^e as a float for e in [-127, 127] (2^-127 is a subnormal).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? exp2i(e) : exp2i(-126) * 0.5f;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The 8 BF16 elements of one lane's 16-byte chunk as floats.
__device__ __forceinline__ void unpack8(const uint4& xv, float (&v)[8]) {
  const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = bf16lo(w[j]);
    v[2 * j + 1] = bf16hi(w[j]);
  }
}

// Up to three tensors of one call (Q, K, V: the same T, d and documents)
// quantised by one launch: grid.y runs over the heads of tensor 0, then of
// tensor 1, then of tensor 2, so one launch fills the GPU three times longer
// and pays one tail.  f4codes[z] == nullptr: no NVFP4 copy for tensor z.
// With D fused (one tensor, dO), map1 describes O's rows.
struct QuantJob {
  uint8_t* codes[3];
  uint8_t* scales[3];
  uint8_t* f4codes[3];
  uint8_t* f4scales[3];
  int H[3];
  int n;
  int blk;    // tokens per scale block: 32, or 1 (per-token operand scales)
  int ahead;  // CTAs resident at once: each CTA brings the rows of the CTA one
              // wave ahead into L2, so HBM keeps streaming while waves compute
};

template <int DIM, bool HAD, bool FUSE_D>
__global__ void __launch_bounds__(kQThreads)
    quantize_kernel(const __grid_constant__ CUtensorMap map0,
                    const __grid_constant__ CUtensorMap map1,
                    const __grid_constant__ CUtensorMap map2, int T,
                    const int32_t* __restrict__ cu, int ndocs, const QuantJob job,
                    const uint4* __restrict__ o, float* __restrict__ D, int* dev_status) {
  constexpr int LPR = DIM / 8;    // lanes per row: 16 bytes (8 BF16) per lane
  constexpr int RPI = 32 / LPR;   // rows per warp-wide read
  constexpr int NLD = 32 / RPI;   // reads per 32 rows
  // the rows [seg0, seg0 + 160) of this head, staged by one TMA box
  __shared__ alignas(128) uint4 s_x[kQThreads * LPR];
  __shared__ float s_rmax[kQThreads];
  __shared__ float s_pre[kQThreads], s_suf[kQThreads];
  __shared__ int s_exp[kQThreads];
  __shared__ int s_bounds[2];
  __shared__ int s_doc[2];
  __shared__ int s_cu[kCuCache];
  __shared__ alignas(8) uint64_t s_bar;

  const int seg0 = blockIdx.x * kSeg;
  // head h of tensor z (fields picked by selects: no indexed copy of the job)
  int h = blockIdx.y, z = 0;
  if (job.n > 1 && h >= job.H[0]) {
    h -= job.H[0];
    z = 1;
    if (job.n > 2 && h >= job.H[1]) {
      h -= job.H[1];
      z = 2;
    }
  }
  const int H = z == 0 ? job.H[0] : z == 1 ? job.H[1] : job.H[2];
  uint8_t* __restrict__ codes = z == 0 ? job.codes[0] : z == 1 ? job.codes[1] : job.codes[2];
  uint8_t* __restrict__ scales = z == 0 ? job.scales[0] : z == 1 ? job.scales[1] : job.scales[2];
  uint8_t* __restrict__ f4codes =
      z == 0 ? job.f4codes[0] : z == 1 ? job.f4codes[1] : job.f4codes[2];
  uint8_t* __restrict__ f4scales =
      z == 0 ? job.f4scales[0] : z == 1 ? job.f4scales[1] : job.f4scales[2];
  const CUtensorMap* map_x = z == 0 ? &map0 : z == 1 ? &map1 : &map2;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(smem_u32(&s_bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(smem_u32(&s_bar), kQThreads * DIM * 2);
    tma_load_3d(smem_u32(s_x), map_x, smem_u32(&s_bar), 0, h, seg0);
    // the rows of the CTA one wave ahead (same grid order: segment fastest)
    const int nx = static_cast<int>(gridDim.x);
    const int ahead = static_cast<int>(blockIdx.y) * nx + static_cast<int>(blockIdx.x) + job.ahead;
    if (job.ahead > 0 && ahead < nx * static_cast<int>(gridDim.y)) {
      int ha = ahead / nx, za = 0;
      const int sa = (ahead % nx) * kSeg;
      if (job.n > 1 && ha >= job.H[0]) {
        ha -= job.H[0];
        za = 1;
        if (job.n > 2 && ha >= job.H[1]) {
          ha -= job.H[1];
          za = 2;
        }
      }
      tma_prefetch_l2_3d(za == 0 ? &map0 : za == 1 ? &map1 : &map2, 0, ha, sa);
      if (FUSE_D) tma_prefetch_l2_3d(&map1, 0, ha, sa);
    }
  }
  const int chunk = lane % LPR;
  // D = dO . O: this lane's O chunks of its rows, loaded while the rows of
  // dO are staged and reduced (their latency hides behind phases 1 and 2)
  uint4 ov[FUSE_D ? NLD : 1];
  if (FUSE_D) {
#pragma unroll
    for (int i = 0; i < NLD; ++i) {
      const int tt = seg0 + warp * 32 + i * RPI + lane / LPR;
      ov[i] = tt < T ? __ldg(o + (static_cast<size_t>(tt) * H + h) * LPR + chunk)
                     : make_uint4(0, 0, 0, 0);
    }
  }

  // Light validation of cu_seqlens, spread over the CTAs of the first head.
  if (blockIdx.y == 0) {
    for (int i = blockIdx.x * kQThreads + tid; i < ndocs; i += gridDim.x * kQThreads)
      if (__ldg(cu + i) > __ldg(cu + i + 1)) report(dev_status, FLAMIA_DEV_BAD_SEQLENS);
    if (blockIdx.x == 0 && tid == 0 && (__ldg(cu) != 0 || __ldg(cu + ndocs) != T))
      report(dev_status, FLAMIA_DEV_BAD_SEQLENS);
  }

  // Documents of the staged rows.  With many documents, warps 0 and 1 find
  // those of the first and the last row, the offsets between them are cached
  // in shared memory once, and each thread searches there (17 dependent
  // loads per thread on 131,072 one-token documents otherwise); with a few,
  // each thread's own search is shorter than the extra step.
  int d0 = 0, nd = 0;
  bool cached = false;
  if (ndocs > kFewDocs) {  // uniform over the grid
    const int tlast = min(seg0 + kQThreads, T) - 1;
    if (warp < 2) {
      const int d = warp_doc_of(cu, ndocs, warp == 0 ? seg0 : tlast, lane);
      if (lane == 0) s_doc[warp] = d;
    }
    __syncthreads();
    d0 = s_doc[0];
    const int d1 = s_doc[1];
    nd = d1 - d0 + 2;  // offsets cu[d0 .. d1 + 1]
    cached = d1 >= d0 && nd <= kCuCache;
    if (cached)
      for (int i = tid; i < nd; i += kQThreads) s_cu[i] = __ldg(cu + d0 + i);
    __syncthreads();
  }
  // Block of this thread's token.
  const int t = seg0 + tid;
  int bs = 0, be = 0;
  if (t < T) {
    int sraw, eraw;
    if (cached) {
      // s_cu[0] <= seg0 <= t < s_cu[nd - 1] for well-formed offsets: the
      // same largest document with cu <= t as the search over all of them
      int lo = 0, hi = nd - 1;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_cu[mid] <= t) lo = mid;
        else hi = mid;
      }
      sraw = s_cu[lo];
      eraw = s_cu[lo + 1];
    } else {
      const int b = doc_of(cu, ndocs, t);
      sraw = __ldg(cu + b);
      eraw = __ldg(cu + b + 1);
    }
    // clamped so that malformed offsets (flagged above) cannot move any
    // index outside [t - 31, t + 31] and [0, T)
    const int s = min(max(sraw, 0), t);
    const int e = max(min(eraw, T), t + 1);
    bs = s + ((t - s) & ~(job.blk - 1));
    be = min(bs + job.blk, e);
  }
  // This CTA owns the rows [A, Bend): blocks starting inside [seg0, seg0 + kSeg).
  if (tid == 0) s_bounds[0] = (bs == seg0) ? seg0 : be;
  if (tid == min(kSeg, T - seg0) - 1) s_bounds[1] = be;
  __syncthreads();
  const int A = s_bounds[0], Bend = s_bounds[1];
  // every thread waits for the staged rows (bounded: a timeout is reported)
  if (!mbar_wait(smem_u32(&s_bar), 0)) {
    if (tid == 0) report(dev_status, FLAMIA_DEV_TIMEOUT);
    return;
  }

  // Phase 1: per-row maximum of this warp's 32 tokens.
#pragma unroll
  for (int i = 0; i < NLD; ++i) {
    const int rl = warp * 32 + i * RPI + lane / LPR;  // row inside the staged box
    const int tt = seg0 + rl;
    const bool valid = tt >= A && tt < Bend;
    float v[8];
    unpack8(s_x[rl * LPR + chunk], v);
    if (HAD) fwht_row<8, LPR>(v, chunk);  // the LPR lanes of a row, all lanes together
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (chunk == 0) s_rmax[rl] = valid ? m : 0.f;
  }
  __syncthreads();

  // Phase 2: block maxima by segmented scans over each warp's 32 rows (lane =
  // row): prefix maxima restart at block starts, suffix maxima at block ends;
  // a block's maximum is suffix(first row) max prefix(last row), whether or
  // not it crosses a warp boundary.  Rows outside [A, Bend) stand alone.
  {
    const bool own = t >= A && t < Bend;
    float pre = s_rmax[tid], suf = pre;
    int hf = own ? (t == bs) : 1, tf = own ? (t == be - 1) : 1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float yp = __shfl_up_sync(0xffffffffu, pre, off);
      const int fp = __shfl_up_sync(0xffffffffu, hf, off);
      const float ys = __shfl_down_sync(0xffffffffu, suf, off);
      const int fs = __shfl_down_sync(0xffffffffu, tf, off);
      if (lane >= off && !hf) {
        pre = fmaxf(pre, yp);
        hf |= fp;
      }
      if (lane + off < 32 && !tf) {
        suf = fmaxf(suf, ys);
        tf |= fs;
      }
    }
    s_pre[tid] = pre;
    s_suf[tid] = suf;
  }
  __syncthreads();
  // block maximum -> round-up exponent -> dense per-token scale byte
  if (t >= A && t < Bend) {
    const float amax = fmaxf(s_suf[max(bs, A) - seg0], s_pre[min(be, Bend) - 1 - seg0]);
    const int e = roundup_exponent(amax);
    s_exp[tid] = e;
    scales[static_cast<size_t>(h) * T + t] = static_cast<uint8_t>(e + 127);
  }
  __syncthreads();

  // Phase 3: codes (+ NVFP4 copy, + D) from the registers (fully unrolled
  // with D, so that the prefetched O chunks stay in registers).
  constexpr int kUnroll = FUSE_D ? NLD : 4;
#pragma unroll kUnroll
  for (int i = 0; i < NLD; ++i) {
    const int rl = warp * 32 + i * RPI + lane / LPR;
    const int tt = seg0 + rl;
    const bool valid = tt >= A && tt < Bend;
    const int e = valid ? s_exp[rl] : 0;
    const float inv = exp2i(-e);  // e in [-127, 120]: 2^-e is a normal float
    float v[8];
    unpack8(s_x[rl * LPR + chunk], v);
    if (HAD) fwht_row<8, LPR>(v, chunk);
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = cvt_e4m3x2(v[2 * j] * inv, v[2 * j + 1] * inv);
    const size_t row = static_cast<size_t>(tt) * H + h;
    if (valid) {
      uint2 packed = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
      reinterpret_cast<uint2*>(codes + row * DIM)[chunk] = packed;
    }
    if (f4codes != nullptr) {
      // NVFP4: one E4M3 scale per 16 elements = two neighbouring lanes.
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      const float q = __fdiv_rn(m, 6.0f);
      uint32_t sc = cvt_e4m3x2(q, 0.f) & 0xFFu;          // nearest E4M3 (saturating)
      const float sv = e4m3x2_to_float2(sc).x;
      if (sv < q && sc < 0x7Eu) sc += 1;                  // round up to >= amax / 6
      const float s = e4m3x2_to_float2(sc).x;
      uint32_t f4 = 0;
      if (s > 0.f) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          f4 |= cvt_e2m1x2(__fdiv_rn(v[2 * j], s), __fdiv_rn(v[2 * j + 1], s)) << (8 * j);
      }
      if (valid) {
        reinterpret_cast<uint32_t*>(f4codes + row * (DIM / 2))[chunk] = f4;
        if ((chunk & 1) == 0) f4scales[row * (DIM / 16) + chunk / 2] = static_cast<uint8_t>(sc);
      }
    }
    if (FUSE_D) {
      const uint4 oi = valid ? ov[i] : make_uint4(0, 0, 0, 0);
      const uint32_t ow[4] = {oi.x, oi.y, oi.z, oi.w};
      const float scale = pow2f(e);
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 dq = e4m3x2_to_float2(c[j]);
        acc = fmaf(dq.x * scale, bf16lo(ow[j]), acc);
        acc = fmaf(dq.y * scale, bf16hi(ow[j]), acc);
      }
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (chunk == 0 && valid) D[static_cast<size_t>(h) * T + tt] = acc;
    }
  }
}

// Tensor map of BF16 rows seen as 2-byte elements (dim, head, token); box =
// one head x 160 rows.
bool make_rows_map(CUtensorMap* map, const void* x, int T, int H, int d) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * 2 * H};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 1u, static_cast<cuuint32_t>(kQThreads)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(x), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Host checks of one tensor's arguments; on success fills its slot of the job.
flamia_status check_tensor(const void* x, int H, int format, const flamia_qtensor* out,
                           QuantJob& job, int z) {
  // (FLAMIA_FORMAT_TOKEN_SCALES is taken off by the callers)
  if (format != FLAMIA_FORMAT_MXFP8 && format != FLAMIA_FORMAT_MXFP8_NVFP4)
    return FLAMIA_ERR_UNSUPPORTED;
  if (x == nullptr || out == nullptr || out->codes == nullptr || out->scales == nullptr)
    return FLAMIA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out->codes, 16)) return FLAMIA_ERR_INVALID_ARG;
  job.codes[z] = out->codes;
  job.scales[z] = out->scales;
  job.f4codes[z] = nullptr;
  job.f4scales[z] = nullptr;
  if (format == FLAMIA_FORMAT_MXFP8_NVFP4) {
    if (out->nvfp4_codes == nullptr || out->nvfp4_scales == nullptr ||
        !aligned(out->nvfp4_codes, 16))
      return FLAMIA_ERR_INVALID_ARG;
    job.f4codes[z] = out->nvfp4_codes;
    job.f4scales[z] = out->nvfp4_scales;
  }
  job.H[z] = H;
  return FLAMIA_OK;
}

// One launch over the job's tensors (xs[z] their BF16 inputs).
flamia_status launch_quantize(const void* const* xs, QuantJob& job, int T, int d,
                              const int32_t* cu, int ndocs, bool had, const void* o_bf16,
                              float* D, int* dev_status, cudaStream_t s) {
  CUtensorMap maps[3] = {};
  int rows = 0;
  for (int z = 0; z < job.n; ++z) {
    if (!make_rows_map(&maps[z], xs[z], T, job.H[z], d)) return FLAMIA_ERR_CUDA;
    rows += job.H[z];
  }
  for (int z = job.n; z < 3; ++z) maps[z] = maps[0];
  // D fused: the second map describes O's rows (prefetched one wave ahead)
  if (D != nullptr && !make_rows_map(&maps[1], o_bf16, T, job.H[0], d)) return FLAMIA_ERR_CUDA;
  if (rows > 65535) return FLAMIA_ERR_UNSUPPORTED;
  dim3 grid((T + kSeg - 1) / kSeg, rows);
  const bool fd = D != nullptr;
  auto kern = d == 128 ? (had ? quantize_kernel<128, true, false>
                              : fd ? quantize_kernel<128, false, true> : quantize_kernel<128, false, false>)
                       : (had ? quantize_kernel<64, true, false>
                              : fd ? quantize_kernel<64, false, true> : quantize_kernel<64, false, false>);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kQThreads, 0) != cudaSuccess)
    return FLAMIA_ERR_CUDA;
  job.ahead = per_sm * num_sms();
  kern<<<grid, kQThreads, 0, s>>>(maps[0], maps[1], maps[2], T, cu, ndocs, job,
                                  static_cast<const uint4*>(o_bf16), D, dev_status);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

}  // namespace
}  // namespace flamia

using namespace flamia;

extern "C" flamia_status flamia_quantize_tokenblock(const void* x_bf16, int T, int H, int d,
                                                    const int32_t* cu_seqlens, int ndocs,
                                                    int format, const void* o_bf16, float* D,
                                                    const flamia_qtensor* out, int* dev_status,
                                                    void* stream) {
  if (!supported_dim(d)) return FLAMIA_ERR_UNSUPPORTED;
  const bool had = (format & FLAMIA_FORMAT_HADAMARD) != 0;
  const bool tok = (format & FLAMIA_FORMAT_TOKEN_SCALES) != 0;
  format &= ~(FLAMIA_FORMAT_HADAMARD | FLAMIA_FORMAT_TOKEN_SCALES);
  if (had && (format != FLAMIA_FORMAT_MXFP8 || o_bf16 != nullptr || D != nullptr))
    return FLAMIA_ERR_UNSUPPORTED;
  if (tok && format != FLAMIA_FORMAT_MXFP8) return FLAMIA_ERR_UNSUPPORTED;
  if (!valid_sizes(T, H, d, ndocs) || cu_seqlens == nullptr) return FLAMIA_ERR_INVALID_ARG;
  if ((o_bf16 == nullptr) != (D == nullptr)) return FLAMIA_ERR_INVALID_ARG;
  if (o_bf16 && !aligned(o_bf16, 16)) return FLAMIA_ERR_INVALID_ARG;
  QuantJob job{};
  job.n = 1;
  job.blk = tok ? 1 : kBlock;
  const flamia_status st = check_tensor(x_bf16, H, format, out, job, 0);
  if (st != FLAMIA_OK) return st;
  const void* xs[1] = {x_bf16};
  return launch_quantize(xs, job, T, d, cu_seqlens, ndocs, had, o_bf16, D, dev_status,
                         static_cast<cudaStream_t>(stream));
}

extern "C" flamia_status flamia_quantize_qkv(const void* q_bf16, const void* k_bf16,
                                             const void* v_bf16, int T, int H, int H_kv, int d,
                                             const int32_t* cu_seqlens, int ndocs, int format_qk,
                                             const flamia_qtensor* q, const flamia_qtensor* k,
                                             const flamia_qtensor* v, int* dev_status,
                                             void* stream) {
  if (!supported_dim(d)) return FLAMIA_ERR_UNSUPPORTED;
  const bool had = (format_qk & FLAMIA_FORMAT_HADAMARD) != 0;
  const bool tok = (format_qk & FLAMIA_FORMAT_TOKEN_SCALES) != 0;
  const int fmt = format_qk & ~(FLAMIA_FORMAT_HADAMARD | FLAMIA_FORMAT_TOKEN_SCALES);
  if (had && fmt != FLAMIA_FORMAT_MXFP8) return FLAMIA_ERR_UNSUPPORTED;
  if (tok && fmt != FLAMIA_FORMAT_MXFP8) return FLAMIA_ERR_UNSUPPORTED;
  if (H_kv <= 0 || H <= 0 || H % H_kv != 0) return FLAMIA_ERR_INVALID_ARG;
  if (!valid_sizes(T, H, d, ndocs) || cu_seqlens == nullptr) return FLAMIA_ERR_INVALID_ARG;
  QuantJob job{};
  job.blk = tok ? 1 : kBlock;  // V takes the same scale blocks as Q and K
  flamia_status st;
  if ((st = check_tensor(q_bf16, H, fmt, q, job, 0)) != FLAMIA_OK ||
      (st = check_tensor(k_bf16, H_kv, fmt, k, job, 1)) != FLAMIA_OK)
    return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (had) {  // Q and K rotated in one launch, V (never rotated) in its own
    job.n = 2;
    const void* xs[2] = {q_bf16, k_bf16};
    if ((st = launch_quantize(xs, job, T, d, cu_seqlens, ndocs, true, nullptr, nullptr,
                              dev_status, s)) != FLAMIA_OK)
      return st;
    QuantJob jv{};
    jv.n = 1;
    jv.blk = job.blk;
    if ((st = check_tensor(v_bf16, H_kv, FLAMIA_FORMAT_MXFP8, v, jv, 0)) != FLAMIA_OK) return st;
    const void* xv[1] = {v_bf16};
    return launch_quantize(xv, jv, T, d, cu_seqlens, ndocs, false, nullptr, nullptr, dev_status,
                           s);
  }
  if ((st = check_tensor(v_bf16, H_kv, FLAMIA_FORMAT_MXFP8, v, job, 2)) != FLAMIA_OK) return st;
  job.n = 3;
  const void* xs[3] = {q_bf16, k_bf16, v_bf16};
  return launch_quantize(xs, job, T, d, cu_seqlens, ndocs, false, nullptr, nullptr, dev_status, s);
}
