// GPU work-list builder (FLAMIA review page, sec. 3.4 "Work scheduling").
//
// Forward items are 256-query chunks of a document (cost = 128-key blocks
// seen by the chunk's last query); backward items are 128-key tiles (cost =
// 128-query tiles that see them).  Both lists are sorted by descending cost,
// stable over generation order (document, then position), entirely on the
// device with no host synchronisation:
//   count per document with in-chunk prefixes -> scan of the chunk totals ->
//   emit in generation order with a per-chunk cost histogram -> per-bucket
//   scan over chunks -> scan over buckets in descending cost -> stable
//   scatter (rank inside a chunk).  Every step is a parallel, coalesced pass.
//
// The scatter also writes the tile lists: the same order without the items
// of documents of at most kShortDoc tokens (those run on the CUDA-core
// kernels).  Such a document has exactly one item per list, of cost 1, and
// cost-1 items sort last, so items of cost >= 2 keep their position and the
// long cost-1 items follow in document order: a forward one for documents of
// kShortDoc+1 .. 128 tokens, a backward one (the last key tile) for every
// document longer than kShortDoc.  Their rank is a per-document prefix count.
#include <mutex>
#include <vector>

#include "common.cuh"
#include "ptx.cuh"

namespace flamia {
namespace {

constexpr int kScanThreads = 1024;

// Per-document counts: items of each list, and the 0/1 flags of a long
// cost-1 item in each list.
enum : int { kCntFwd = 0, kCntBwd = 1, kCntLongFwd = 2, kCntLongBwd = 3, kNumCounts = 4 };

struct WlPtrs {
  int* header;
  int4* fwd;
  int4* bwd;
  int4* tile_fwd;
  int4* tile_bwd;
  int* counts;   // [4][ndocs]: prefix of each count inside its 1024-doc chunk
  int* offsets;  // [4][doc chunks]: chunk totals, then chunk start offsets
  int4* gen_fwd;
  int4* gen_bwd;
  int* hist_fwd;  // [chunks][nbuckets]
  int* hist_bwd;
  int* bucket_fwd;  // [nbuckets] bucket totals, then bucket starts
  int* bucket_bwd;
};

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024);
// returns the exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane], wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    s_warp[lane] = wi - w;  // exclusive prefix of the warp totals
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  return s_warp[warp] + incl - v;
}

// Per document: item counts; per 1024-document chunk: the exclusive prefix
// of the counts inside the chunk (counts area) and the chunk totals
// (offsets area, one pair per chunk).
__global__ void __launch_bounds__(kScanThreads)
    wl_count(const int32_t* __restrict__ cu, int ndocs, int T, WlPtrs p, int* dev_status) {
  __shared__ int s_warp[kNumCounts][32];
  __shared__ int s_tot[kNumCounts];
  const int b = blockIdx.x * kScanThreads + threadIdx.x;
  if (b == 0 && (cu[0] != 0 || cu[ndocs] != T)) report(dev_status, FLAMIA_DEV_BAD_SEQLENS);
  int c[kNumCounts] = {0, 0, 0, 0};
  if (b < ndocs) {
    int L = cu[b + 1] - cu[b];
    if (L < 0) {
      report(dev_status, FLAMIA_DEV_BAD_SEQLENS);
      L = 0;
    }
    c[kCntFwd] = (L + kFwdItem - 1) / kFwdItem;
    c[kCntBwd] = (L + kTile - 1) / kTile;
    c[kCntLongFwd] = (L > kShortDoc && L <= kTile) ? 1 : 0;  // its only item, of cost 1
    c[kCntLongBwd] = L > kShortDoc ? 1 : 0;                   // its last key tile
  }
  const int nchunks = gridDim.x;
#pragma unroll
  for (int l = 0; l < kNumCounts; ++l) {
    const int ex = block_exclusive_scan(c[l], s_warp[l], &s_tot[l]);
    if (b < ndocs) p.counts[l * ndocs + b] = ex;
  }
  if (threadIdx.x == 0)
    for (int l = 0; l < kNumCounts; ++l) p.offsets[l * nchunks + blockIdx.x] = s_tot[l];
}

// Exclusive scan of the per-chunk totals (in place); list sizes to the header.
__global__ void __launch_bounds__(kScanThreads)
    wl_scan_docs(int nchunks, int cap_fwd, int cap_bwd, WlPtrs p, int* dev_status) {
  __shared__ int s_warp[kNumCounts][32];
  __shared__ int s_tot[kNumCounts];
  // nchunks <= 2 * kScanThreads (at most 2^20 + 1 documents): two per thread
  int v[kNumCounts][2];
  for (int l = 0; l < kNumCounts; ++l)
    for (int i = 0; i < 2; ++i) {
      const int c = 2 * threadIdx.x + i;
      v[l][i] = c < nchunks ? p.offsets[l * nchunks + c] : 0;
    }
  __syncthreads();  // every total is read before any is overwritten
  for (int l = 0; l < kNumCounts; ++l) {
    const int ex = block_exclusive_scan(v[l][0] + v[l][1], s_warp[l], &s_tot[l]);
    for (int i = 0; i < 2; ++i) {
      const int c = 2 * threadIdx.x + i;
      if (c < nchunks) p.offsets[l * nchunks + c] = ex + (i == 1 ? v[l][0] : 0);
    }
  }
  if (threadIdx.x == 0) {
    p.header[kHdrLong1Fwd] = s_tot[kCntLongFwd];
    p.header[kHdrLong1Bwd] = s_tot[kCntLongBwd];
    p.header[kHdrFwdNext] = 0;
    p.header[kHdrFwdExit] = 0;
    p.header[kHdrBwdNext] = 0;
    p.header[kHdrBwdExit] = 0;
    int nf = s_tot[0], nb = s_tot[1];
    if (nf > cap_fwd || nb > cap_bwd) {
      report(dev_status, FLAMIA_DEV_CAPACITY);
      nf = min(nf, cap_fwd);
      nb = min(nb, cap_bwd);
    }
    p.header[kHdrNFwd] = nf;
    p.header[kHdrNBwd] = nb;
    p.header[kHdrCapFwd] = cap_fwd;
    p.header[kHdrCapBwd] = cap_bwd;
    p.header[kHdrMaxCost] = 0;
  }
}

// Document of generation-order item g: the largest b whose first item is at
// or before g (empty documents share their successor's offset, so the
// largest index is the one that owns g).  Offsets are chunk base + in-chunk
// prefix; both levels are non-decreasing.
__device__ __forceinline__ int doc_of_item(const int* __restrict__ chunk_off,
                                           const int* __restrict__ local, int nchunks, int ndocs,
                                           int g) {
  int lo = 0, hi = nchunks;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (chunk_off[mid] <= g) lo = mid;
    else hi = mid;
  }
  const int c = lo, base = chunk_off[c];
  lo = c * kScanThreads;
  hi = min((c + 1) * kScanThreads, ndocs);
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (base + local[mid] <= g) lo = mid;
    else hi = mid;
  }
  return lo;
}

// One CTA per 1024-item chunk of either list: emit the items in generation
// order and count their costs.
__global__ void __launch_bounds__(kSortChunk)
    wl_emit(const int32_t* __restrict__ cu, int ndocs, int chunks_fwd, int nbuckets, WlPtrs p) {
  extern __shared__ int s_hist[];
  const bool fwd = blockIdx.x < chunks_fwd;
  const int chunk = fwd ? blockIdx.x : blockIdx.x - chunks_fwd;
  const int n = p.header[fwd ? kHdrNFwd : kHdrNBwd];
  const int ndchunks = (ndocs + kScanThreads - 1) / kScanThreads;
  const int* chunk_off = p.offsets + (fwd ? 0 : ndchunks);
  const int* local = p.counts + (fwd ? 0 : ndocs);
  for (int i = threadIdx.x; i < nbuckets; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int g = chunk * kSortChunk + threadIdx.x;
  if (g < n) {
    const int b = doc_of_item(chunk_off, local, ndchunks, ndocs, g);
    const int k = g - (chunk_off[b / kScanThreads] + local[b]);
    const int s = cu[b], e = cu[b + 1];
    int4 it;
    if (fwd) {
      const int q0 = s + kFwdItem * k, q1 = min(q0 + kFwdItem, e);
      it = make_int4(b, q0, q1, (q1 - s + kTile - 1) / kTile);
      p.gen_fwd[g] = it;
    } else {
      const int k0 = s + kTile * k, k1 = min(k0 + kTile, e);
      it = make_int4(b, k0, k1, (e - k0 + kTile - 1) / kTile);
      p.gen_bwd[g] = it;
    }
    atomicAdd(&s_hist[min(it.w, nbuckets - 1)], 1);
  }
  __syncthreads();
  int* hist = (fwd ? p.hist_fwd : p.hist_bwd) + static_cast<size_t>(chunk) * nbuckets;
  for (int i = threadIdx.x; i < nbuckets; i += blockDim.x) hist[i] = s_hist[i];
}

// Per bucket (one warp each): exclusive prefix over chunks (in place);
// bucket totals out.
__global__ void wl_scan_chunks(int nbuckets, int chunks_fwd, int chunks_bwd, WlPtrs p) {
  const int wg = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wg >= 2 * nbuckets) return;  // whole warps exit together
  const bool fwd = wg < nbuckets;
  const int bucket = fwd ? wg : wg - nbuckets;
  int* hist = fwd ? p.hist_fwd : p.hist_bwd;
  const int chunks = fwd ? chunks_fwd : chunks_bwd;
  int run = 0;
  for (int c0 = 0; c0 < chunks; c0 += 32) {
    const int c = c0 + lane;
    const int v = c < chunks ? hist[static_cast<size_t>(c) * nbuckets + bucket] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (c < chunks) hist[static_cast<size_t>(c) * nbuckets + bucket] = run + incl - v;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    (fwd ? p.bucket_fwd : p.bucket_bwd)[bucket] = run;
    if (run > 0) atomicMax(&p.header[kHdrMaxCost], bucket);
  }
}

// Bucket starts in descending cost: start[c] = sum of totals of costs > c.
__global__ void __launch_bounds__(kScanThreads) wl_scan_buckets(int nbuckets, WlPtrs p) {
  __shared__ int s_sum[kScanThreads];
  int* tot = blockIdx.x == 0 ? p.bucket_fwd : p.bucket_bwd;
  const int tid = threadIdx.x;
  const int per = (nbuckets + kScanThreads - 1) / kScanThreads;
  // position j in descending order is bucket nbuckets-1-j
  const int j0 = min(tid * per, nbuckets), j1 = min(j0 + per, nbuckets);
  int loc = 0;
  for (int j = j0; j < j1; ++j) loc += tot[nbuckets - 1 - j];
  s_sum[tid] = loc;
  __syncthreads();
  for (int off = 1; off < kScanThreads; off <<= 1) {
    int a = tid >= off ? s_sum[tid - off] : 0;
    __syncthreads();
    s_sum[tid] += a;
    __syncthreads();
  }
  int run = s_sum[tid] - loc;
  for (int j = j0; j < j1; ++j) {
    const int v = tot[nbuckets - 1 - j];
    tot[nbuckets - 1 - j] = run;
    run += v;
  }
  __syncthreads();
  if (tid == 0) {
    // tile list: items of cost >= 2 (they end where cost 1 starts) and the
    // long cost-1 items
    const bool fwd = blockIdx.x == 0;
    const int cap = p.header[fwd ? kHdrCapFwd : kHdrCapBwd];
    p.header[fwd ? kHdrTileFwd : kHdrTileBwd] =
        min(tot[1] + p.header[fwd ? kHdrLong1Fwd : kHdrLong1Bwd], cap);
  }
}

// Stable scatter of one chunk: rank among equal costs inside the chunk is
// taken warp by warp in order.
__global__ void __launch_bounds__(kSortChunk)
    wl_scatter(const int32_t* __restrict__ cu, int ndocs, int chunks_fwd, int nbuckets, WlPtrs p) {
  extern __shared__ int s_cnt[];
  const bool fwd = blockIdx.x < chunks_fwd;
  const int chunk = fwd ? blockIdx.x : blockIdx.x - chunks_fwd;
  const int n = p.header[fwd ? kHdrNFwd : kHdrNBwd];
  const int cap = p.header[fwd ? kHdrCapFwd : kHdrCapBwd];
  const int4* gen = fwd ? p.gen_fwd : p.gen_bwd;
  int4* out = fwd ? p.fwd : p.bwd;
  int4* tile = fwd ? p.tile_fwd : p.tile_bwd;
  const int* hist = (fwd ? p.hist_fwd : p.hist_bwd) + static_cast<size_t>(chunk) * nbuckets;
  const int* start = fwd ? p.bucket_fwd : p.bucket_bwd;
  for (int i = threadIdx.x; i < nbuckets; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  const int g = chunk * kSortChunk + threadIdx.x;
  const bool have = g < n;
  int4 it = have ? gen[g] : make_int4(0, 0, 0, 0);
  const int c = have ? min(it.w, nbuckets - 1) : -1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned peers = __match_any_sync(0xffffffffu, c);
  const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
  const bool leader = rank_in_warp == 0;
  // position in the tile list (-1: an item of a short document)
  int tpos = -1;
  if (have) {
    if (c >= 2) {
      tpos = -2;  // same position as in the full list
    } else {
      const int b = it.x;
      const int L = cu[b + 1] - cu[b];
      if (L > kShortDoc) {
        const int l = fwd ? kCntLongFwd : kCntLongBwd;
        const int ndchunks = (ndocs + kScanThreads - 1) / kScanThreads;
        tpos = start[1] + p.offsets[l * ndchunks + b / kScanThreads] + p.counts[l * ndocs + b];
      }
    }
  }
  for (int w = 0; w < kSortChunk / 32; ++w) {
    if (warp == w && have) {
      const int pos = start[c] + hist[c] + s_cnt[c] + rank_in_warp;
      out[pos] = it;
      const int tp = tpos == -2 ? pos : tpos;
      if (tp >= 0 && tp < cap) tile[tp] = it;
    }
    __syncthreads();
    if (warp == w && have && leader) s_cnt[c] += __popc(peers);
    __syncthreads();
  }
}

// The six launches of one build; returns FLAMIA_ERR_CUDA if the shared-memory
// opt-in or a launch fails.
flamia_status launch_builder(const int32_t* cu_seqlens, int ndocs, int T,
                             const WorklistLayout& L, const WlPtrs& p, int* dev_status,
                             cudaStream_t s) {
  const size_t smem = static_cast<size_t>(L.nbuckets) * sizeof(int);
  if (smem > 200 * 1024) return FLAMIA_ERR_UNSUPPORTED;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(wl_emit, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(wl_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return FLAMIA_ERR_CUDA;
  }
  const int ndchunks = (ndocs + kScanThreads - 1) / kScanThreads;
  wl_count<<<ndchunks, kScanThreads, 0, s>>>(cu_seqlens, ndocs, T, p, dev_status);
  wl_scan_docs<<<1, kScanThreads, 0, s>>>(ndchunks, L.cap_fwd, L.cap_bwd, p, dev_status);
  wl_emit<<<L.chunks_fwd + L.chunks_bwd, kSortChunk, smem, s>>>(cu_seqlens, ndocs, L.chunks_fwd,
                                                               L.nbuckets, p);
  wl_scan_chunks<<<(2 * L.nbuckets * 32 + 255) / 256, 256, 0, s>>>(L.nbuckets, L.chunks_fwd,
                                                                   L.chunks_bwd, p);
  wl_scan_buckets<<<2, kScanThreads, 0, s>>>(L.nbuckets, p);
  wl_scatter<<<L.chunks_fwd + L.chunks_bwd, kSortChunk, smem, s>>>(cu_seqlens, ndocs, L.chunks_fwd,
                                                                  L.nbuckets, p);
  count_launches(6);
  return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

}  // namespace
}  // namespace flamia

using namespace flamia;

extern "C" size_t flamia_worklist_bytes(int T, int ndocs) {
  if (T <= 0 || ndocs <= 0) return 0;
  return worklist_layout(T, ndocs).total;
}

extern "C" flamia_status flamia_build_worklist(const int32_t* cu_seqlens, int ndocs, int T,
                                               void* wl, size_t wl_bytes, int* dev_status,
                                               void* stream) {
  if (cu_seqlens == nullptr || wl == nullptr || T <= 0 || ndocs <= 0 || ndocs > T + 1 ||
      T > kMaxTokens)
    return FLAMIA_ERR_INVALID_ARG;
  if (!aligned(wl, 256)) return FLAMIA_ERR_INVALID_ARG;
  const WorklistLayout L = worklist_layout(T, ndocs);
  if (wl_bytes < L.total) return FLAMIA_ERR_WORKSPACE;
  char* base = static_cast<char*>(wl);
  WlPtrs p;
  p.header = reinterpret_cast<int*>(base);
  p.fwd = reinterpret_cast<int4*>(base + L.off_fwd);
  p.bwd = reinterpret_cast<int4*>(base + L.off_bwd);
  p.tile_fwd = reinterpret_cast<int4*>(base + L.off_tile_fwd);
  p.tile_bwd = reinterpret_cast<int4*>(base + L.off_tile_bwd);
  p.counts = reinterpret_cast<int*>(base + L.off_doc_counts);
  p.offsets = reinterpret_cast<int*>(base + L.off_doc_offsets);
  p.gen_fwd = reinterpret_cast<int4*>(base + L.off_gen_fwd);
  p.gen_bwd = reinterpret_cast<int4*>(base + L.off_gen_bwd);
  p.hist_fwd = reinterpret_cast<int*>(base + L.off_hist_fwd);
  p.hist_bwd = reinterpret_cast<int*>(base + L.off_hist_bwd);
  p.bucket_fwd = reinterpret_cast<int*>(base + L.off_buckets);
  p.bucket_bwd = p.bucket_fwd + L.nbuckets;
  return launch_builder(cu_seqlens, ndocs, T, L, p, dev_status,
                        static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the work-list builder.
//
// Some callers cannot allocate device memory for the builder's scratch: a
// framework whose caching allocator owns the device memory and hands the
// library only the output tensors, a plugin host that gives the library no
// allocator at all, or a latency-critical loop where the implicit device
// synchronisation of cudaMalloc / cudaFree is not acceptable.  This entry point
// keeps the scratch (per-document counts and offsets, items in generation
// order, per-chunk cost histograms, bucket starts) in a fixed array in the
// library's own device memory instead.
namespace flamia {
namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB per GPU, held until exit
static __device__ __align__(256) unsigned char g_wl_scratch[kStaticScratchBytes];

// Device address of g_wl_scratch in the current context.  The name is only a
// host-side stand-in; the address belongs to the module instance loaded in one
// CUDA context, so it is cached per context under the context's unique ID
// (cuCtxGetId: never reused within a process, unlike a context handle), and a
// context created after cudaDeviceReset looks the address up afresh.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

std::mutex g_scratch_mu;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
std::vector<ScratchEntry> g_scratch_addr;

template <typename Fn>
Fn driver_entry(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// The unique ID of the calling thread's current context (0 if there is none).
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = driver_entry<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_entry<CtxGetIdFn>("cuCtxGetId");
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
      ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

void* static_scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = current_context_id();
  for (const ScratchEntry& e : g_scratch_addr)
    if (id != 0 && e.ctx_id == id) return e.addr;
  // first call in this context: the lookup also makes the runtime's primary
  // context current if no context was current yet
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_wl_scratch) != cudaSuccess || p == nullptr) return nullptr;
  id = current_context_id();
  if (id != 0) g_scratch_addr.push_back({id, p});
  return p;
}

}  // namespace
}  // namespace flamia

extern "C" flamia_status flamia_build_worklist_static(const int32_t* cu_seqlens, int ndocs,
                                                      int T, void* wl, size_t wl_bytes,
                                                      int* dev_status, void* stream) {
  if (cu_seqlens == nullptr || wl == nullptr || T <= 0 || ndocs <= 0 || ndocs > T + 1 ||
      T > kMaxTokens)
    return FLAMIA_ERR_INVALID_ARG;
  if (!aligned(wl, 256)) return FLAMIA_ERR_INVALID_ARG;
  const WorklistLayout L = worklist_layout(T, ndocs);
  // the caller's buffer holds the header, both item arrays and both tile lists
  if (wl_bytes < L.off_doc_counts) return FLAMIA_ERR_WORKSPACE;
  // everything after the tile lists lives in the static scratch
  if (L.total - L.off_doc_counts > kStaticScratchBytes) return FLAMIA_ERR_WORKSPACE;
  char* scratch = static_cast<char*>(static_scratch_address());
  if (scratch == nullptr) return FLAMIA_ERR_CUDA;
  char* base = static_cast<char*>(wl);
  // scratch keeps the layout's spacing, shifted to the start of the array
  auto at = [&](size_t off) { return scratch + (off - L.off_doc_counts); };
  WlPtrs p;
  p.header = reinterpret_cast<int*>(base);
  p.fwd = reinterpret_cast<int4*>(base + L.off_fwd);
  p.bwd = reinterpret_cast<int4*>(base + L.off_bwd);
  p.tile_fwd = reinterpret_cast<int4*>(base + L.off_tile_fwd);
  p.tile_bwd = reinterpret_cast<int4*>(base + L.off_tile_bwd);
  p.counts = reinterpret_cast<int*>(at(L.off_doc_counts));
  p.offsets = reinterpret_cast<int*>(at(L.off_doc_offsets));
  p.gen_fwd = reinterpret_cast<int4*>(at(L.off_gen_fwd));
  p.gen_bwd = reinterpret_cast<int4*>(at(L.off_gen_bwd));
  p.hist_fwd = reinterpret_cast<int*>(at(L.off_hist_fwd));
  p.hist_bwd = reinterpret_cast<int*>(at(L.off_hist_bwd));
  p.bucket_fwd = reinterpret_cast<int*>(at(L.off_buckets));
  p.bucket_bwd = p.bucket_fwd + L.nbuckets;
  // Every buffer of scratch is fully written before it is read within one
  // call, so nothing left by an earlier call needs clearing.
  return launch_builder(cu_seqlens, ndocs, T, L, p, dev_status,
                        static_cast<cudaStream_t>(stream));
}
