// GPU work-list builder (FLAMIA review page, sec. 3.4 "Work scheduling").
//
// Forward items are 256-query chunks of a document (cost = 128-key blocks
// seen by the chunk's last query); backward items are 128-key tiles (cost =
// 128-query tiles that see them).  Both lists are sorted by descending cost,
// stable over generation order (document, then position), entirely on the
// device with no host synchronisation:
//   count per document -> exclusive scan -> emit in generation order with a
//   per-chunk cost histogram -> per-bucket scan over chunks -> scan over
//   buckets in descending cost -> stable scatter (rank inside a chunk).
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace flamia {
namespace {

constexpr int kScanThreads = 1024;

struct WlPtrs {
  int* header;
  int4* fwd;
  int4* bwd;
  int* counts;   // [2][ndocs]
  int* offsets;  // [2][ndocs]
  int4* gen_fwd;
  int4* gen_bwd;
  int* hist_fwd;  // [chunks][nbuckets]
  int* hist_bwd;
  int* bucket_fwd;  // [nbuckets] bucket totals, then bucket starts
  int* bucket_bwd;
};

__global__ void wl_count(const int32_t* __restrict__ cu, int ndocs, int T, WlPtrs p,
                         int* dev_status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0 && (cu[0] != 0 || cu[ndocs] != T)) report(dev_status, FLAMIA_DEV_BAD_SEQLENS);
  if (b >= ndocs) return;
  int L = cu[b + 1] - cu[b];
  if (L < 0) {
    report(dev_status, FLAMIA_DEV_BAD_SEQLENS);
    L = 0;
  }
  p.counts[b] = (L + kFwdItem - 1) / kFwdItem;
  p.counts[ndocs + b] = (L + kTile - 1) / kTile;
}

// Exclusive scan of both count arrays in one CTA; totals go to the header.
__global__ void __launch_bounds__(kScanThreads)
    wl_scan_docs(int ndocs, int cap_fwd, int cap_bwd, WlPtrs p, int* dev_status) {
  __shared__ int s_sum[2][kScanThreads];
  const int tid = threadIdx.x;
  const int per = (ndocs + kScanThreads - 1) / kScanThreads;
  const int b0 = min(tid * per, ndocs), b1 = min(b0 + per, ndocs);
  int loc[2] = {0, 0};
  for (int b = b0; b < b1; ++b) {
    loc[0] += p.counts[b];
    loc[1] += p.counts[ndocs + b];
  }
  s_sum[0][tid] = loc[0];
  s_sum[1][tid] = loc[1];
  __syncthreads();
  // Hillis-Steele inclusive scan over the 1024 partial sums.
  for (int off = 1; off < kScanThreads; off <<= 1) {
    int a0 = tid >= off ? s_sum[0][tid - off] : 0;
    int a1 = tid >= off ? s_sum[1][tid - off] : 0;
    __syncthreads();
    s_sum[0][tid] += a0;
    s_sum[1][tid] += a1;
    __syncthreads();
  }
  int run0 = s_sum[0][tid] - loc[0], run1 = s_sum[1][tid] - loc[1];
  for (int b = b0; b < b1; ++b) {
    p.offsets[b] = run0;
    p.offsets[ndocs + b] = run1;
    run0 += p.counts[b];
    run1 += p.counts[ndocs + b];
  }
  if (tid == kScanThreads - 1) {
    int nf = s_sum[0][tid], nb = s_sum[1][tid];
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

__device__ __forceinline__ int upper_doc(const int* __restrict__ off, int ndocs, int g) {
  // largest b with off[b] <= g (offsets are non-decreasing, off[0] == 0)
  int lo = 0, hi = ndocs;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= g) lo = mid;
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
  const int* off = p.offsets + (fwd ? 0 : ndocs);
  for (int i = threadIdx.x; i < nbuckets; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int g = chunk * kSortChunk + threadIdx.x;
  if (g < n) {
    const int b = upper_doc(off, ndocs, g);
    const int k = g - off[b];
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

// Per bucket: exclusive prefix over chunks (in place); bucket totals out.
__global__ void wl_scan_chunks(int nbuckets, int chunks_fwd, int chunks_bwd, WlPtrs p) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 2 * nbuckets) return;
  const bool fwd = i < nbuckets;
  const int bucket = fwd ? i : i - nbuckets;
  int* hist = fwd ? p.hist_fwd : p.hist_bwd;
  const int chunks = fwd ? chunks_fwd : chunks_bwd;
  int run = 0;
  for (int c = 0; c < chunks; ++c) {
    const int v = hist[static_cast<size_t>(c) * nbuckets + bucket];
    hist[static_cast<size_t>(c) * nbuckets + bucket] = run;
    run += v;
  }
  (fwd ? p.bucket_fwd : p.bucket_bwd)[bucket] = run;
  if (run > 0) atomicMax(&p.header[kHdrMaxCost], bucket);
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
}

// Stable scatter of one chunk: rank among equal costs inside the chunk is
// taken warp by warp in order.
__global__ void __launch_bounds__(kSortChunk)
    wl_scatter(int chunks_fwd, int nbuckets, WlPtrs p) {
  extern __shared__ int s_cnt[];
  const bool fwd = blockIdx.x < chunks_fwd;
  const int chunk = fwd ? blockIdx.x : blockIdx.x - chunks_fwd;
  const int n = p.header[fwd ? kHdrNFwd : kHdrNBwd];
  const int4* gen = fwd ? p.gen_fwd : p.gen_bwd;
  int4* out = fwd ? p.fwd : p.bwd;
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
  for (int w = 0; w < kSortChunk / 32; ++w) {
    if (warp == w && have) {
      const int pos = start[c] + hist[c] + s_cnt[c] + rank_in_warp;
      out[pos] = it;
    }
    __syncthreads();
    if (warp == w && have && leader) s_cnt[c] += __popc(peers);
    __syncthreads();
  }
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
      T > (1 << 20))
    return FLAMIA_ERR_INVALID_ARG;
  if (!aligned(wl, 256)) return FLAMIA_ERR_INVALID_ARG;
  const WorklistLayout L = worklist_layout(T, ndocs);
  if (wl_bytes < L.total) return FLAMIA_ERR_WORKSPACE;
  char* base = static_cast<char*>(wl);
  WlPtrs p;
  p.header = reinterpret_cast<int*>(base);
  p.fwd = reinterpret_cast<int4*>(base + L.off_fwd);
  p.bwd = reinterpret_cast<int4*>(base + L.off_bwd);
  p.counts = reinterpret_cast<int*>(base + L.off_doc_counts);
  p.offsets = reinterpret_cast<int*>(base + L.off_doc_offsets);
  p.gen_fwd = reinterpret_cast<int4*>(base + L.off_gen_fwd);
  p.gen_bwd = reinterpret_cast<int4*>(base + L.off_gen_bwd);
  p.hist_fwd = reinterpret_cast<int*>(base + L.off_hist_fwd);
  p.hist_bwd = reinterpret_cast<int*>(base + L.off_hist_bwd);
  p.bucket_fwd = reinterpret_cast<int*>(base + L.off_buckets);
  p.bucket_bwd = p.bucket_fwd + L.nbuckets;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t smem = static_cast<size_t>(L.nbuckets) * sizeof(int);
  if (smem > 200 * 1024) return FLAMIA_ERR_UNSUPPORTED;
  if (smem > 48 * 1024) {
    cudaFuncSetAttribute(wl_emit, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    cudaFuncSetAttribute(wl_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
  }
  wl_count<<<(ndocs + 255) / 256, 256, 0, s>>>(cu_seqlens, ndocs, T, p, dev_status);
  wl_scan_docs<<<1, kScanThreads, 0, s>>>(ndocs, L.cap_fwd, L.cap_bwd, p, dev_status);
  wl_emit<<<L.chunks_fwd + L.chunks_bwd, kSortChunk, smem, s>>>(cu_seqlens, ndocs, L.chunks_fwd,
                                                               L.nbuckets, p);
  wl_scan_chunks<<<(2 * L.nbuckets + 255) / 256, 256, 0, s>>>(L.nbuckets, L.chunks_fwd,
                                                              L.chunks_bwd, p);
  wl_scan_buckets<<<2, kScanThreads, 0, s>>>(L.nbuckets, p);
  wl_scatter<<<L.chunks_fwd + L.chunks_bwd, kSortChunk, smem, s>>>(L.chunks_fwd, L.nbuckets, p);
  return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
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

std::mutex g_scratch_mu;
void* g_scratch_addr[128] = {};

// Device address of g_wl_scratch on the current device (looked up once per
// device; the name is only a host-side stand-in).
void* static_scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wl_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace flamia

extern "C" flamia_status flamia_build_worklist_static(const int32_t* cu_seqlens, int ndocs,
                                                      int T, void* wl, size_t wl_bytes,
                                                      int* dev_status, void* stream) {
  if (cu_seqlens == nullptr || wl == nullptr || T <= 0 || ndocs <= 0 || ndocs > T + 1 ||
      T > (1 << 20))
    return FLAMIA_ERR_INVALID_ARG;
  if (!aligned(wl, 256)) return FLAMIA_ERR_INVALID_ARG;
  const WorklistLayout L = worklist_layout(T, ndocs);
  // the caller's buffer holds the header and both item arrays
  if (wl_bytes < L.off_doc_counts) return FLAMIA_ERR_WORKSPACE;
  // everything after the item arrays lives in the static scratch
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
  p.counts = reinterpret_cast<int*>(at(L.off_doc_counts));
  p.offsets = reinterpret_cast<int*>(at(L.off_doc_offsets));
  p.gen_fwd = reinterpret_cast<int4*>(at(L.off_gen_fwd));
  p.gen_bwd = reinterpret_cast<int4*>(at(L.off_gen_bwd));
  p.hist_fwd = reinterpret_cast<int*>(at(L.off_hist_fwd));
  p.hist_bwd = reinterpret_cast<int*>(at(L.off_hist_bwd));
  p.bucket_fwd = reinterpret_cast<int*>(at(L.off_buckets));
  p.bucket_bwd = p.bucket_fwd + L.nbuckets;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t smem = static_cast<size_t>(L.nbuckets) * sizeof(int);
  if (smem > 200 * 1024) return FLAMIA_ERR_UNSUPPORTED;
  if (smem > 48 * 1024) {
    cudaFuncSetAttribute(wl_emit, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    cudaFuncSetAttribute(wl_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
  }
  // Every buffer of scratch is fully written before it is read within one
  // call, so nothing left by an earlier call needs clearing.
  wl_count<<<(ndocs + 255) / 256, 256, 0, s>>>(cu_seqlens, ndocs, T, p, dev_status);
  wl_scan_docs<<<1, kScanThreads, 0, s>>>(ndocs, L.cap_fwd, L.cap_bwd, p, dev_status);
  wl_emit<<<L.chunks_fwd + L.chunks_bwd, kSortChunk, smem, s>>>(cu_seqlens, ndocs, L.chunks_fwd,
                                                               L.nbuckets, p);
  wl_scan_chunks<<<(2 * L.nbuckets + 255) / 256, 256, 0, s>>>(L.nbuckets, L.chunks_fwd,
                                                              L.chunks_bwd, p);
  wl_scan_buckets<<<2, kScanThreads, 0, s>>>(L.nbuckets, p);
  wl_scatter<<<L.chunks_fwd + L.chunks_bwd, kSortChunk, smem, s>>>(L.chunks_fwd, L.nbuckets, p);
  return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}
