// Host-side helpers shared by the entry points: argument checks, tensor-map
// encoding through the driver entry point (no link-time libcuda dependency),
// and the work-list buffer layout.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/flamia.h"

namespace flamia {

constexpr int kTile = 128;       // query / key tile (MMA M and N)
constexpr int kBlock = 32;       // token block of the scales
constexpr int kFwdItem = 256;    // queries per forward work item
// Documents of at most this many tokens (one 32-token scale block) run on the
// CUDA-core kernels of attn_short.cu; the tile kernels skip them.
constexpr int kShortDoc = 32;

// ------------------------------------------------------------------ work list

struct WorklistLayout {
  int cap_fwd, cap_bwd;        // item capacities
  int nbuckets;                // costs 0 .. nbuckets-1
  int chunks_fwd, chunks_bwd;  // 1024-item chunks of the counting sort
  size_t off_fwd, off_bwd;     // byte offsets of the sorted item arrays
  size_t off_tile_fwd, off_tile_bwd;  // the same lists without short-document items
  size_t off_doc_counts;       // int32 [4][ndocs]: in-chunk prefixes of 4 per-document counts
  size_t off_doc_offsets;      // int32 [4][doc chunks]: chunk totals, then chunk offsets
  size_t off_gen_fwd, off_gen_bwd;  // int4 items in generation order
  size_t off_hist_fwd, off_hist_bwd;  // int32 [chunks][nbuckets]
  size_t off_buckets;                 // int32 [2][nbuckets]
  size_t total;
};

constexpr int kSortChunk = 1024;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WorklistLayout worklist_layout(int T, int ndocs) {
  WorklistLayout L{};
  L.cap_fwd = T / kFwdItem + ndocs + 1;
  L.cap_bwd = T / kTile + ndocs + 1;
  L.nbuckets = (T + kTile - 1) / kTile + 2;
  L.chunks_fwd = (L.cap_fwd + kSortChunk - 1) / kSortChunk;
  L.chunks_bwd = (L.cap_bwd + kSortChunk - 1) / kSortChunk;
  size_t o = 64;  // header
  L.off_fwd = o;
  o = align_up(o + 16ull * L.cap_fwd, 256);
  L.off_bwd = o;
  o = align_up(o + 16ull * L.cap_bwd, 256);
  L.off_tile_fwd = o;
  o = align_up(o + 16ull * L.cap_fwd, 256);
  L.off_tile_bwd = o;
  o = align_up(o + 16ull * L.cap_bwd, 256);
  // everything below is the builder's scratch
  L.off_doc_counts = o;
  o = align_up(o + 16ull * (ndocs + 1), 256);
  L.off_doc_offsets = o;
  o = align_up(o + 16ull * ((ndocs + kSortChunk - 1) / kSortChunk + 1), 256);
  L.off_gen_fwd = o;
  o = align_up(o + 16ull * L.cap_fwd, 256);
  L.off_gen_bwd = o;
  o = align_up(o + 16ull * L.cap_bwd, 256);
  L.off_hist_fwd = o;
  o = align_up(o + 4ull * L.chunks_fwd * L.nbuckets, 256);
  L.off_hist_bwd = o;
  o = align_up(o + 4ull * L.chunks_bwd * L.nbuckets, 256);
  L.off_buckets = o;
  o = align_up(o + 8ull * L.nbuckets, 256);
  L.total = o;
  return L;
}

// Header words of the work-list buffer: list sizes and capacities, the
// largest cost, the sizes of the tile lists (items of documents longer than
// kShortDoc, which the tile kernels process), internal to the builder the
// number of documents with a long cost-1 item in each list, and the tile
// kernels' item claim counters.
enum : int {
  kHdrNFwd = 0,
  kHdrNBwd = 1,
  kHdrCapFwd = 2,
  kHdrCapBwd = 3,
  kHdrMaxCost = 4,
  kHdrTileFwd = 5,
  kHdrTileBwd = 6,
  kHdrLong1Fwd = 7,
  kHdrLong1Bwd = 8,
  // claim counters of the forward / backward tile kernels and their CTA exit
  // counts; zero after the build and after every launch
  kHdrFwdNext = 9,
  kHdrFwdExit = 10,
  kHdrBwdNext = 11,
  kHdrBwdExit = 12
};

// ------------------------------------------------------------------ checks

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline bool supported_dim(int d) { return d == 64 || d == 128; }

// Largest packed token count of a call.  The work-list builder's per-chunk
// cost histograms grow with T^2 (chunks x cost buckets), which sets this one
// limit for every entry point.
constexpr int kMaxTokens = 1 << 20;

// Sizes the kernels index safely: token x head counts fit an int (per-row
// tables and counters are indexed by token * H + head in 32 bits), elements
// in 40 bits (64-bit offsets everywhere else).
inline bool valid_sizes(int T, int H, int d, int ndocs) {
  return T > 0 && T <= kMaxTokens && H > 0 && H <= 4096 && ndocs >= 1 && ndocs <= T + 1 &&
         static_cast<long long>(T) * H < (1ll << 31) &&
         static_cast<long long>(T) * H * d < (1ll << 40) && supported_dim(d);
}

// Kernel launches enqueued by the library since it was loaded (all entry
// points, all threads); each launch site adds its count after enqueuing.
void count_launches(int n);  // defined in abi.cu

// Streaming multiprocessors of the current device (persistent grids).
inline int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// ------------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_tiled();  // defined in abi.cu

// A [rows][row_bytes] byte matrix inside a [T, H, row_bytes] packed tensor,
// seen as 3-D (inner bytes, head, token); box = (row_bytes, 1, box_rows).
inline bool make_token_map(CUtensorMap* map, const void* base, int T, int H, int row_bytes,
                           int box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes),
                           static_cast<cuuint64_t>(row_bytes) * H};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(row_bytes), 1u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same [T, H, row_bytes] byte tensor with a box of box_bytes of a row
// (a column slice of the head dimension) x box_rows tokens of one head.
inline bool make_token_slice_map(CUtensorMap* map, const void* base, int T, int H, int row_bytes,
                                 int box_bytes, int box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes),
                           static_cast<cuuint64_t>(row_bytes) * H};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_bytes), 1u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A plain [rows][row_bytes] byte matrix; box = (row_bytes, box_rows).
inline bool make_matrix_map(CUtensorMap* map, const void* base, int rows, int row_bytes,
                            int box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A float32 [T, H, d] tensor seen as 3-D (dim, head, token); box = (32, 1,
// box_rows) with 128-byte swizzle (one 128-byte row of 32 floats per token).
inline bool make_f32_token_map(CUtensorMap* map, const void* base, int T, int H, int d,
                               int box_rows,
                               CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(d) * 4 * H};
  cuuint32_t box[3] = {32u, 1u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same [T, H, d] layout with FP16 elements; box = 64 elements (128 bytes)
// x box_rows tokens of one head.
inline bool make_f16_token_map(CUtensorMap* map, const void* base, int T, int H, int d,
                               int box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(d) * 2 * H};
  cuuint32_t box[3] = {64u, 1u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The work distribution a call's flags ask for: 0 dynamic (default), 1 the
// pages' rule, 2 static; -1 if both flags were given.
inline int schedule_of(int flags) {
  const bool st = (flags & FLAMIA_FLAG_SCHEDULE_STATIC) != 0;
  const bool ru = (flags & FLAMIA_FLAG_SCHEDULE_RULE) != 0;
  return st && ru ? -1 : st ? 2 : ru ? 1 : 0;
}

inline CUtensorMapSwizzle swizzle_for_row_bytes(int row_bytes) {
  return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
         : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                           : CU_TENSOR_MAP_SWIZZLE_32B;
}

}  // namespace flamia
