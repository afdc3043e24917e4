/*
 * flamia.h -- C ABI of the token-block microscaled (MXFP8) causal flash
 * attention hot path for one GB300 (sm_103a) GPU.
 *
 * The method is the one described in "FLAMIA: FLAsh MIcroscaling Attention
 * for Fast and Causally Safe Training on Blackwell" (review page
 * jaehun.me/en/posts/paper-2611-03344v1, sections cited per entry point; and
 * the summary page agihunt.info/en/papers/2611.03344).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Packed layout.  Documents are concatenated along the token axis.  A tensor
 *   "[T, H, d]" is row-major (token, head, dim) with no padding.
 *   cu_seqlens is int32[ndocs + 1] in DEVICE memory: document b is tokens
 *   [cu_seqlens[b], cu_seqlens[b+1]); cu_seqlens[0] == 0, cu_seqlens[ndocs]
 *   == T, non-decreasing (empty documents are allowed).
 * - Ownership.  Every pointer argument is a DEVICE pointer owned by the caller
 *   unless stated otherwise.  The library never allocates, frees or
 *   synchronises, and never reads device data on the host.  All work is
 *   enqueued on `stream` (a cudaStream_t, NULL = legacy default stream).
 * - Errors.  Argument errors found on the host return a flamia_status and
 *   enqueue nothing.  Errors found on the device (malformed cu_seqlens,
 *   capacity overflow, a bounded wait that timed out) are OR-ed into the
 *   int at `dev_status` (device memory, may be NULL to ignore) as
 *   FLAMIA_DEV_* bits; read it after synchronising the stream.  No kernel
 *   traps or spins without bound.
 * - Support.  head_dim d in {64, 128}; 1 <= H <= 4096; T <= 2^20 tokens,
 *   T * H < 2^31, T * H * d < 2^40; multi-head attention, and grouped K / V
 *   heads through the _gqa entry points; causal masking, or none with
 *   FLAMIA_FLAG_NONCAUSAL.  Larger sizes return FLAMIA_ERR_INVALID_ARG.
 * - Formats.  E4M3 = OCP FP8 E4M3FN (bias 7, max 448, subnormals kept).
 *   E8M0 = 2^(byte - 127).  E2M1 = {0, .5, 1, 1.5, 2, 3, 4, 6} with sign,
 *   two codes per byte, element 2i in the low nibble.
 */
#ifndef FLAMIA_H
#define FLAMIA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLAMIA_OK = 0,
  FLAMIA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer      */
  FLAMIA_ERR_UNSUPPORTED = 2,   /* d not in {64,128}, unknown format or flag      */
  FLAMIA_ERR_WORKSPACE = 3,     /* workspace / work-list buffer too small         */
  FLAMIA_ERR_CUDA = 4           /* a CUDA runtime call failed (launch, memset)    */
} flamia_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define FLAMIA_DEV_BAD_SEQLENS 0x1  /* cu_seqlens not monotone or not ending at T */
#define FLAMIA_DEV_CAPACITY    0x2  /* more work items than the buffer holds      */
#define FLAMIA_DEV_TIMEOUT     0x4  /* a bounded wait gave up; outputs invalid    */
#define FLAMIA_DEV_RANGE       0x8  /* a scale exponent left the E8M0 range a mode
                                       supports (per-token operand scales with
                                       |V| near 2^96 or beyond); outputs invalid */

/* Quantiser output formats. */
#define FLAMIA_FORMAT_MXFP8       0 /* E4M3 codes + per-token E8M0 scales          */
#define FLAMIA_FORMAT_MXFP8_NVFP4 1 /* the above plus NVFP4 codes and scales       */
#define FLAMIA_FORMAT_HADAMARD 0x10 /* OR-ed into FLAMIA_FORMAT_MXFP8: rotate each
                                       (token, head) row by H_d before the block
                                       statistics (for Q and K; see below)       */
#define FLAMIA_FORMAT_TOKEN_SCALES 0x20 /* OR-ed into FLAMIA_FORMAT_MXFP8 (with or
                                       without FLAMIA_FORMAT_HADAMARD): one
                                       exponent per (token, head) instead of per
                                       32-token block (per-token operand scales,
                                       see FLAMIA_FLAG_TOKEN_SCALES)             */

/* Attention flags. */
#define FLAMIA_FLAG_NVFP4_QK 0x1    /* score product QK^T (fwd and bwd recompute)
                                       from the NVFP4 copy of Q and K (d == 64)   */
#define FLAMIA_FLAG_NONCAUSAL 0x4   /* every query sees every key of its own
                                       document (no causal mask)                 */
#define FLAMIA_FLAG_HADAMARD 0x2    /* q and k were quantised with
                                       FLAMIA_FORMAT_HADAMARD: scores use
                                       softmax_scale / d; the backward returns
                                       dQ and dK rotated back by H_d            */
#define FLAMIA_FLAG_DETERMINISTIC_DQ 0x8 /* backward only: the float32 dQ
                                       partials of a query tile are added in
                                       a fixed key-tile order, so dQ is the
                                       same bit for bit on every run            */
#define FLAMIA_FLAG_DQ_FP16 0x10    /* backward only: dQ partials reduce-added
                                       in FP16 behind a power-of-two prescale
                                       from sequence-wide maxima                */
#define FLAMIA_FLAG_DQ_CAUSAL_SCALE 0x20 /* with FLAMIA_FLAG_DQ_FP16: the prescale
                                       of a query row from the keys it sees     */
#define FLAMIA_FLAG_SCHEDULE_STATIC 0x40 /* forward / backward: the persistent CTAs
                                       take their work items in a static snake
                                       over the cost-sorted list instead of
                                       claiming the next unclaimed item        */
#define FLAMIA_FLAG_DS_ROW_EXPONENTS 0x100 /* backward only: dQ's dS
                                       operand rounded with one exponent per
                                       (query row, 32-key block) instead of per
                                       32 x 32 block (dK keeps the block ones) */
#define FLAMIA_FLAG_TOKEN_SCALES 0x200 /* forward / backward: q, k, v and dout were
                                       quantised with FLAMIA_FORMAT_TOKEN_SCALES
                                       (one exponent per token); the per-token
                                       factors along each contraction are folded
                                       into the opposite operand before its E4M3
                                       rounding (see the forward and backward);
                                       the backward implies
                                       FLAMIA_FLAG_DS_ROW_EXPONENTS.  Not with
                                       FLAMIA_FLAG_NVFP4_QK                      */
#define FLAMIA_FLAG_DS_ZERO_COUNT 0x400 /* backward only: count, over every pair
                                       a query sees, the dS entries that are
                                       nonzero and, of those, the ones whose
                                       E4M3 code under the 32 x 32 block exponent
                                       is zero (rounded to zero), into two uint64
                                       at flamia_bwd_ds_counts_offset of the
                                       workspace (cleared by the call); not with
                                       FLAMIA_FLAG_DETERMINISTIC_DQ or
                                       FLAMIA_FLAG_DQ_FP16                       */
#define FLAMIA_FLAG_SCHEDULE_RULE 0x80 /* forward / backward: the pages' rule,
                                       dynamic claims for causal calls and, for
                                       non-causal ones, only when the longest
                                       document is at least 4x the average
                                       (static snake otherwise).  Default, no
                                       flag: dynamic claims (measured fastest
                                       on every workload here)                 */
#define FLAMIA_FLAG_BWD_CTA_PAIR 0x800 /* backward only, head dim 128: the
                                       2-CTA mode (review page sec. 3.4
                                       "Backward pass"): clusters of two CTAs,
                                       each pair splitting 256 keys and running
                                       its products together; FLAMIA_ERR_
                                       UNSUPPORTED with the NVFP4 path,
                                       FLAMIA_FLAG_DETERMINISTIC_DQ,
                                       FLAMIA_FLAG_DQ_FP16, query-row dS
                                       exponents, per-token scales, the dS
                                       diagnostic or a static schedule          */
#define FLAMIA_FLAG_BWD_ONE_CTA 0x1000 /* backward only: one CTA per 128-key
                                       tile.  With neither flag the backward
                                       takes the measured rule, which picks
                                       one-CTA items on every shape (the pair
                                       measured about 1.5x slower on the
                                       packed 4 x 4096 and variable-length
                                       workloads)                              */

/*
 * One quantised operand, all device pointers owned by the caller.
 *  codes        u8  [T, H, d]     E4M3 codes.
 *  scales       u8  [H, T]        E8M0 byte of each token's 32-token block
 *                                 (dense: one entry per token and head).
 *  nvfp4_codes  u8  [T, H, d/2]   packed E2M1 (NULL unless NVFP4 requested).
 *  nvfp4_scales u8  [T, H, d/16]  E4M3 scale of each 16-element group (NULL
 *                                 unless NVFP4 requested).
 * codes and nvfp4_codes must be 16-byte aligned.
 */
typedef struct {
  uint8_t* codes;
  uint8_t* scales;
  uint8_t* nvfp4_codes;
  uint8_t* nvfp4_scales;
} flamia_qtensor;

/*
 * Fused token-block quantiser.
 * Source: review page sec. 3.1 (one power-of-two exponent per 32 consecutive
 * tokens x the full head dimension, E4M3 codes; the scale is constant along
 * the head dimension, so the payload serves K-major and MN-major products),
 * sec. 3.2 (exponent rounded up: the scaled block maximum never exceeds 448),
 * sec. 3.4 "Quantization fusion" (statistics, codes and scales in one launch)
 * and "Packed documents" (blocks never cross a document; dense per-token
 * scale table).  Blocks of document [s, e) are [s + 32i, min(s + 32i + 32, e)).
 * Exponent: smallest e with amax <= 448 * 2^e, clamped to [-127, 127]
 * (amax == 0 -> -127); codes = RNE_E4M3(x * 2^-e); scale byte = e + 127.
 * With format FLAMIA_FORMAT_MXFP8_NVFP4 the same pass also writes the NVFP4
 * copy (sec. 3.1 mixed path): per token and 16-element group, scale = the
 * smallest E4M3 value >= amax / 6, codes = RNE_E2M1(x / scale).
 * With FLAMIA_FORMAT_HADAMARD (sec. 3.4 "Hadamard rotation": the head-dim
 * channels of Q and K are mixed by an orthogonal transform inside the
 * quantiser) each row x is first replaced by x H_d, H_d the unnormalised
 * Sylvester-Hadamard matrix (entries +-1, H_d H_d = d I), computed in float32
 * by butterflies of stride 1, 2, .., d/2 in that order; the statistics and
 * codes are those of the rotated rows.  Not combinable with the NVFP4 copy
 * (FLAMIA_ERR_UNSUPPORTED) nor with o_bf16 / D.
 *
 *  x_bf16     [T, H, d] BF16 input (finite values).
 *  o_bf16, D  optional (both NULL or both set): the forward output O [T, H, d]
 *             BF16 and D float [H, T] = sum_k dequant(x)[t,h,k] * O[t,h,k]
 *             (review sec. 3.3: D from the same quantised dO used for dP).
 *  out        host pointer to a flamia_qtensor naming the caller's buffers.
 */
flamia_status flamia_quantize_tokenblock(const void* x_bf16, int T, int H, int d,
                                         const int32_t* cu_seqlens, int ndocs, int format,
                                         const void* o_bf16, float* D,
                                         const flamia_qtensor* out, int* dev_status,
                                         void* stream);

/*
 * Q, K and V of one call quantised by one launch (review page, sec. 3.4
 * "Quantization fusion": one pass per operand; one launch for the three
 * fills the GPU for longer and pays one tail).  The results are bit for bit
 * those of flamia_quantize_tokenblock on q with format_qk (H heads), on k
 * with format_qk (H_kv heads) and on v with FLAMIA_FORMAT_MXFP8 (H_kv heads).
 * format_qk: FLAMIA_FORMAT_MXFP8, FLAMIA_FORMAT_MXFP8_NVFP4 or
 * FLAMIA_FORMAT_MXFP8 | FLAMIA_FORMAT_HADAMARD (then V, never rotated, takes
 * a second launch).  q_bf16 [T, H, d], k_bf16 and v_bf16 [T, H_kv, d];
 * H_kv divides H.  Errors as for flamia_quantize_tokenblock.
 */
flamia_status flamia_quantize_qkv(const void* q_bf16, const void* k_bf16, const void* v_bf16,
                                  int T, int H, int H_kv, int d, const int32_t* cu_seqlens,
                                  int ndocs, int format_qk, const flamia_qtensor* q,
                                  const flamia_qtensor* k, const flamia_qtensor* v,
                                  int* dev_status, void* stream);

/*
 * Work list.  Source: review page sec. 3.4 "Work scheduling": a forward item
 * is 256 consecutive queries of one document (two 128-query tiles), its cost
 * the number of 128-key blocks it visits; items are sorted by descending
 * cost, built on the GPU once per micro-batch without a host sync.  The
 * backward items are 128-key tiles costed by the 128-query tiles that see
 * them.  Ties keep generation order (document, then position).
 *
 * Buffer layout (device, caller-owned, flamia_worklist_bytes(T, ndocs) bytes,
 * 256-byte aligned):
 *   int32 header[16]: [0] n_fwd, [1] n_bwd, [2] cap_fwd, [3] cap_bwd,
 *                     [4] max cost, [5] n_tile_fwd, [6] n_tile_bwd;
 *                     [7], [8] used by the builder; [9] .. [12] item claim
 *                     counters of the attention kernels (zero between
 *                     calls); the rest reserved.
 *   int32x4 fwd_items[cap_fwd] at byte 64: {doc, q_start, q_end, cost}
 *   int32x4 bwd_items[cap_bwd] after it:    {doc, k_start, k_end, cost}
 *   int32x4 tile_fwd[cap_fwd], tile_bwd[cap_bwd] after them: the same two
 *     lists without the items of documents of at most 32 tokens (n_tile_*
 *     entries each); the tensor-core kernels walk these, while documents of
 *     one 32-token block run on a CUDA-core kernel that needs no list.
 *   followed by the builder's scratch.
 * Each array starts on a 256-byte boundary.
 * cap_fwd = T/256 + ndocs + 1, cap_bwd = T/128 + ndocs + 1 (upper bounds).
 */
size_t flamia_worklist_bytes(int T, int ndocs);
flamia_status flamia_build_worklist(const int32_t* cu_seqlens, int ndocs, int T,
                                    void* wl, size_t wl_bytes, int* dev_status,
                                    void* stream);

/*
 * Work list without any device allocation, for callers that cannot allocate:
 * a framework whose caching allocator owns the device memory and hands the
 * library only its output tensors, a plugin host that gives the library no
 * allocator, or a latency-critical loop that cannot afford the implicit device
 * synchronisation of cudaMalloc / cudaFree.  The paper has no counterpart:
 * it is a convenience of this library's interface.
 *
 * Same inputs and the same output as flamia_build_worklist, but `wl` only
 * needs the header and the four item arrays (the layout above up to the end
 * of tile_bwd; a flamia_worklist_bytes-sized buffer always suffices).  The
 * builder's scratch lives in an 8 MiB array in the library's own device
 * memory, allocated on every GPU that loads the library and held until the
 * process exits.  The scratch grows mainly with the number of documents: any
 * document mix of up to 131,072 tokens fits, and at the 1,048,576-token
 * maximum up to 65,536 documents do; a layout whose scratch would exceed
 * 8 MiB returns FLAMIA_ERR_WORKSPACE without launching.
 * No cudaMalloc / cudaFree is called.  The first call in a CUDA context (with
 * its device current) looks up the array's device address and caches it under
 * the context's unique ID; make that first call before any stream capture.  A
 * context created later (after cudaDeviceReset, say) looks it up again.  All calls share the one array:
 * calls whose kernels overlap on the GPU (different streams, or different
 * host threads without ordering) race and produce garbage; serialise them.
 * Nothing left in the array by an earlier call is read by a later one.
 */
flamia_status flamia_build_worklist_static(const int32_t* cu_seqlens, int ndocs, int T,
                                           void* wl, size_t wl_bytes, int* dev_status,
                                           void* stream);

/*
 * Causal forward.  Source: review page sec. 1.2 (S = QK^T scale, P =
 * softmax(S), O = PV, row statistics saved), sec. 3.1 (unscaled E4M3 product
 * for QK^T with the query factor folded into the softmax scale and the key
 * factor applied separately; E4M3 probability operand; BF16 output), sec. 3.4
 * "Packed documents" (outputs written in place to the packed buffer).
 * Numerics: s_ij = scale * log2(e) * 2^eQ(i) * 2^eK(j) * <q_i, k_j> (codes),
 * running integer row maximum m_i = ceil(max_j s_ij), P~ = exp2(s - m),
 * l = sum P~, operand P^ = RNE_E4M3(2^8 P~), O = 2^-8 sum_j P^ V^_j / l,
 * LSE = (m + log2 l) ln 2.
 * FLAMIA_FLAG_HADAMARD: q and k hold Q H_d and K H_d, so the call uses
 * softmax_scale / d for the scores (the same S exactly, d a power of two).
 * Not combinable with FLAMIA_FLAG_NVFP4_QK.
 * FLAMIA_FLAG_NONCAUSAL (review page sec. 4.8, the non-causal packed call):
 * every query sees every key of its own document; the same numerics, the
 * same work list (its costs are the causal ones: only the order of the items
 * follows from them).
 *
 *  q, k, v      host pointers to quantised operands (E4M3 + scales; with
 *               FLAMIA_FLAG_NVFP4_QK also the NVFP4 copies of q and k).
 *  wl           a work list built for the same cu_seqlens / T.  Items are
 *               claimed dynamically in list order (longest first, sec. 3.4:
 *               the paper's dynamic assignment for causal calls) through a
 *               counter in the list's header, which the call updates and
 *               resets before it ends; calls that share one work list must
 *               not run at the same time (a forward and a backward may).
 *  o_bf16       [T, H, d] BF16 output.   lse  float [H, T] (natural log).
 * Only tokens inside documents are written.
 */
flamia_status flamia_attn_fwd(const flamia_qtensor* q, const flamia_qtensor* k,
                              const flamia_qtensor* v, const int32_t* cu_seqlens, int ndocs,
                              int T, int H, int d, float softmax_scale, int flags,
                              void* wl, void* o_bf16, float* lse, int* dev_status,
                              void* stream);

/*
 * Grouped-query attention: k and v carry H_kv heads (H_kv divides H); query
 * head h reads K / V head h / (H / H_kv).  k, v codes [T, H_kv, d], scales
 * [H_kv, T]; q, o [T, H, d]; lse [H, T].  flamia_attn_fwd is this call with
 * H_kv = H.  FLAMIA_ERR_INVALID_ARG if H_kv does not divide H.
 */
flamia_status flamia_attn_fwd_gqa(const flamia_qtensor* q, const flamia_qtensor* k,
                                  const flamia_qtensor* v, const int32_t* cu_seqlens, int ndocs,
                                  int T, int H, int H_kv, int d, float softmax_scale, int flags,
                                  void* wl, void* o_bf16, float* lse, int* dev_status,
                                  void* stream);

/*
 * Workspace of the forward: 0 bytes for every size (the review page, sec.
 * 3.4, keeps the forward's running statistics and P^ on chip; O and LSE are
 * its outputs).  Kept so that a caller sizes both calls the same way;
 * returns 0 also for unsupported sizes.
 */
size_t flamia_fwd_workspace_bytes(int T, int H, int d);

/*
 * Workspace of the backward, each part padded to 256 bytes: a float32
 * [T, H, d] dQ accumulator (FLAMIA_FLAG_DQ_FP16 uses its first half as an
 * FP16 [T, H, d] one), an int32 [T, H] array of turn counters
 * (FLAMIA_FLAG_DETERMINISTIC_DQ), the int8 [H, T] prescale exponents of the
 * FP16 accumulator, 3 H ints of scratch and the two dS counters
 * (FLAMIA_FLAG_DS_ZERO_COUNT).  The caller allocates it; the
 * backward clears what it uses itself.
 */
size_t flamia_bwd_workspace_bytes(int T, int H, int d);

/*
 * Byte offset, inside the backward workspace, of the two uint64 counters that
 * FLAMIA_FLAG_DS_ZERO_COUNT fills: [0] nonzero dS entries among the pairs the
 * queries see, [1] those of them whose E4M3 code in the 32 x 32 block payload
 * is zero.  The review page (sec. 3.3, and the dS-scale ablation of sec. 4)
 * takes this fraction as the sign of a badly set dS scale.  Read it after the
 * backward has completed.  0 for unsupported sizes.
 */
size_t flamia_bwd_ds_counts_offset(int T, int H, int d);

/*
 * Causal backward.  Source: review page sec. 1.2 (recompute P; dV = P^T dO,
 * dP = dO V^T, dS = P o (dP - D), dQ = dS K, dK = dS^T Q), sec. 3.3 (the
 * recompute uses the forward's quantised Q, K, tiling, masks and exp; D from
 * the same quantised dO), sec. 3.1 (dS to E4M3 with one scale per 32x32 block
 * so one payload feeds dQ and dK), sec. 3.4 "Backward pass".
 * Numerics: P = exp2(s - LSE log2 e); dV operand RNE_E4M3(2^8 P); dS in float
 * from the unquantised P; dS exponent = round-up rule on each document-aligned
 * 32x32 block maximum; dQ and dK scaled by softmax_scale after the products;
 * dQ partial sums are added in float32 (no prescale), then converted to BF16.
 * FLAMIA_FLAG_NONCAUSAL: as for the forward; dS is masked only at the
 * document ends.
 * FLAMIA_FLAG_HADAMARD: as for the forward, with softmax_scale / d, and the
 * gradients of the rotated operands are rotated back before the BF16
 * conversion: dQ = dQ_r H_d, dK = dK_r H_d (float32 butterflies as in the
 * quantiser).
 * FLAMIA_FLAG_DETERMINISTIC_DQ: by default the key tiles' dQ partials reach
 * the float32 accumulator in whatever order the CTAs finish (the sum varies
 * in its last bits from run to run).  With the flag, the 128-key tiles of a
 * document add their partials to a query tile in descending order (a turn
 * counter per query tile, bounded waits; each head's work items are claimed
 * shortest first, so a key tile never waits for one claimed after it), and
 * O, dQ, dK and dV are bitwise reproducible.  A wait that times out (2 s)
 * sets FLAMIA_DEV_TIMEOUT.
 * FLAMIA_FLAG_DS_ROW_EXPONENTS (review page, sec. 3.2: the query-row-wise dS
 * exponents that remove the leakage inside blocks): a 32 x 32 dS block
 * shares one exponent across 32 query rows, so a later row's gradient moves
 * the rounding of an earlier row's dQ; with the flag the dQ product takes dS
 * rounded per (query row, 32-key block), carried as its block scales, while
 * dK keeps the shared exponents (dK of a key sums every later query anyway).
 * FLAMIA_FLAG_DQ_FP16 (review page, sec. 3.2 "accumulator leakage", sec.
 * 3.5.3: the FP16 dQ reduce that halves the reduction traffic): each key
 * tile's float32 dQ partial of query row i is multiplied by 2^p(i), rounded
 * to FP16 and reduce-added into an FP16 accumulator; dQ = softmax_scale *
 * 2^-p(i) * acc.  p(i) = 15 - ceil(log2(16 d 448^3)) - (e_dO(i) + max e_V +
 * max e_K), e the E8M0 block exponents (every element |x| <= 448 2^e), which
 * bounds |2^p acc| by 2^15; clamped to [-126, 126].  The maxima run over
 * the head's whole sequence, so a later token changes the rounding of
 * earlier rows; with FLAMIA_FLAG_DQ_CAUSAL_SCALE they run over the keys the
 * row sees (its document up to the row; the whole document in a non-causal
 * call), which removes that dependence.  Combinable with every other flag.
 *
 *  dout         host pointer to the quantised dO (from the quantiser run with
 *               o_bf16 = the forward output, which also produced D).
 *  D, lse       float [H, T] from the quantiser and the forward.
 *  dq, dk, dv   [T, H, d] BF16 outputs (only tokens inside documents written).
 *  ws           flamia_bwd_workspace_bytes(T, H, d) bytes, 256-byte aligned.
 *  wl           as for the forward (its own claim counter).
 */
flamia_status flamia_attn_bwd(const flamia_qtensor* q, const flamia_qtensor* k,
                              const flamia_qtensor* v, const flamia_qtensor* dout,
                              const float* D, const float* lse,
                              const int32_t* cu_seqlens, int ndocs, int T, int H, int d,
                              float softmax_scale, int flags, void* wl,
                              void* dq_bf16, void* dk_bf16, void* dv_bf16,
                              void* ws, size_t ws_bytes, int* dev_status, void* stream);

/*
 * Grouped-query backward: as flamia_attn_bwd with K / V heads shared as in
 * flamia_attn_fwd_gqa; dq [T, H, d], dk and dv [T, H_kv, d] (the gradient of
 * a K / V head sums over its H / H_kv query heads); dout, D, lse per query
 * head.  The workspace is flamia_bwd_workspace_bytes(T, H, d).
 */
flamia_status flamia_attn_bwd_gqa(const flamia_qtensor* q, const flamia_qtensor* k,
                                  const flamia_qtensor* v, const flamia_qtensor* dout,
                                  const float* D, const float* lse, const int32_t* cu_seqlens,
                                  int ndocs, int T, int H, int H_kv, int d, float softmax_scale,
                                  int flags, void* wl, void* dq_bf16, void* dk_bf16,
                                  void* dv_bf16, void* ws, size_t ws_bytes, int* dev_status,
                                  void* stream);

/* Static description of a status code (never NULL). */
const char* flamia_status_str(flamia_status s);

#ifdef __cplusplus
}
#endif

#endif /* FLAMIA_H */
