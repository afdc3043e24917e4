// Documents of at most kShortDoc tokens run on the CUDA cores (attn_short.cu);
// the tile kernels skip them.
#pragma once

#include <cuda_runtime.h>

#include "../../include/flamia.h"
#include "common.cuh"

namespace flamia {

cudaError_t launch_fwd_short(const flamia_qtensor* q, const flamia_qtensor* k,
                             const flamia_qtensor* v, const int32_t* cu, int ndocs, int T, int H,
                             int Hkv, int d, float softmax_scale, bool nvfp4_qk, bool causal,
                             bool token, void* o, float* lse, cudaStream_t stream);

cudaError_t launch_bwd_short(const flamia_qtensor* q, const flamia_qtensor* k,
                             const flamia_qtensor* v, const flamia_qtensor* dout, const float* D,
                             const float* lse, const int32_t* cu, int ndocs, int T, int H,
                             int Hkv, int d, float softmax_scale, bool nvfp4_qk, bool hadamard,
                             bool causal, bool ds_rows, bool token,
                             unsigned long long* ds_count, float* dq_acc,
                             const int8_t* dq_pre, void* dk, void* dv, cudaStream_t stream);

}  // namespace flamia
