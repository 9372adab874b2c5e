// Host-side interface of the decode kernel's grouped launch (decode.cu),
// shared with the C ABI layer (api.cu).
#pragma once

#include <cuda_runtime.h>

#include "../../include/tm_w4a16.h"

namespace w4 {

// One product of a grouped launch: Y = X . dequant(W) (or the fused
// silu(gate) * up when silu is set).
struct DecodeJob {
  const void* X;
  const tm_packed* p;
  void* Y;
  bool silu;
};

// Launch settings for n products of M rows that share the group size: the
// CTA shape, the cluster size (out->split_k) and, when `splits` is not NULL,
// each product's split along K (a power of two dividing the cluster size).
tm_status plan_decode_group(const tm_packed* const* ps, int n, int M, const tm_gemm_config* in, tm_gemm_config* out,
                            int* splits);

// The n products in one launch of the decode kernel (1 <= n <= TM_GROUP_MAX),
// planned by plan_decode_group from `in` (NULL = automatic).
tm_status launch_decode_group(const DecodeJob* jobs, int n, int M, const tm_gemm_config* in, cudaStream_t stream);

}  // namespace w4
