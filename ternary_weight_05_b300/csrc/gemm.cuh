// Prefill-path W2A8 ternary GEMM on tcgen05 tensor cores (in progress).
#pragma once

#include "common.cuh"

namespace bitnet {

inline size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  (void)N;
  return (size_t)M * (size_t)K * 2 + (size_t)M * 4 + 1024;
}

inline int gemm_launch(const int8_t *, const float *, int64_t, const uint8_t *, const float *, int64_t, int64_t,
                       float *, int32_t *, void *, int, cudaStream_t) {
  return 4;  // BITNET_ERR_UNSUPPORTED until the tcgen05 kernel lands
}

}  // namespace bitnet
