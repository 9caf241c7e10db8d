// ep.h -- declarations of the expert-parallel exchange's kernels, shared by
// permute_combine.cu and moe_abi.cu.  Not part of the C ABI.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// dst[i] = src[idx[i]] for i < n: rows of d bf16 (d % 8 == 0); with gates,
// dgate[i] = sgate[idx[i]] as well (fp32).  Rows (and gates) whose idx
// entry is < 0 are left as they are.
cudaError_t launch_gather_rows(const void* src, const int32_t* idx, void* dst, int64_t n, int d,
                               const float* sgate, float* dgate, cudaStream_t stream);

}  // namespace moe
