// backward.h -- declarations of the layer backward's launchers, shared by
// backward.cu, wgrad_gemm.cu and moe_abi.cu.  Not part of the C ABI.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Weight-gradient GEMM: out[e][m][n] = sum over rows r in [seg[e], seg[e+1])
// of A[r][m] * B[r][n]; A [rows, M] and B [rows, N] bf16 row-major (pad rows
// zero; M % 64 == 0, N % 128 == 0), out bf16 [n_experts, M, N] (or split into
// gate/up halves through out2).
struct WgradArgs {
    const int32_t* seg;  // [n_experts + 1] row offsets (device), or null: rows [0, dense_rows)
    int32_t dense_rows;
    int32_t rows;        // rows of the operands; a segment past them is skipped
    int32_t n_experts, M, N, m_tiles, n_tiles;
    void* out;   // [n_experts, M, N], or with out2 the gate half [n_experts, M, N / 2]
    void* out2;  // null, or the up half: N is the gate/up interleave of the packed weights
    bool f32;    // fp32 output [n_experts, M, n_valid] (columns >= n_valid dropped)
    int32_t n_valid;
    uint32_t* status;
    // null, or [n_experts]: rows of each segment that hold data; the rest of
    // the segment is zero pad rows, and whole 64-row steps of them are skipped
    const int32_t* valid;
};
cudaError_t launch_wgrad(const void* A, int64_t M, const void* B, int64_t N, int64_t rows,
                         const int32_t* seg, int n_experts, int dense_rows, void* out, void* out2,
                         uint32_t* status, cudaStream_t stream, int f32_cols = 0,
                         const int32_t* valid = nullptr);
// dl [T, E] (fp32) and dl16 [T, ld16] (bf16, zero past E) from dgates; dbias
// (if not null) = column sums of dl.
cudaError_t launch_router_bwd(const float* dgates, const int32_t* idx, const float* gates, float* dl,
                              void* dl16, int T, int E, int k, int ld16, float* dbias,
                              cudaStream_t st);
// From gu [rows, 2w] (rows r < *used_rows; all when used_rows is null):
// hp [rows, w] = row_gate[r] * silu(g) u (bf16) and dgu [rows, 2w] = the
// SwiGLU backward for the gradient row_gate[r] * dh [rows, w];
// dgates[row_src[r]] = <dh[r], h[r]> when dgates is not null.  Pad rows
// (row_src < 0) are zeroed in hp, dgu, z0 and z1 ([rows, zw], may be null).
// row_src null: row r holds r; row_gate null means 1.
cudaError_t launch_swiglu_bwd(const void* gu, const void* dh, const int32_t* row_src,
                              const float* row_gate, const int32_t* used_rows, void* hp, void* dgu,
                              float* dgates, void* z0, void* z1, int zw, int64_t rows, int w,
                              cudaStream_t st);
// mode 0: out2 [n, 2w] <- gate a, up b [n, w] (interleaved per 128 columns);
// mode 1: the inverse.
cudaError_t launch_interleave(void* a, void* b, void* out2, int64_t n, int w, int mode,
                              cudaStream_t st);

}  // namespace moe
