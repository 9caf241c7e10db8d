// pack.cu -- one-time weight preparation: the pages store weights as
// [in, out] (x @ W); the tcgen05 GEMMs read both operands K-major, so every
// weight is transposed to [out, in].  For the routed and shared gate/up
// weights the output rows of W1 (gate) and W3 (up) are interleaved per 128
// columns so that one 256-wide N tile holds both halves of 128 SwiGLU outputs
// (dual GEMM: one read of the activations feeds gate and up, "MoE & MLA
// operators", sec. 2.4(c)).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {

__device__ __forceinline__ int64_t packed_row(int c, int mode) {
    if (mode == 0) return c;
    const int blk = c >> 7, off = c & 127;
    return (int64_t)blk * 256 + (mode == 2 ? 128 : 0) + off;
}

// in [rows, cols] (batch stride in_bstride) -> out[packed_row(c), r]
// (row stride out_ld, batch stride out_bstride).  32x32 tiles through
// shared memory.
__global__ void k_pack_transpose(const __nv_bfloat16* __restrict__ in, __nv_bfloat16* __restrict__ out,
                                 int rows, int cols, int64_t in_bstride, int64_t out_bstride,
                                 int out_ld, int mode) {
    __shared__ __nv_bfloat16 tile[32][33];
    const int b = blockIdx.z;
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const __nv_bfloat16* src = in + b * in_bstride;
    __nv_bfloat16* dst = out + b * out_bstride;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[i][threadIdx.x] = src[(int64_t)r * cols + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < rows && c < cols) dst[packed_row(c, mode) * out_ld + r] = tile[threadIdx.x][i];
    }
}

cudaError_t launch_pack_transpose(const void* in, void* out, int rows, int cols, int64_t in_bstride,
                                  int64_t out_bstride, int out_ld, int mode, int batch,
                                  cudaStream_t stream) {
    dim3 grid((cols + 31) / 32, (rows + 31) / 32, batch);
    dim3 block(32, 8);
    k_pack_transpose<<<grid, block, 0, stream>>>(static_cast<const __nv_bfloat16*>(in),
                                                 static_cast<__nv_bfloat16*>(out), rows, cols,
                                                 in_bstride, out_bstride, out_ld, mode);
    return cudaGetLastError();
}

}  // namespace moe
