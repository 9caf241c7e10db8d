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
#include "ptx.cuh"

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

// ------------------------------------------------------- e4m3 weights --
// Per-output-channel scale of in [rows, cols] (column c = output channel c):
// amax over the column (exact in fp32), scale = amax / 448 by an IEEE
// single-precision division, 1 for an all-zero column.  One thread per
// column, rows walked in order (coalesced across the warp).
__global__ void k_col_scale(const __nv_bfloat16* __restrict__ in, float* __restrict__ scale,
                            int rows, int cols, int64_t in_bstride, int64_t scale_bstride,
                            int mode) {
    const int b = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    const __nv_bfloat16* src = in + b * in_bstride + c;
    float amax = 0.0f;
    for (int r = 0; r < rows; ++r) amax = fmaxf(amax, fabsf(__bfloat162float(src[(int64_t)r * cols])));
    scale[b * scale_bstride + packed_row(c, mode)] = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

// Codes of the transposed matrix: out[packed_row(c), r] = e4m3(in[r, c] /
// scale[c]), the quotient an IEEE single-precision division and the code its
// nearest e4m3 value (ties to even, saturating).  32x32 tiles through shared
// memory as in k_pack_transpose.
__global__ void k_pack_quant(const __nv_bfloat16* __restrict__ in, uint8_t* __restrict__ out,
                             const float* __restrict__ scale, int rows, int cols,
                             int64_t in_bstride, int64_t out_bstride, int64_t scale_bstride,
                             int out_ld, int mode) {
    __shared__ float tile[32][33];
    const int b = blockIdx.z;
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const __nv_bfloat16* src = in + b * in_bstride;
    uint8_t* dst = out + b * out_bstride;
    const float* sc = scale + b * scale_bstride;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[i][threadIdx.x] = __bfloat162float(src[(int64_t)r * cols + c]);
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < rows && c < cols) {
            const int64_t pr = packed_row(c, mode);
            dst[pr * out_ld + r] = f32_to_e4m3(__fdiv_rn(tile[threadIdx.x][i], __ldg(sc + pr)));
        }
    }
}

cudaError_t launch_pack_fp8(const void* in, uint8_t* out, float* scale, int rows, int cols,
                            int64_t in_bstride, int64_t out_bstride, int64_t scale_bstride,
                            int out_ld, int mode, int batch, cudaStream_t stream) {
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(in);
    k_col_scale<<<dim3((cols + 127) / 128, batch), 128, 0, stream>>>(src, scale, rows, cols, in_bstride,
                                                                      scale_bstride, mode);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 grid((cols + 31) / 32, (rows + 31) / 32, batch);
    k_pack_quant<<<grid, dim3(32, 8), 0, stream>>>(src, out, scale, rows, cols, in_bstride, out_bstride,
                                                   scale_bstride, out_ld, mode);
    return cudaGetLastError();
}

// Widens e4m3 codes to bf16 (every e4m3 value is a bf16 value: exact), 16
// codes per thread, grid-stride.  For the e4m3 layer at batch sizes where the
// tensor pipe, not the weight bytes, sets the pace: the bf16 GEMMs then run
// on the widened codes and scale their accumulators per output channel.
__global__ void k_widen_e4m3(const uint4* __restrict__ q, uint4* __restrict__ out, int64_t n16) {
    pdl_trigger();
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 c = ld_dep(q + i);
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t hf = e4m3x2_to_f16x2(static_cast<uint16_t>(w[j] >> (16 * h)));
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hf));
                o[2 * j + h] = pack_bf16x2(f.x, f.y);
            }
        }
        out[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
        out[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

cudaError_t launch_widen_e4m3(const void* q, void* out, int64_t n, cudaStream_t stream) {
    if (n % 16) return cudaErrorInvalidValue;
    const int64_t n16 = n / 16;
    int64_t grid = (n16 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    return launch_pdl(k_widen_e4m3, dim3(static_cast<unsigned>(grid)), dim3(256), 0, stream,
                      static_cast<const uint4*>(q), static_cast<uint4*>(out), n16);
}

}  // namespace moe
