// backward.cu -- the element-wise and data-movement kernels of the layer
// backward (the GEMMs run on the grouped kernels of grouped_gemm.cu and
// wgrad_gemm.cu).  With out[t] = sum_j p_j (h_a W2) + ys[t], the routed rows
// of dout are permuted like x (dz_a = dout[t]) and dh_a = dz_a W2^T is the
// gradient before the routing weight:
//   k_router_bwd    dlogit = p_j (dp_j - sum_i p_i dp_i) for the k chosen
//                   experts of a token, 0 for the others (softmax over the
//                   chosen logits; the choice itself is a constant)
//   k_colsum        the logit-bias gradient: column sums in token order
//   k_swiglu_bwd    h = silu(g) u recomputed from the recomputed g, u, stored
//                   as p h; dg = p dh * u * silu'(g), du = p dh * silu(g) in
//                   the gate/up interleaved column order of the packed
//                   weights; the routing-weight gradient dp_a = <dh_a, h_a>;
//                   pad rows of the weight-gradient operands zeroed
//   k_interleave    row-wise interleave of gate and up blocks of 128 columns
//                   ([.., w] x 2 -> [.., 2w]): the backward weight layout
// Reads of data written by earlier kernels of the stream use ld_dep.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "backward.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// One warp per token.  Lanes j < k hold choice j: its expert, its routing
// weight p_j and dp_j = dgates[t][j]; s = sum_j p_j dp_j (a fixed shuffle
// tree); then lane c writes column c of dl[t] (fp32, [T, E]) and of dl16[t]
// (bf16, row stride ld16, zero past E): p_j (dp_j - s) summed over the j that
// chose expert c, 0 for the others.
__global__ void __launch_bounds__(kWarps * 32)
    k_router_bwd(const float* __restrict__ dgates, const int32_t* __restrict__ idx,
                 const float* __restrict__ gates, float* __restrict__ dl,
                 __nv_bfloat16* __restrict__ dl16, int T, int E, int k, int ld16) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t t = blockIdx.x * static_cast<int64_t>(kWarps) + (threadIdx.x >> 5);
    if (t >= T) return;
    float p = 0.0f, dp = 0.0f;
    int ex = -1;
    if (lane < k) {
        p = ld_dep(gates + t * k + lane);
        dp = ld_dep(dgates + t * k + lane);
        ex = ld_dep(idx + t * k + lane);
    }
    const float s = warp_sum(p * dp);
    const float gj = p * (dp - s);
    int ej[8];
    float vj[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        ej[j] = __shfl_sync(0xFFFFFFFFu, ex, j);
        vj[j] = __shfl_sync(0xFFFFFFFFu, gj, j);
    }
    for (int c = lane; c < ld16; c += 32) {
        float v = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < k && ej[j] == c && c < E) v += vj[j];
        if (c < E) dl[t * E + c] = v;
        dl16[t * ld16 + c] = __float2bfloat16_rn(v);
    }
}

// One block of 256 threads per column: thread i sums rows i, i + 256, ... in
// order, then a fixed tree over the threads (deterministic).
__global__ void __launch_bounds__(256)
    k_colsum(const float* __restrict__ m, float* __restrict__ out, int rows, int cols) {
    pdl_trigger();
    pdl_wait();
    __shared__ float part[8];
    const int c = blockIdx.x;
    float s = 0.0f;
    for (int r = threadIdx.x; r < rows; r += 256) s += ld_dep(m + (int64_t)r * cols + c);
    s = warp_sum(s);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int i = 0; i < 8; ++i) t += part[i];
        out[c] = t;
    }
}

// One warp per padded row r < *used_rows (all rows when used_rows is null).
// gu and dgu are [rows, 2w] in the interleaved order (block j of 256: 128
// gate columns, 128 up columns); dh is the row's gradient before its routing
// weight p.  For a row that holds assignment a: recomputes h = silu(g) u and
// writes hp = p h (bf16, the weight-gradient operand of the down projection),
// dgu = f'(g, u) * (p dh) and, when dgates is not null, dgates[a] = <dh, h>
// with h rounded to bf16.  A pad row (row_src < 0) inside a 64-row block that
// holds data is zeroed in hp, dgu and the two extra row-major buffers z0, z1
// (width zw; may be null): the weight-gradient GEMMs reduce over every
// 64-row step of a segment up to its last valid row.  Segments start on
// 64-row boundaries and hold their valid rows first, so a block holds data
// exactly when its first row is valid; pad rows of all-pad blocks are not
// read by anyone and are left as they are.
__global__ void __launch_bounds__(kWarps * 32)
    k_swiglu_bwd(const __nv_bfloat16* __restrict__ gu, const __nv_bfloat16* __restrict__ dh,
                 const int32_t* __restrict__ row_src, const float* __restrict__ row_gate,
                 const int32_t* __restrict__ used_rows, __nv_bfloat16* __restrict__ hp,
                 __nv_bfloat16* __restrict__ dgu, float* __restrict__ dgates,
                 __nv_bfloat16* __restrict__ z0, __nv_bfloat16* __restrict__ z1, int zw,
                 int64_t rows, int w) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    if (used_rows) {
        const int64_t u = ld_dep(used_rows);
        rows = u < rows ? u : rows;
    }
    const uint4 zero = make_uint4(0, 0, 0, 0);
    for (int64_t r = blockIdx.x * static_cast<int64_t>(kWarps) + (threadIdx.x >> 5); r < rows;
         r += nwarps) {
        const int a = row_src ? ld_dep(row_src + r) : static_cast<int>(r);
        if (a < 0 && ld_dep(row_src + (r & ~static_cast<int64_t>(63))) < 0) continue;  // all-pad block
        if (a < 0) {
            for (int c = lane * 8; c < w; c += 256) *reinterpret_cast<uint4*>(hp + r * w + c) = zero;
            for (int c = lane * 8; c < 2 * w; c += 256)
                *reinterpret_cast<uint4*>(dgu + r * 2 * w + c) = zero;
            for (int c = lane * 8; c < zw; c += 256) {
                if (z0) *reinterpret_cast<uint4*>(z0 + r * zw + c) = zero;
                if (z1) *reinterpret_cast<uint4*>(z1 + r * zw + c) = zero;
            }
            continue;
        }
        const float p = row_gate ? ld_dep(row_gate + r) : 1.0f;
        float dot = 0.0f;
        for (int c = lane * 8; c < w; c += 256) {
            const int64_t gcol = (c / 128) * 256 + (c % 128);
            float g[8], u[8], d[8], hv[8], dg[8], du[8];
            unpack8(ld_dep(reinterpret_cast<const uint4*>(gu + r * 2 * w + gcol)), g);
            unpack8(ld_dep(reinterpret_cast<const uint4*>(gu + r * 2 * w + gcol + 128)), u);
            unpack8(ld_dep(reinterpret_cast<const uint4*>(dh + r * w + c)), d);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float s = 1.0f / (1.0f + expf(-g[q]));
                hv[q] = g[q] * s * u[q];
                const float pd = p * d[q];
                dg[q] = pd * u[q] * s * (1.0f + g[q] * (1.0f - s));
                du[q] = pd * g[q] * s;
            }
            if (dgates) {
                float hb[8];
                unpack8(pack8(hv), hb);  // h as the forward stored it: bf16
#pragma unroll
                for (int q = 0; q < 8; ++q) dot += d[q] * hb[q];
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) hv[q] *= p;
            *reinterpret_cast<uint4*>(hp + r * w + c) = pack8(hv);
            *reinterpret_cast<uint4*>(dgu + r * 2 * w + gcol) = pack8(dg);
            *reinterpret_cast<uint4*>(dgu + r * 2 * w + gcol + 128) = pack8(du);
        }
        if (dgates) {
            dot = warp_sum(dot);
            if (lane == 0) dgates[a] = dot;
        }
    }
}

// mode 0: out2 [n, 2w] <- (a, b) [n, w] interleaved per 128 columns;
// mode 1: (a, b) [n, w] <- out2 [n, 2w].  One thread per 8 columns.
__global__ void k_interleave(__nv_bfloat16* __restrict__ a, __nv_bfloat16* __restrict__ b,
                             __nv_bfloat16* __restrict__ out2, int64_t n, int w, int mode) {
    pdl_trigger();
    pdl_wait();
    const int gpr = w / 8;
    const int64_t total = n * gpr;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / gpr;
        const int c = static_cast<int>(i - r * gpr) * 8;
        const int64_t g = r * 2 * w + (c / 128) * 256 + (c % 128);
        uint4* pa = reinterpret_cast<uint4*>(a + r * w + c);
        uint4* pb = reinterpret_cast<uint4*>(b + r * w + c);
        uint4* po = reinterpret_cast<uint4*>(out2 + g);
        uint4* pu = reinterpret_cast<uint4*>(out2 + g + 128);
        if (mode == 0) {
            *po = ld_dep(pa);
            *pu = ld_dep(pb);
        } else {
            *pa = ld_dep(po);
            *pb = ld_dep(pu);
        }
    }
}

int grid_for(int64_t work, int per_block) {
    int64_t g = (work + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
    if (g > cap) g = cap;
    return g < 1 ? 1 : static_cast<int>(g);
}

}  // namespace

cudaError_t launch_router_bwd(const float* dgates, const int32_t* idx, const float* gates, float* dl,
                              void* dl16, int T, int E, int k, int ld16, float* dbias,
                              cudaStream_t st) {
    // Plain launches (no programmatic dependent launch): these grids are
    // small and come right behind the weight-gradient kernel, which fills
    // every SM.  Launched early, their CTAs would be packed onto the first
    // SMs that free up and run there with a few SMs' share of the machine
    // (measured: 395 us instead of 24 us at T = 8192); launched plainly they
    // start once the SMs are free and spread over all of them.
    k_router_bwd<<<static_cast<unsigned>((T + kWarps - 1) / kWarps), kWarps * 32, 0, st>>>(
        dgates, idx, gates, dl, static_cast<__nv_bfloat16*>(dl16), T, E, k, ld16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !dbias) return e;
    k_colsum<<<E, 256, 0, st>>>(static_cast<const float*>(dl), dbias, T, E);
    return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(const void* gu, const void* dh, const int32_t* row_src,
                              const float* row_gate, const int32_t* used_rows, void* hp, void* dgu,
                              float* dgates, void* z0, void* z1, int zw, int64_t rows, int w,
                              cudaStream_t st) {
    return launch_pdl(k_swiglu_bwd, dim3(grid_for(rows, kWarps)), dim3(kWarps * 32), 0, st,
                      static_cast<const __nv_bfloat16*>(gu), static_cast<const __nv_bfloat16*>(dh),
                      row_src, row_gate, used_rows, static_cast<__nv_bfloat16*>(hp),
                      static_cast<__nv_bfloat16*>(dgu), dgates, static_cast<__nv_bfloat16*>(z0),
                      static_cast<__nv_bfloat16*>(z1), zw, rows, w);
}

cudaError_t launch_interleave(void* a, void* b, void* out2, int64_t n, int w, int mode,
                              cudaStream_t st) {
    const int64_t work = n * (w / 8);
    return launch_pdl(k_interleave, dim3(grid_for(work, 256)), dim3(256), 0, st,
                      static_cast<__nv_bfloat16*>(a), static_cast<__nv_bfloat16*>(b),
                      static_cast<__nv_bfloat16*>(out2), n, w, mode);
}

}  // namespace moe
