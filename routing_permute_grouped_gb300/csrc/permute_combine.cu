// permute_combine.cu -- the two zero-FLOP stages of the layer, both bound by
// HBM bandwidth ("MoE & MLA operators", sec. 2.3 and 2.5).
//
// permute: token-major scatter.  A warp owns one token: it reads the token's
//          row once with 16-byte loads and writes it to the k padded rows
//          perm_row[t*k + j] with 16-byte stores.  Bytes per token:
//          d*2 read + k*d*2 written.
// combine: a warp owns one token: it reads the k routed rows y[perm_row[...]]
//          (and the shared-expert row) 16 bytes at a time, sums in fp32 in
//          the fixed order j = 0..k-1 then shared, and writes one bf16 row
//          (sec. 6.4: fixed summation order, wide accumulation, no atomics).
//          Bytes per token: (k + 1 [+1]) * d * 2.
// The rows are also split into column chunks over grid.y: for few tokens
// (decode) so that the grid still covers the SMs (8 tokens per CTA would
// otherwise leave a 64-token batch on 8 of them), and for grids of only a
// few waves so that the last wave's per-warp chains stay short.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ep.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

constexpr int kPCWarps = 8;  // warps per CTA
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kPCWarps * 32)
    k_permute(const uint4* __restrict__ x, const int32_t* __restrict__ perm_row,
              uint4* __restrict__ x_perm, int T, int nvec, int k, int chunk) {
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kPCWarps + warp;
    if (t >= T) return;
    const int vb = blockIdx.y * chunk;
    const int ve = min(nvec, vb + chunk);
    int rows[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) rows[j] = (j < k) ? ld_dep(perm_row + (int64_t)t * k + j) : -1;
    const uint4* src = x + (int64_t)t * nvec;
    for (int v0 = vb + lane; v0 < ve; v0 += 32 * kUnroll) {
        uint4 buf[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + u * 32;
            if (v < ve) buf[u] = ld_dep(src + v);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (rows[j] < 0) continue;
            uint4* dst = x_perm + (int64_t)rows[j] * nvec;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + u * 32;
                if (v < ve) dst[v] = buf[u];
            }
        }
    }
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Largest magnitude of a bf16 row of nvec 16-byte vectors, over the warp
// (kUnroll loads in flight per lane; absent vectors count as zeros).
__device__ __forceinline__ float row_amax(const uint4* src, int nvec, int lane) {
    float m = 0.0f;
    for (int v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
        uint4 b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + 32 * u;
            b[u] = v < nvec ? ld_dep(src + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float f[8];
            bf16x8_to_f32(b[u], f);
#pragma unroll
            for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
        }
    }
    return warp_max(m);
}

// Eight bf16 values of a row -> their e4m3 pair (hi, lo) under the row scale.
__device__ __forceinline__ void split_vec(const uint4& v, float scale, uint2& hi, uint2& lo) {
    float f[8];
    bf16x8_to_f32(v, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] *= scale;  // exact: a power of two
    e4m3_split8(f, hi, lo);
}

// The permute of the e4m3-weight path: the same token-major scatter, each row
// written as its e4m3 pair (rows 2r and 2r + 1 of x8, d bytes each) with the
// row's scale factor 2^-sig in x_scale[r]; xs8 / xs_scale (if given) also
// receive the dense pairs of every token row for the shared expert.  The
// pair and its scale are those of ptx.cuh (e4m3_row_scale, e4m3_split8).
__global__ void __launch_bounds__(kPCWarps * 32)
    k_permute_fp8(const uint4* __restrict__ x, const int32_t* __restrict__ perm_row,
                  uint8_t* __restrict__ x8, float* __restrict__ x_scale, uint8_t* __restrict__ xs8,
                  float* __restrict__ xs_scale, int T, int d, int k) {
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kPCWarps + warp;
    if (t >= T) return;
    const int nvec = d / 8;
    int rows[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) rows[j] = (j < k) ? ld_dep(perm_row + (int64_t)t * k + j) : -1;
    const uint4* src = x + (int64_t)t * nvec;
    const float scale = e4m3_row_scale(row_amax(src, nvec, lane));
    for (int v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
        uint4 b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (v0 + 32 * u < nvec) b[u] = ld_dep(src + v0 + 32 * u);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + 32 * u;
            if (v >= nvec) break;
            uint2 hi, lo;
            split_vec(b[u], scale, hi, lo);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (rows[j] < 0) continue;
                uint8_t* dst = x8 + (int64_t)rows[j] * 2 * d + (int64_t)v * 8;
                *reinterpret_cast<uint2*>(dst) = hi;
                *reinterpret_cast<uint2*>(dst + d) = lo;
            }
            if (xs8) {
                uint8_t* dst = xs8 + (int64_t)t * 2 * d + (int64_t)v * 8;
                *reinterpret_cast<uint2*>(dst) = hi;
                *reinterpret_cast<uint2*>(dst + d) = lo;
            }
        }
    }
    if (lane == 0) {
        const float inv = 1.0f / scale;  // exact: a power of two
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (rows[j] >= 0) x_scale[rows[j]] = inv;
        if (xs_scale) xs_scale[t] = inv;
    }
}

// The same permute with a CTA per token (few tokens: a warp per token would
// leave the batch on a handful of SMs).  The eight warps split the row; the
// row's largest magnitude is reduced over them in shared memory.
__global__ void __launch_bounds__(kPCWarps * 32)
    k_permute_fp8_cta(const uint4* __restrict__ x, const int32_t* __restrict__ perm_row,
                      uint8_t* __restrict__ x8, float* __restrict__ x_scale,
                      uint8_t* __restrict__ xs8, float* __restrict__ xs_scale, int T, int d, int k) {
    pdl_trigger();
    pdl_wait();
    __shared__ float s_max[kPCWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    if (t >= T) return;
    const int nvec = d / 8;
    int rows[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) rows[j] = (j < k) ? ld_dep(perm_row + (int64_t)t * k + j) : -1;
    const uint4* src = x + (int64_t)t * nvec;
    // this warp's vectors: v = warp * 32 + lane + 256 * i
    constexpr int kStride = kPCWarps * 32;
    float m = 0.0f;
    for (int v0 = warp * 32 + lane; v0 < nvec; v0 += kStride * kUnroll) {
        uint4 b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + kStride * u;
            b[u] = v < nvec ? ld_dep(src + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float f[8];
            bf16x8_to_f32(b[u], f);
#pragma unroll
            for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(f[q]));
        }
    }
    m = warp_max(m);
    if (lane == 0) s_max[warp] = m;
    __syncthreads();
    float amax = s_max[0];
#pragma unroll
    for (int w = 1; w < kPCWarps; ++w) amax = fmaxf(amax, s_max[w]);
    const float scale = e4m3_row_scale(amax);
    for (int v0 = warp * 32 + lane; v0 < nvec; v0 += kStride * kUnroll) {
        uint4 b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (v0 + kStride * u < nvec) b[u] = ld_dep(src + v0 + kStride * u);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + kStride * u;
            if (v >= nvec) break;
            uint2 hi, lo;
            split_vec(b[u], scale, hi, lo);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (rows[j] < 0) continue;
                uint8_t* dst = x8 + (int64_t)rows[j] * 2 * d + (int64_t)v * 8;
                *reinterpret_cast<uint2*>(dst) = hi;
                *reinterpret_cast<uint2*>(dst + d) = lo;
            }
            if (xs8) {
                uint8_t* dst = xs8 + (int64_t)t * 2 * d + (int64_t)v * 8;
                *reinterpret_cast<uint2*>(dst) = hi;
                *reinterpret_cast<uint2*>(dst + d) = lo;
            }
        }
    }
    if (threadIdx.x == 0) {
        const float inv = 1.0f / scale;  // exact: a power of two
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (rows[j] >= 0) x_scale[rows[j]] = inv;
        if (xs_scale) xs_scale[t] = inv;
    }
}

// The e4m3 pairs of the rows of h between the two expert GEMMs: CTA b <
// nb_cap takes block b of the table (its valid rows only, if b < num_blocks);
// CTA nb_cap + c takes dense rows [128 c, 128 c + 128) of hs.  A warp per row:
// its largest magnitude, the row scale, then the pair.
__global__ void __launch_bounds__(kPCWarps * 32)
    k_split_rows_e4m3(const uint4* __restrict__ h, const int32_t* __restrict__ block_metadata,
                      const int32_t* __restrict__ num_blocks, int nb_cap, int K,
                      uint8_t* __restrict__ h8, float* __restrict__ h_scale,
                      const uint4* __restrict__ hs, int Ts, int Ks, uint8_t* __restrict__ hs8,
                      float* __restrict__ hs_scale) {
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint4* src;
    uint8_t* dst;
    float* scl;
    int r0, nrows, width;
    if (static_cast<int>(blockIdx.x) < nb_cap) {
        const int nb = num_blocks ? ld_dep(num_blocks) : 0;
        if (static_cast<int>(blockIdx.x) >= nb) return;
        r0 = ld_dep(block_metadata + 3 * blockIdx.x + 1);
        nrows = ld_dep(block_metadata + 3 * blockIdx.x + 2);
        src = h;
        dst = h8;
        scl = h_scale;
        width = K;
    } else {
        r0 = (blockIdx.x - nb_cap) * 128;
        nrows = min(128, Ts - r0);
        src = hs;
        dst = hs8;
        scl = hs_scale;
        width = Ks;
    }
    const int nvec = width / 8;
    for (int i = warp; i < nrows; i += kPCWarps) {
        const int64_t r = r0 + i;
        const uint4* row = src + r * nvec;
        const float scale = e4m3_row_scale(row_amax(row, nvec, lane));
        for (int v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
            uint4 b[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (v0 + 32 * u < nvec) b[u] = ld_dep(row + v0 + 32 * u);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + 32 * u;
                if (v >= nvec) break;
                uint2 hi, lo;
                split_vec(b[u], scale, hi, lo);
                uint8_t* o = dst + r * 2 * width + (int64_t)v * 8;
                *reinterpret_cast<uint2*>(o) = hi;
                *reinterpret_cast<uint2*>(o + width) = lo;
            }
        }
        if (lane == 0) scl[r] = 1.0f / scale;
    }
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(w[i] << 16);
        acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8]) {
    uint4 o;
    __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[0], acc[1]);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[2], acc[3]);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(acc[4], acc[5]);
    __nv_bfloat162 p3 = __floats2bfloat162_rn(acc[6], acc[7]);
    o.x = *reinterpret_cast<uint32_t*>(&p0);
    o.y = *reinterpret_cast<uint32_t*>(&p1);
    o.z = *reinterpret_cast<uint32_t*>(&p2);
    o.w = *reinterpret_cast<uint32_t*>(&p3);
    return o;
}

// Each lane handles two 16-byte vectors per iteration, so up to 2 * (K + 1)
// independent loads are in flight per lane before the first add; K is a
// template parameter so the load buffers take only the registers they need.
template <int K>
__global__ void __launch_bounds__(kPCWarps * 32)
    k_combine(const uint4* __restrict__ y, const int32_t* __restrict__ perm_row,
              const uint4* __restrict__ shared_out, const uint4* __restrict__ extra2,
              uint4* __restrict__ out, int T, int nvec, int chunk) {
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kPCWarps + warp;
    if (t >= T) return;
    const int vb = blockIdx.y * chunk;
    const int ve = min(nvec, vb + chunk);
    int rows[K];
#pragma unroll
    for (int j = 0; j < K; ++j) rows[j] = ld_dep(perm_row + (int64_t)t * K + j);
    for (int v0 = vb + lane; v0 < ve; v0 += 64) {
        const int v1 = v0 + 32;
        const bool has1 = v1 < ve;
        uint4 in0[K], in1[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (rows[j] >= 0) {
                const uint4* src = y + (int64_t)rows[j] * nvec;
                in0[j] = ld_dep(src + v0);
                if (has1) in1[j] = ld_dep(src + v1);
            }
        }
        uint4 sh0 = make_uint4(0, 0, 0, 0), sh1 = make_uint4(0, 0, 0, 0);
        if (shared_out) {
            sh0 = ld_dep(shared_out + (int64_t)t * nvec + v0);
            if (has1) sh1 = ld_dep(shared_out + (int64_t)t * nvec + v1);
        }
        float a0[8], a1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a0[i] = a1[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (rows[j] >= 0) {
                add_bf16x8(a0, in0[j]);
                if (has1) add_bf16x8(a1, in1[j]);
            }
        if (shared_out) {
            add_bf16x8(a0, sh0);
            add_bf16x8(a1, sh1);
        }
        if (extra2) {
            add_bf16x8(a0, ld_dep(extra2 + (int64_t)t * nvec + v0));
            if (has1) add_bf16x8(a1, ld_dep(extra2 + (int64_t)t * nvec + v1));
        }
        __stcs(out + (int64_t)t * nvec + v0, pack_bf16x8(a0));
        if (has1) __stcs(out + (int64_t)t * nvec + v1, pack_bf16x8(a1));
    }
}

// Waits on an mbarrier that nothing ever signals, with the bounded wait that
// every kernel of the library uses; after limit_ns it records a timeout in
// *status and returns, leaving the context usable.
__global__ void k_wait_selftest(uint64_t limit_ns, uint32_t* status) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag, limit_ns)) atomicOr(status, 0x2u);
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, uint32_t* status, cudaStream_t stream) {
    k_wait_selftest<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError();
}

// Column chunks (in 16-byte vectors) for a grid of `rows_grid` CTAs along
// the tokens (8 tokens per CTA), over grid.y.
//  - Few tokens (fewer CTAs than twice the SMs): chunks of a multiple of 32
//    vectors, enough for twice the SMs.
//  - Otherwise: a warp walks its token's row one step at a time (`step`
//    vectors, one memory round trip each), and the grid runs in waves of
//    the CTAs resident at once (`per_sm` per SM).  With only two or three
//    waves the last one runs whole-row chains at partial occupancy, so the
//    rows are split into chunks of a multiple of `step` until the grid spans
//    about kTargetWaves waves.
constexpr int kTargetWaves = 6;

static int column_chunk(int rows_grid, int nvec, int step, int per_sm) {
    const int sms = num_sms();
    if (rows_grid <= 0) return nvec;
    if (rows_grid < 2 * sms) {
        const int want = 2 * sms;
        const int split = (want + rows_grid - 1) / rows_grid;
        int chunk = (nvec + split - 1) / split;
        chunk = ((chunk + 31) / 32) * 32;
        return chunk < nvec ? chunk : nvec;
    }
    const int want = kTargetWaves * sms * (per_sm > 0 ? per_sm : 1);
    if (rows_grid >= want) return nvec;
    const int split = (want + rows_grid - 1) / rows_grid;
    int chunk = (nvec + split - 1) / split;
    chunk = ((chunk + step - 1) / step) * step;
    return chunk < nvec ? chunk : nvec;
}

// Resident CTAs per SM of a permute/combine kernel (256 threads).
template <typename Kernel>
static int resident_per_sm(Kernel kernel) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kPCWarps * 32, 0) != cudaSuccess)
        n = 1;
    return n > 0 ? n : 1;
}

cudaError_t launch_permute(const void* x, const int32_t* perm_row, void* x_perm, int T, int d,
                           int k, cudaStream_t stream) {
    const int nvec = d / 8;
    const int grid = (T + kPCWarps - 1) / kPCWarps;
    if (grid == 0 || nvec == 0) return cudaSuccess;
    const int chunk = column_chunk(grid, nvec, 32 * kUnroll, resident_per_sm(k_permute));
    const int ny = (nvec + chunk - 1) / chunk;
    return launch_pdl(k_permute, dim3(grid, ny), dim3(kPCWarps * 32), 0, stream,
                      static_cast<const uint4*>(x), perm_row, static_cast<uint4*>(x_perm), T, nvec,
                      k, chunk);
}

// One warp per destination row: dst[i] = src[idx[i]] with 16-byte loads and
// stores; a negative idx[i] leaves row i untouched (the expert-parallel
// exchange: the rows a rank keeps are gathered here, the others arrive from
// its peers).
__global__ void __launch_bounds__(kPCWarps * 32)
    k_gather_rows(const uint4* __restrict__ src, const int32_t* __restrict__ idx,
                  uint4* __restrict__ dst, int64_t n, int nvec, const float* __restrict__ sgate,
                  float* __restrict__ dgate) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t i = blockIdx.x * static_cast<int64_t>(kPCWarps) + (threadIdx.x >> 5);
    if (i >= n) return;
    const int r = ld_dep(idx + i);
    if (r < 0) return;  // a row that another path fills: left as it is
    uint4* d = dst + i * nvec;
    const uint4* sr = src + static_cast<int64_t>(r) * nvec;
    for (int v = lane; v < nvec; v += 32) d[v] = ld_dep(sr + v);
    if (dgate && lane == 0) dgate[i] = ld_dep(sgate + r);
}

cudaError_t launch_gather_rows(const void* src, const int32_t* idx, void* dst, int64_t n, int d,
                               const float* sgate, float* dgate, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    const int64_t grid = (n + kPCWarps - 1) / kPCWarps;
    return launch_pdl(k_gather_rows, dim3(static_cast<unsigned>(grid)), dim3(kPCWarps * 32), 0, stream,
                      static_cast<const uint4*>(src), idx, static_cast<uint4*>(dst), n, d / 8, sgate,
                      dgate);
}

// Row pieces between two row-major buffers: piece i moves rows
// [src_row[i], src_row[i] + rows[i]) of src to [dst_row[i], ...) of dst (and
// their gates).  Grid (row groups, pieces); one warp per row, 16-byte
// accesses.  The piece descriptors live in device memory, so the local part
// of an expert-parallel exchange needs no index array from the host.
__global__ void __launch_bounds__(kPCWarps * 32)
    k_copy_pieces(const uint4* __restrict__ src, uint4* __restrict__ dst, int nvec,
                  const int32_t* __restrict__ src_row, const int32_t* __restrict__ dst_row,
                  const int32_t* __restrict__ rows, const float* __restrict__ sgate,
                  float* __restrict__ dgate) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int p = blockIdx.y;
    const int r = blockIdx.x * kPCWarps + (threadIdx.x >> 5);
    if (r >= ld_dep(rows + p)) return;
    const int64_t s = ld_dep(src_row + p) + static_cast<int64_t>(r);
    const int64_t d = ld_dep(dst_row + p) + static_cast<int64_t>(r);
    const uint4* sr = src + s * nvec;
    uint4* dr = dst + d * nvec;
    for (int v = lane; v < nvec; v += 32) dr[v] = ld_dep(sr + v);
    if (dgate && lane == 0) dgate[d] = ld_dep(sgate + s);
}

cudaError_t launch_copy_pieces(const void* src, void* dst, int d, const int32_t* src_row,
                               const int32_t* dst_row, const int32_t* rows, int n, int max_rows,
                               const float* sgate, float* dgate, cudaStream_t stream) {
    if (n <= 0 || max_rows <= 0) return cudaSuccess;
    const int gx = (max_rows + kPCWarps - 1) / kPCWarps;
    return launch_pdl(k_copy_pieces, dim3(gx, n), dim3(kPCWarps * 32), 0, stream,
                      static_cast<const uint4*>(src), static_cast<uint4*>(dst), d / 8, src_row,
                      dst_row, rows, sgate, dgate);
}

cudaError_t launch_permute_fp8(const void* x, const int32_t* perm_row, uint8_t* x8, float* x_scale,
                               uint8_t* xs8, float* xs_scale, int T, int d, int k,
                               cudaStream_t stream) {
    const int grid = (T + kPCWarps - 1) / kPCWarps;
    if (grid < 2 * num_sms())  // few tokens: a CTA per token
        return launch_pdl(k_permute_fp8_cta, dim3(T), dim3(kPCWarps * 32), 0, stream,
                          static_cast<const uint4*>(x), perm_row, x8, x_scale, xs8, xs_scale, T, d,
                          k);
    return launch_pdl(k_permute_fp8, dim3(grid), dim3(kPCWarps * 32), 0, stream,
                      static_cast<const uint4*>(x), perm_row, x8, x_scale, xs8, xs_scale, T, d, k);
}

cudaError_t launch_split_rows_e4m3(const void* h, const int32_t* block_metadata,
                                   const int32_t* num_blocks, int nb_cap, int K, uint8_t* h8,
                                   float* h_scale, const void* hs, int Ts, int Ks, uint8_t* hs8,
                                   float* hs_scale, cudaStream_t stream) {
    const int dense = hs ? (Ts + 127) / 128 : 0;
    const int grid = nb_cap + dense;
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(k_split_rows_e4m3, dim3(grid), dim3(kPCWarps * 32), 0, stream,
                      static_cast<const uint4*>(h), block_metadata, num_blocks, nb_cap, K, h8, h_scale,
                      static_cast<const uint4*>(hs), Ts, Ks, hs8, hs_scale);
}

cudaError_t launch_combine(const void* y, const int32_t* perm_row, const void* shared_out,
                           void* out, int T, int d, int k, cudaStream_t stream, const void* extra2) {
    const int nvec = d / 8;
    const int grid = (T + kPCWarps - 1) / kPCWarps;
    if (grid == 0 || nvec == 0) return cudaSuccess;
    const uint4* y4 = static_cast<const uint4*>(y);
    const uint4* s4 = static_cast<const uint4*>(shared_out);
    const uint4* x4 = static_cast<const uint4*>(extra2);
    uint4* o4 = static_cast<uint4*>(out);
    switch (k) {
#define MOE_COMBINE_K(KK)                                                                       \
    case KK: {                                                                                  \
        const int chunk = column_chunk(grid, nvec, 64, resident_per_sm(k_combine<KK>));         \
        const int ny = (nvec + chunk - 1) / chunk;                                              \
        return launch_pdl(k_combine<KK>, dim3(grid, ny), dim3(kPCWarps * 32), 0, stream, y4,    \
                          perm_row, s4, x4, o4, T, nvec, chunk);                                \
    }
        MOE_COMBINE_K(1) MOE_COMBINE_K(2) MOE_COMBINE_K(3) MOE_COMBINE_K(4)
        MOE_COMBINE_K(5) MOE_COMBINE_K(6) MOE_COMBINE_K(7) MOE_COMBINE_K(8)
#undef MOE_COMBINE_K
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace moe
