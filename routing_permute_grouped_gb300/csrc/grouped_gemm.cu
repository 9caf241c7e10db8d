// grouped_gemm.cu -- the tensor-core stages of the layer, tcgen05 + TMA:
//
//   k_grouped_gemm       one CTA per SM, M = 128 x N = BN tiles (BN = E
//                        rounded up to 16..256): the router, logits = x Wg^T
//                        (+ bias) with top-k in the epilogue, or fp32
//                        partial logits of one K slice (split-K router)
//   k_grouped_gemm_pair  CTA pairs (cta_group::2, M = 256 x N = 256): the
//                        grouped expert GEMMs over the block table
//                          GEMM1: [g | u] = x_perm W13[e]^T, h = bf16(silu(g) u)
//                          GEMM2: y = bf16(row_gate * (h W2[e]^T))
//                        and the dense shared expert on a dense tile list
//
// The expert work list is the block table [expert, m_start, valid_m] built on
// the device ("MoE & MLA operators", sec. 2.3; "Dropless and grouped GEMM",
// sec. 5: a tile reads exactly one expert's weights, the tile count lives in
// device memory and the host never learns the per-expert sizes).
//
// Both kernels are persistent and warp-specialised (6 warps per CTA):
//   warp 0      TMA producer: A and B tiles (64 K-columns, 128-byte swizzle)
//               into a ring of shared-memory stages guarded by mbarriers
//   warp 1      allocates tensor memory; one lane issues tcgen05.mma into one
//               of two TMEM accumulators
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one row per thread),
//               fused SwiGLU / gate / top-k, stores to global memory; on the
//               shared expert's token-major tiles also the permute (GEMM1,
//               after the accumulator is handed back) or the combine (GEMM2)
//   warps 6..7  (pair kernel, launched only when GEMM1 does the permute)
//               copy the token rows into the permuted layout ahead of the
//               TMA producer, which waits on per-visit counts
// The two accumulators let the epilogue of tile i overlap the MMAs of tile
// i+1.  Every wait is bounded; on a timeout the CTA flags the status word,
// drains what it has in flight and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

constexpr int BM = 128;
constexpr int BK = 64;  // bf16 elements per 128-byte swizzled row
constexpr int kOutStageBytes = 4 * 2 * 4096;  // pair-kernel epilogue staging
constexpr int kThreads = 192;
constexpr int kPairThreads = 256;  // the pair kernel with its 2 copy warps (6 warps without)
constexpr uint32_t kDevErrTimeout = 0x2u;

template <int BN>
struct GemmCfg {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES_RAW = (196 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                     : (2 * BN <= 256) ? 256 : 512;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + BAR_BYTES;
    static_assert(B_BYTES % 1024 == 0, "B stage must keep 1024-byte alignment");
    static_assert(STAGES >= 2, "need at least two stages");
};

// One tile of the 1-CTA kernel: 128 token rows [m0, m0 + 128) of the dense
// router GEMM, of which rows [lo, hi) (relative to m0) exist, and column panel
// (or, for the split-K router, K slice) nb.  The pair kernel's epilogue uses
// the same record for its 128-row half of a visit.
struct TileInfo {
    int e, m0, lo, hi, nb;
    bool skip;
};

__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, int t) {
    TileInfo ti;
    const int mb = t / a.n_tiles;
    ti.nb = t - mb * a.n_tiles;
    ti.skip = false;
    ti.e = 0;
    ti.m0 = mb * BM;
    ti.lo = 0;
    ti.hi = min(BM, a.dense_rows - ti.m0);
    return ti;
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

// ----------------------------------------------------------- epilogues --

// GEMM1: columns [0, 128) of the tile are gate, [128, 256) up, for the 128
// SwiGLU outputs [nb*128, nb*128 + 128) of row m0 + row.
// Multiplies 32 accumulators by the scales of their columns (cs: the first
// of them, 16-byte aligned; null = no scale).  The scales were written by a
// packing kernel that finished long before this launch: read-only loads.
__device__ __forceinline__ void scale_cols(uint32_t (&v)[32], const float* cs) {
    if (!cs) return;
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 s4 = __ldg(reinterpret_cast<const float4*>(cs + i));
        v[i] = __float_as_uint(__uint_as_float(v[i]) * s4.x);
        v[i + 1] = __float_as_uint(__uint_as_float(v[i + 1]) * s4.y);
        v[i + 2] = __float_as_uint(__uint_as_float(v[i + 2]) * s4.z);
        v[i + 3] = __float_as_uint(__uint_as_float(v[i + 3]) * s4.w);
    }
}

// Scales of the tile's first B row (packed row col0 of expert e), or null.
__device__ __forceinline__ const float* tile_scales(const GemmArgs& a, const TileInfo& ti, int col0) {
    return a.col_scale ? a.col_scale + (int64_t)ti.e * a.b_rows_per_expert + col0 : nullptr;
}

// Stores 32 gate and 32 up accumulators of one row as bf16 at column c of
// the tile in the saved gate/up array (packed order: the tile's 128 gate
// columns, then its 128 up columns).
__device__ __forceinline__ void save_gate_up(const GemmArgs& a, const TileInfo& ti, int row, int c,
                                             const uint32_t (&g)[32], const uint32_t (&u)[32]) {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.gu_out) + (int64_t)(ti.m0 + row) * a.ld_gu +
                         (int64_t)ti.nb * 256 + c;
    uint32_t pg[16], pu[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        pg[i] = pack_bf16x2(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
        pu[i] = pack_bf16x2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
    }
    uint4* dg = reinterpret_cast<uint4*>(dst);
    uint4* du = reinterpret_cast<uint4*>(dst + 128);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        dg[i] = make_uint4(pg[4 * i], pg[4 * i + 1], pg[4 * i + 2], pg[4 * i + 3]);
        du[i] = make_uint4(pu[4 * i], pu[4 * i + 1], pu[4 * i + 2], pu[4 * i + 3]);
    }
}

__device__ __forceinline__ void epi_swiglu(const GemmArgs& a, const TileInfo& ti, uint32_t taddr,
                                           int row) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const bool valid = row >= ti.lo && row < ti.hi;
    __nv_bfloat16* dst = out + (int64_t)(ti.m0 + row) * a.ldo + (int64_t)ti.nb * 128;
    const float* cs = tile_scales(a, ti, ti.nb * 256);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t g[32], u[32];
        tmem_ld32(taddr + c * 32, g);
        tmem_ld32(taddr + 128 + c * 32, u);
        tmem_ld_wait();
        if (cs) {
            scale_cols(g, cs + c * 32);
            scale_cols(u, cs + 128 + c * 32);
        }
        if (valid && a.gu_out) save_gate_up(a, ti, row, c * 32, g, u);
        if (valid) {
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
                p[i] = pack_bf16x2(silu_f32(g0) * u0, silu_f32(g1) * u1);
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
        }
    }
}

// GEMM2: y = bf16(gate * acc) for the BN output columns of the tile.
template <int BN>
__device__ __forceinline__ void epi_gate(const GemmArgs& a, const TileInfo& ti, uint32_t taddr,
                                         int row) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const bool valid = row >= ti.lo && row < ti.hi;
    const float gate = (valid && a.row_gate) ? ld_dep(a.row_gate + ti.m0 + row) : 1.0f;
    __nv_bfloat16* dst = out + (int64_t)(ti.m0 + row) * a.ldo + (int64_t)ti.nb * BN;
    const float* cs = tile_scales(a, ti, ti.nb * BN);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(taddr + c * 32, v);
        tmem_ld_wait();
        if (cs) scale_cols(v, cs + c * 32);
        if (valid) {
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                p[i] = pack_bf16x2(gate * __uint_as_float(v[2 * i]), gate * __uint_as_float(v[2 * i + 1]));
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
        }
    }
}

// ---------------------------------------------------- combine epilogue --
// The shared expert's GEMM2 tile covers token rows in token order, so the
// layer's combine ("MoE & MLA operators", sec. 2.5: the k weighted expert
// rows of a token summed back in token order, plus the shared expert's row)
// can be taken by the thread that owns the token's output row: no atomics,
// and the same fixed order as the stand-alone combine kernel, so the result
// is bit for bit the one of GEMM2 followed by the combine.

// The routed rows of the token (comb_perm[token * k + j], j < k), -1 past k
// or for a row past the tile's valid rows.
__device__ __forceinline__ void combine_rows_of(const GemmArgs& a, int token, bool valid,
                                                int (&pr)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        pr[j] = (valid && j < a.comb_k) ? ld_dep(a.comb_perm + (int64_t)token * a.comb_k + j) : -1;
}

// s[i] = sum over j ascending (rows < 0 skipped) of comb_y[pr[j]][col + i],
// fp32 from zero, for 32 columns; the loads of two rows are in flight at a
// time (the rows were fetched into L2 ahead of the epilogue).
__device__ __forceinline__ void combine_sum32(const GemmArgs& a, const int (&pr)[8], int64_t col,
                                              float (&s)[32]) {
    const __nv_bfloat16* y = static_cast<const __nv_bfloat16*>(a.comb_y);
#pragma unroll
    for (int i = 0; i < 32; ++i) s[i] = 0.0f;
#pragma unroll
    for (int j0 = 0; j0 < 8; j0 += 2) {
        uint4 in[2][4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
            if (pr[j0 + jj] >= 0) {
                const uint4* src = reinterpret_cast<const uint4*>(y + (int64_t)pr[j0 + jj] * a.comb_ldy + col);
#pragma unroll
                for (int u = 0; u < 4; ++u) in[jj][u] = ld_dep(src + u);
            }
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
            if (pr[j0 + jj] >= 0) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t w[4] = {in[jj][u].x, in[jj][u].y, in[jj][u].z, in[jj][u].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        s[8 * u + 2 * i] += __uint_as_float(w[i] << 16);
                        s[8 * u + 2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
                    }
                }
            }
    }
}

// The tile's own result rounded to bf16 (as the stand-alone GEMM2 stores it)
// added last, then one rounding to bf16.
__device__ __forceinline__ uint32_t combine_pack2(float s0, float s1, uint32_t v0, uint32_t v1) {
    const float r0 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(v0)));
    const float r1 = __bfloat162float(__float2bfloat16_rn(__uint_as_float(v1)));
    return pack_bf16x2(s0 + r0, s1 + r1);
}

// Per-thread path of the combine epilogue (rows of a partly valid warp).
template <int BN>
__device__ __forceinline__ void epi_combine(const GemmArgs& a, const TileInfo& ti, uint32_t taddr,
                                            int row, const int (&pr)[8]) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const bool valid = row >= ti.lo && row < ti.hi;
    __nv_bfloat16* dst = out + (int64_t)(ti.m0 + row) * a.ldo + (int64_t)ti.nb * BN;
    const float* cs = tile_scales(a, ti, ti.nb * BN);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        float sum[32];
        combine_sum32(a, pr, (int64_t)ti.nb * BN + c * 32, sum);
        uint32_t v[32];
        tmem_ld32(taddr + c * 32, v);
        tmem_ld_wait();
        if (cs) scale_cols(v, cs + c * 32);
        if (valid) {
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) p[i] = combine_pack2(sum[2 * i], sum[2 * i + 1], v[2 * i], v[2 * i + 1]);
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
        }
    }
}

// ---------------------------------------------------- permute epilogue --
// The permute ("MoE & MLA operators", sec. 2.3: every token row copied to its
// k expert-major positions) in the slack of the shared expert's GEMM1.  That
// GEMM's tiles are long (K = d) and its epilogue waits for the next
// accumulator most of the time; after handing the accumulator back, the warp
// copies the tile's column slice of its 32 token rows, 8 rows at a time with
// the lanes across the columns (coalesced 512-byte accesses).  The tiles of
// one 256-row visit cover the row's columns once between them.
__device__ __forceinline__ void permute_slice(const GemmArgs& a, const TileInfo& ti, int q, int lane) {
    const int nvec = a.perm_nvec, k = a.perm_k;
    const int v0 = static_cast<int>(static_cast<int64_t>(ti.nb) * nvec / a.n_tiles);
    const int v1 = static_cast<int>(static_cast<int64_t>(ti.nb + 1) * nvec / a.n_tiles);
    const uint4* x = static_cast<const uint4*>(a.perm_x);
    uint4* xp = static_cast<uint4*>(a.perm_out);
    const int row = q * 32 + lane;  // this lane's row of the tile, for the positions
    const bool valid = row >= ti.lo && row < ti.hi;
    int dst[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        dst[j] = (valid && j < k) ? ld_dep(a.perm_rows + static_cast<int64_t>(ti.m0 + row) * k + j) : -1;
#pragma unroll 1
    for (int vb = v0; vb < v1; vb += 64) {
#pragma unroll 1
        for (int r0 = 0; r0 < 32; r0 += 8) {
            uint4 buf[8][2];
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int r = q * 32 + r0 + rr;
                const bool rv = r >= ti.lo && r < ti.hi;  // the same for every lane
                const uint4* src = x + static_cast<int64_t>(ti.m0 + r) * nvec;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int v = vb + lane + 32 * h;
                    if (rv && v < v1) buf[rr][h] = ld_dep(src + v);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int dj = __shfl_sync(0xFFFFFFFFu, dst[j], r0 + rr);
                    if (dj < 0) continue;
                    uint4* o = xp + static_cast<int64_t>(dj) * nvec;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int v = vb + lane + 32 * h;
                        if (v < v1) o[v] = buf[rr][h];
                    }
                }
            }
        }
    }
}

// Router: the thread owns token m0 + row and its E logits (TMEM columns
// [0, E)).  Group-limited routing keeps the topk_groups groups with the
// largest maximum logit; top-k runs over the eligible experts in ascending
// index order with strict comparisons, so the lower index wins a tie; the
// gates are a softmax over the k chosen logits.
template <int BN>
__device__ __forceinline__ void epi_router(const GemmArgs& a, const TileInfo& ti, uint32_t taddr,
                                           int row) {
    const int E = a.E, k = a.k;
    const int token = ti.m0 + row;
    const bool valid = row >= ti.lo && row < ti.hi;
    uint32_t gmask = 0xFFFFFFFFu;
    int gsz = E;
    if (a.n_groups > 0) {
        gsz = E / a.n_groups;
        float gs[32];
#pragma unroll
        for (int g = 0; g < 32; ++g) gs[g] = -FLT_MAX;
#pragma unroll 1
        for (int c = 0; c < BN / 16; ++c) {
            uint32_t v[16];
            tmem_ld16(taddr + c * 16, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = c * 16 + i;
                if (e < E) {
                    const float l = __uint_as_float(v[i]) + (a.bias ? ld_dep(a.bias + e) : 0.0f);
                    const int g = e / gsz;
                    gs[g] = fmaxf(gs[g], l);
                }
            }
        }
        gmask = 0;
        for (int r = 0; r < a.topk_groups; ++r) {
            int bi = -1;
            float bv = -FLT_MAX;
            for (int g = 0; g < a.n_groups; ++g) {
                if (gmask & (1u << g)) continue;
                if (bi < 0 || gs[g] > bv) {
                    bi = g;
                    bv = gs[g];
                }
            }
            gmask |= 1u << bi;
        }
    }
    float tv[8];
    int ti_[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        tv[s] = -FLT_MAX;
        ti_[s] = -1;
    }
#pragma unroll 1
    for (int c = 0; c < BN / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(taddr + c * 16, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int e = c * 16 + i;
            if (e < E && ((gmask >> (e / gsz)) & 1u)) {
                float cv = __uint_as_float(v[i]) + (a.bias ? ld_dep(a.bias + e) : 0.0f);
                int ci = e;
                bool shifting = false;
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    if (s < k && (shifting || ti_[s] < 0 || cv > tv[s])) {
                        const float tf = tv[s];
                        const int tii = ti_[s];
                        tv[s] = cv;
                        ti_[s] = ci;
                        cv = tf;
                        ci = tii;
                        shifting = true;
                    }
                }
            }
        }
    }
    if (valid) {
        float sum = 0.0f;
#pragma unroll
        for (int s = 0; s < 8; ++s)
            if (s < k) sum += expf(tv[s] - tv[0]);
        const float inv = 1.0f / sum;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            if (s < k) {
                a.topk_idx[(int64_t)token * k + s] = ti_[s];
                a.topk_w[(int64_t)token * k + s] = expf(tv[s] - tv[0]) * inv;
            }
        }
    }
}

// Split-K router: fp32 partial logits of this K slice for the token rows of
// the tile, columns [0, E).
template <int BN>
__device__ __forceinline__ void epi_partial(const GemmArgs& a, const TileInfo& ti, uint32_t taddr,
                                            int row) {
    const bool valid = row >= ti.lo && row < ti.hi;
    float* dst = a.partial + (static_cast<int64_t>(ti.nb) * a.dense_rows + ti.m0 + row) * a.E;
#pragma unroll 1
    for (int c = 0; c < BN / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(taddr + c * 16, v);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (c * 16 + i < a.E) dst[c * 16 + i] = __uint_as_float(v[i]);
        }
    }
}

// Where a CTA of the dense router GEMMs starts its K loop.  Every CTA streams
// its own 128 token rows, and with a power-of-two row pitch the rows of all
// CTAs at the same K offset fall on few DRAM channels; starting each CTA at
// a different K block (and wrapping around) spreads the concurrent reads.
// The MMAs accumulate in the rotated order: a fixed order per CTA.
__device__ __forceinline__ int k_rotation(int nk) {
    return nk > 1 ? static_cast<int>((blockIdx.x * 7u) % static_cast<unsigned>(nk)) : 0;
}
__device__ __forceinline__ int rotated_k(int kb, int kb0, int kb1, int rot) {
    int k = kb + rot;
    return k >= kb1 ? k - (kb1 - kb0) : k;
}

// -------------------------------------------------------------- kernel --
template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs args) {
    using C = GemmCfg<BN>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * C::A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S * C::B_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* tfull = bars + 2 * S;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_holder + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull + i, 1);
            mbar_init(tempty + i, 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    // Inputs written by earlier kernels are visible after pdl_wait().  Tensor
    // memory is taken only after it too: by then every earlier kernel of the
    // stream has finished and released its own, and no later kernel has
    // allocated (each of them waits in the same place first).  Allocating
    // before the wait could deadlock a chain A -> B -> C of tensor-memory
    // kernels: a CTA of C, let in early by B's trigger, could take the
    // columns A frees while a CTA of B on the same SM still waits for them,
    // and then wait for B to finish.
    pdl_wait();
    if (warp == 1) tmem_alloc(tmem_holder, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int total = ((args.dense_rows + BM - 1) / BM) * args.n_tiles;
    bool timed_out = false;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;  // stages armed and not yet seen consumed
            for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
                const TileInfo ti = decode_tile(args, t);
                const bool split = EPI == kEpiPartial;
                const int brow = split ? 0 : ti.e * args.b_rows_per_expert + ti.nb * BN;
                const int kb0 = split ? ti.nb * args.k_per_split : 0;
                const int kb1 = split ? min(kb0 + args.k_per_split, args.k_blocks) : args.k_blocks;
                const int rot = k_rotation(kb1 - kb0);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(empty + s, ph ^ 1u, abort_flag)) {
                        timed_out = true;
                        break;
                    }
                    armed &= ~(1u << s);
                    const int kx = rotated_k(kb, kb0, kb1, rot) * BK;
                    mbar_arrive_expect_tx(full + s, C::STAGE_BYTES);
                    tma_load_2d(sA + s * C::A_BYTES, &tmA, kx, ti.m0, full + s);
                    tma_load_2d(sB + s * C::B_BYTES, &tmB, kx, brow, full + s);
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (timed_out || *abort_flag) {
                *abort_flag = 1;
                // let the copies already issued land before the CTA exits
                for (int i = 0; i < S; ++i)
                    if (armed & (1u << i)) {
                        volatile uint32_t never = 0;
                        (void)mbar_wait(full + i, (armed_par >> i) & 1u, &never);
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool issued = false;
            for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
                const TileInfo ti = decode_tile(args, t);
                const int kb0 = EPI == kEpiPartial ? ti.nb * args.k_per_split : 0;
                const int kb1 = EPI == kEpiPartial ? min(kb0 + args.k_per_split, args.k_blocks)
                                                   : args.k_blocks;
                if (!mbar_wait(tempty + acc, aph ^ 1u, abort_flag)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(full + s, ph, abort_flag)) {
                        timed_out = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + s * C::A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        mma_bf16(d_tmem, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(b_addr + kk * 32),
                                 idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                    }
                    issued = true;
                    mma_commit(empty + s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (timed_out) break;
                mma_commit(tfull + acc);
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
            }
            if ((timed_out || *abort_flag) && issued) {
                *abort_flag = 1;
                // wait for the MMAs in flight before tensor memory is freed
                mma_commit(drain);
                volatile uint32_t never = 0;
                (void)mbar_wait(drain, 0, &never);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t aph = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const TileInfo ti = decode_tile(args, t);
            // tcgen05.ld is warp-collective: the whole warp proceeds or stops
            const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(tfull + acc, aph, abort_flag));
            if (!ok) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            if constexpr (EPI == kEpiPartial) {
                epi_partial<BN>(args, ti, taddr, row);
            } else {
                epi_router<BN>(args, ti, taddr, row);
            }
            tc_fence_before();
            mbar_arrive(tempty + acc);
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
        if (timed_out) *abort_flag = 1;
    }

    if (timed_out && args.status) atomicOr(args.status, kDevErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------- split-K router over a cluster --
//
// The router GEMM for batches whose 128-token tiles cannot fill the GPU
// ("MoE & MLA operators", sec. 2.2: logits = x W_g, then top-k and softmax):
// the K range is split into S slices, and the S CTAs that share one 128-token
// tile form a thread-block cluster (rank = slice).  Each CTA accumulates its
// slice's fp32 partial logits in tensor memory; slices 1..S-1 store theirs
// into slice 0's shared memory (distributed shared memory), and slice 0 sums
// them in slice order, adds the bias and picks the experts.  One launch, no
// global scratch, and a fixed summation order.

// Group limit, top-k and softmax of one token's logits held in registers (the
// bias already added).  The same rules as epi_router: a group's score is its
// largest logit, the topk_groups best groups stay eligible, top-k runs over
// the eligible experts in ascending index order with strict comparisons (the
// lower index wins a tie), the gates are a softmax over the k chosen logits.
template <int BN>
__device__ __forceinline__ void route_row(const GemmArgs& a, const float (&l)[BN], int token) {
    const int E = a.E, k = a.k;
    uint32_t gmask = 0xFFFFFFFFu;
    int gsz = E;
    if (a.n_groups > 0) {
        gsz = E / a.n_groups;
        float gs[32];
#pragma unroll
        for (int g = 0; g < 32; ++g) gs[g] = -FLT_MAX;
#pragma unroll
        for (int e = 0; e < BN; ++e)
            if (e < E) gs[e / gsz] = fmaxf(gs[e / gsz], l[e]);
        gmask = 0;
        for (int r = 0; r < a.topk_groups; ++r) {
            int bi = -1;
            float bv = -FLT_MAX;
            for (int g = 0; g < a.n_groups; ++g) {
                if (gmask & (1u << g)) continue;
                if (bi < 0 || gs[g] > bv) {
                    bi = g;
                    bv = gs[g];
                }
            }
            gmask |= 1u << bi;
        }
    }
    float tv[8];
    int te[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        tv[s] = -FLT_MAX;
        te[s] = -1;
    }
#pragma unroll
    for (int e = 0; e < BN; ++e) {
        if (e < E && ((gmask >> (e / gsz)) & 1u)) {
            float cv = l[e];
            int ci = e;
            bool shifting = false;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                if (s < k && (shifting || te[s] < 0 || cv > tv[s])) {
                    const float tf = tv[s];
                    const int tix = te[s];
                    tv[s] = cv;
                    te[s] = ci;
                    cv = tf;
                    ci = tix;
                    shifting = true;
                }
            }
        }
    }
    float sum = 0.0f;
#pragma unroll
    for (int s = 0; s < 8; ++s)
        if (s < k) sum += expf(tv[s] - tv[0]);
    const float inv = 1.0f / sum;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        if (s < k) {
            a.topk_idx[(int64_t)token * k + s] = te[s];
            a.topk_w[(int64_t)token * k + s] = expf(tv[s] - tv[0]) * inv;
        }
    }
}

// Shared memory of k_router_cluster beyond the GEMM ring: the partial logits
// that slices 1..S-1 hand to slice 0 ([S-1][128 rows][BN] fp32) and one flag
// per (slice, epilogue warp) saying that the warp's rows arrived.
template <int BN>
constexpr int router_cluster_smem(int S) {
    return GemmCfg<BN>::SMEM + (S - 1) * BM * BN * 4 + 4 * 8 * 4;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_router_cluster(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs args) {
    using C = GemmCfg<BN>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * C::A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S * C::B_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* tfull = bars + 2 * S;
    uint64_t* drain = tfull + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_holder + 1;
    const int nsl = args.n_tiles;  // slices = CTAs of the cluster
    float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + C::BAR_BYTES);
    int* arrived = reinterpret_cast<int*>(red + (nsl - 1) * BM * BN);  // [S-1][4]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int m0 = (blockIdx.x / nsl) * BM;
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        mbar_init(tfull, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        if (rank == 0)
            for (int i = 0; i < (nsl - 1) * 4; ++i) arrived[i] = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    // inputs written by earlier kernels are visible after the wait; tensor
    // memory is taken after it (see k_grouped_gemm)
    pdl_wait();
    if (warp == 1) tmem_alloc(tmem_holder, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // every CTA of the cluster runs (and slice 0's flags are clear)
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int kb0 = static_cast<int>(rank) * args.k_per_split;
    const int kb1 = min(kb0 + args.k_per_split, args.k_blocks);
    bool timed_out = false;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            uint32_t armed = 0, armed_par = 0;
            const int rot = k_rotation(kb1 - kb0);
            for (int kb = kb0, s = 0, ph = 0; kb < kb1; ++kb) {
                if (!mbar_wait(empty + s, ph ^ 1u, abort_flag)) {
                    timed_out = true;
                    break;
                }
                const int kx = rotated_k(kb, kb0, kb1, rot) * BK;
                mbar_arrive_expect_tx(full + s, C::STAGE_BYTES);
                tma_load_2d(sA + s * C::A_BYTES, &tmA, kx, m0, full + s);
                tma_load_2d(sB + s * C::B_BYTES, &tmB, kx, 0, full + s);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | (static_cast<uint32_t>(ph) << s);
                if (++s == S) {
                    s = 0;
                    ph ^= 1;
                }
            }
            if (timed_out || *abort_flag) {
                *abort_flag = 1;
                for (int i = 0; i < S; ++i)
                    if (armed & (1u << i)) {
                        volatile uint32_t never = 0;
                        (void)mbar_wait(full + i, (armed_par >> i) & 1u, &never);
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            bool issued = false;
            for (int kb = kb0, s = 0, ph = 0; kb < kb1; ++kb) {
                if (!mbar_wait(full + s, ph, abort_flag)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(sA + s * C::A_BYTES);
                const uint32_t b_addr = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_bf16(tmem_base, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(b_addr + kk * 32),
                             idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                issued = true;
                mma_commit(empty + s);
                if (++s == S) {
                    s = 0;
                    ph ^= 1;
                }
            }
            if (!timed_out) mma_commit(tfull);
            if ((timed_out || *abort_flag) && issued) {
                *abort_flag = 1;
                mma_commit(drain);
                volatile uint32_t never = 0;
                (void)mbar_wait(drain, 0, &never);
            }
        }
    }

    // epilogue warps: this thread's row of partial logits, out of tensor memory
    const int q = warp & 3;
    const int row = q * 32 + lane;
    float v[BN];
    bool have = false;
    if (warp >= 2) {
        have = __all_sync(0xFFFFFFFFu, mbar_wait(tfull, 0, abort_flag));
        if (have) {
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
            for (int c = 0; c < BN / 16; ++c) {
                uint32_t r[16];
                tmem_ld16(taddr + c * 16, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) v[c * 16 + i] = __uint_as_float(r[i]);
            }
            if (rank != 0) {
                // hand the row to slice 0, then flag the warp's rows as there
                const uint32_t dst =
                    mapa_shared(smem_u32(red + ((static_cast<int>(rank) - 1) * BM + row) * BN), 0);
#pragma unroll
                for (int i = 0; i < BN; i += 4) st_cluster_v4(dst + 4 * i, v[i], v[i + 1], v[i + 2], v[i + 3]);
                __syncwarp();
                if (lane == 0) {
                    const uint32_t f = mapa_shared(smem_u32(arrived + (static_cast<int>(rank) - 1) * 4 + q), 0);
                    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(f), "r"(1) : "memory");
                }
            }
        } else {
            timed_out = true;
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the partial rows are in slice 0's shared memory
    if (warp >= 2 && rank == 0 && have) {
        bool all = true;
        for (int i = 0; i < (nsl - 1); ++i) all = all && arrived[i * 4 + q] != 0;
        if (all) {
            // slice order: own slice (0), then 1 .. S-1
            for (int sl = 1; sl < nsl; ++sl) {
                const float4* p = reinterpret_cast<const float4*>(red + ((sl - 1) * BM + row) * BN);
#pragma unroll
                for (int i = 0; i < BN / 4; ++i) {
                    const float4 w = p[i];
                    v[4 * i] += w.x;
                    v[4 * i + 1] += w.y;
                    v[4 * i + 2] += w.z;
                    v[4 * i + 3] += w.w;
                }
            }
#pragma unroll
            for (int e = 0; e < BN; ++e)
                if (args.bias && e < args.E) v[e] += ld_dep(args.bias + e);
            if (m0 + row < args.dense_rows) route_row<BN>(args, v, m0 + row);
        } else {
            timed_out = true;  // a slice gave up: its rows never arrived
        }
    }
    if (timed_out && args.status) atomicOr(args.status, kDevErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------ CTA-pair (2-SM) kernel --
//
// The same grouped GEMM on CTA pairs (clusters of 2): one tcgen05.mma with
// cta_group::2 computes a 256 x BN tile whose A rows are split between the
// two CTAs (128 each) and whose B tile is split along N (BN/2 rows each), so
// each SM stages only half of the B operand.  The even CTA issues the MMAs;
// both CTAs run a TMA producer (completions counted on the even CTA's
// barriers) and an epilogue over their own 128 accumulator rows.
//
// A unit of work is a 256-row visit of one expert's segment: visits start at
// every 256th row of the segment (from padded_offsets), so the blocks of one
// expert are taken two (P = 128) or four (P = 64) at a time; rows of a visit
// past the segment's valid rows are computed but never stored.  Only real
// visits are enumerated, so the round-robin over CTA pairs stays balanced.

struct PairTile {
    int e, m0, lo, hi, nb;  // rows [m0 + lo, m0 + hi) of the visit are valid
};

// Visits of expert e are numbered from vpref[e] (exclusive prefix over the
// experts of ceil(blocks_e / (256 / P))); block i of expert e is block
// padded_offsets[e] / P + i of the table, so a visit maps to its first block
// without any search of the table itself.
__device__ __forceinline__ PairTile decode_pair(const GemmArgs& a, int t, const int* vpref) {
    PairTile p;
    const int v = t / a.n_tiles;
    p.nb = t - v * a.n_tiles;
    p.lo = 0;
    if (!a.block_metadata && !a.unpadded) {
        p.e = 0;
        p.m0 = v * 256;
        p.hi = min(256, a.dense_rows - p.m0);
        return p;
    }
    int lo = 0, hi = a.n_experts;  // largest e with vpref[e] <= v
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (vpref[mid] <= v) lo = mid; else hi = mid;
    }
    p.e = lo;
    if (a.unpadded) {
        // the experts' rows lie back to back (padded_offsets holds the plain
        // group offsets): visit v of expert e is the 256-row window
        // first + (v - vpref[e]) of the rows, of which the rows inside
        // [start_e, end_e) are stored; a window cut by an expert boundary
        // is visited once for each expert it holds
        const int s0 = ld_dep(a.padded_offsets + lo), s1 = ld_dep(a.padded_offsets + lo + 1);
        p.m0 = (s0 / 256 + (v - vpref[lo])) * 256;
        p.lo = max(s0 - p.m0, 0);
        p.hi = min(s1 - p.m0, 256);
        return p;
    }
    const int per = 256 / a.block_rows;
    const int mb = ld_dep(a.padded_offsets + lo) / a.block_rows + (v - vpref[lo]) * per;
    const int32_t* bm = a.block_metadata;
    p.m0 = ld_dep(bm + 3 * mb + 1);
    p.hi = ld_dep(bm + 3 * mb + 2);
    const int bend = ld_dep(a.padded_offsets + lo + 1) / a.block_rows;  // next expert's first block
    for (int j = 1; j < per && mb + j < bend; ++j) p.hi += ld_dep(bm + 3 * (mb + j) + 2);
    return p;
}

// Epilogue of the pair kernel with coalesced output: a warp whose 32 rows are
// all valid stages each 32 x 64 box of bf16 outputs in shared memory (the
// 128-byte swizzle the store tensor map expects) and writes it with one TMA
// bulk store; the two 4 KB staging buffers of the warp alternate.  Warps with
// any row past the visit's valid rows take the per-thread path, which stores
// valid rows only.
template <int BN, int EPI>
__device__ __forceinline__ void epi_pair(const GemmArgs& a, const TileInfo& ti, uint32_t taddr,
                                         int q, int lane, uint8_t* stage, const CUtensorMap* tmOut,
                                         int& buf, const int (&pr)[8]) {
    const int row = q * 32 + lane;
    if (q * 32 < ti.lo || q * 32 + 32 > ti.hi) {
        if constexpr (EPI == kEpiSwiGLU) epi_swiglu(a, ti, taddr, row);
        else if constexpr (EPI == kEpiCombine) epi_combine<BN>(a, ti, taddr, row, pr);
        else epi_gate<BN>(a, ti, taddr, row);
        return;
    }
    constexpr int NCH = EPI == kEpiSwiGLU ? 2 : BN / 64;  // 64-column output boxes
    const int col0 = EPI == kEpiSwiGLU ? ti.nb * 128 : ti.nb * BN;
    const float gate = (EPI == kEpiGate && a.row_gate) ? ld_dep(a.row_gate + ti.m0 + row) : 1.0f;
    const float* cs = tile_scales(a, ti, EPI == kEpiSwiGLU ? ti.nb * 256 : ti.nb * BN);
#pragma unroll 1
    for (int c = 0; c < NCH; ++c) {
        if (lane == 0) bulk_wait_read<1>();  // this buffer's previous store has read it
        __syncwarp();
        uint8_t* sb = stage + buf * 4096 + lane * 128;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t p[16];
            if constexpr (EPI == kEpiSwiGLU) {
                uint32_t g[32], u[32];
                tmem_ld32(taddr + c * 64 + half * 32, g);
                tmem_ld32(taddr + 128 + c * 64 + half * 32, u);
                tmem_ld_wait();
                if (cs) {
                    scale_cols(g, cs + c * 64 + half * 32);
                    scale_cols(u, cs + 128 + c * 64 + half * 32);
                }
                if (a.gu_out) save_gate_up(a, ti, row, c * 64 + half * 32, g, u);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                    const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
                    p[i] = pack_bf16x2(silu_f32(g0) * u0, silu_f32(g1) * u1);
                }
            } else if constexpr (EPI == kEpiCombine) {
                float sum[32];
                combine_sum32(a, pr, col0 + c * 64 + half * 32, sum);
                uint32_t v[32];
                tmem_ld32(taddr + c * 64 + half * 32, v);
                tmem_ld_wait();
                if (cs) scale_cols(v, cs + c * 64 + half * 32);
#pragma unroll
                for (int i = 0; i < 16; ++i) p[i] = combine_pack2(sum[2 * i], sum[2 * i + 1], v[2 * i], v[2 * i + 1]);
            } else {
                uint32_t v[32];
                tmem_ld32(taddr + c * 64 + half * 32, v);
                tmem_ld_wait();
                if (cs) scale_cols(v, cs + c * 64 + half * 32);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    p[i] = pack_bf16x2(gate * __uint_as_float(v[2 * i]), gate * __uint_as_float(v[2 * i + 1]));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int chunk = half * 4 + j;  // 16-byte chunk of the 128-byte row
                *reinterpret_cast<uint4*>(sb + ((chunk ^ (lane & 7)) << 4)) =
                    make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmOut, stage + buf * 4096, col0 + c * 64, ti.m0 + q * 32);
            bulk_commit();
        }
        buf ^= 1;
    }
}

// GATHER: the A rows are gathered from the token rows with TMA gather4 (the
// permute fused into GEMM1's A load) instead of a tile load from the
// permuted buffer.
template <int BN, int EPI, bool GATHER>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    k_grouped_gemm_pair(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmOut, const GemmArgs args) {
    constexpr int BH = BN / 2;  // B rows staged by each CTA
    // K blocks per stage.  A and B are loaded as 3D tensors [K block][row][64]
    // whose {64, rows, 2} box lands as two 128-byte-swizzled tiles back to
    // back: one TMA operation per operand carries two K blocks (3 stages of
    // 64 KB instead of 6 of 32 KB), half the operations for the same bytes in
    // flight.  The gather variant keeps one K block per stage.
    constexpr int KP = GATHER ? 1 : 2;
    constexpr int A_TILE = BM * BK * 2, B_TILE = BH * BK * 2;
    constexpr int A_BYTES = A_TILE * KP;
    constexpr int B_BYTES = B_TILE * KP;
    constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    constexpr int S = (196 * 1024) / STAGE_BYTES > 8 ? 8 : (196 * 1024) / STAGE_BYTES;
    constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
    static_assert(B_BYTES % 1024 == 0, "B stage must keep 1024-byte alignment");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * A_BYTES;
    uint8_t* sOut = sB + S * B_BYTES;  // 4 epilogue warps x 2 x 4 KB staging
    uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + kOutStageBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* tfull = bars + 2 * S;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_holder + 1;
    int* vpref = reinterpret_cast<int*>(bars + 64);  // [E + 1]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full + i, 1);  // the even CTA's producer (+ transaction bytes)
            mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull + i, 1);
            mbar_init(tempty + i, 8);  // one arrival per epilogue warp of both CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (threadIdx.x == 32) tma_prefetch_desc(&tmOut);
    // inputs written by earlier kernels are visible from here on; tensor
    // memory is taken after the wait, as in k_grouped_gemm
    pdl_wait();
    if (warp == 1) tmem_alloc_pair(tmem_holder, TMEM_COLS);
    if (warp == 2 && (args.block_metadata || args.unpadded)) {
        // per-expert visit counts from the segment sizes, exclusive warp scan
        const int per = args.unpadded ? 1 : 256 / args.block_rows;
        int running = 0;
        for (int base = 0; base < args.n_experts; base += 32) {
            const int e = base + lane;
            int nv = 0;
            if (e < args.n_experts) {
                const int s0 = ld_dep(args.padded_offsets + e), s1 = ld_dep(args.padded_offsets + e + 1);
                if (args.unpadded) {
                    nv = s1 > s0 ? (s1 - 1) / 256 - s0 / 256 + 1 : 0;  // windows the rows touch
                } else {
                    const int nblk = (s1 - s0) / args.block_rows;
                    nv = (nblk + per - 1) / per;
                }
            }
            int x = nv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            if (e < args.n_experts) vpref[e] = running + x - nv;
            running += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
        if (lane == 0) vpref[args.n_experts] = running;
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers are initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int nvisits = (args.block_metadata || args.unpadded) ? vpref[args.n_experts]
                                                                : (args.dense_rows + 255) / 256;
    const int total = nvisits * args.n_tiles;
    const int cluster = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;
    bool timed_out = false;

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        // Lane 0 loads the B half (and the A tile from the permuted buffer);
        // in the gather variant every lane also gathers 4 of this CTA's 128
        // A rows straight from the token rows (row_src[r] / k) with one
        // gather4 per k-step (4 rows x 128 bytes at offset 512 * lane of the
        // 128-byte-swizzled A stage).
        int s = 0;
        uint32_t ph = 0;
        uint32_t armed = 0, armed_par = 0;
        // an expert's weight panels are re-read by every visit of that
        // expert: keep them in L2 ahead of the streamed activation rows
        const uint64_t keep = l2_policy_evict_last();
        // Consecutive waves of the pair grid run the K loop in opposite
        // directions: a wave's CTA pairs share the weight panels of one expert
        // with the wave before, and starting where that wave stopped finds the
        // panels' last-loaded K blocks still in L2 (GEMM1 at the default
        // workload read 19 % fewer DRAM bytes).  The accumulation order of a
        // tile is fixed by its position in the visit list.
        int wave = 0;
        for (int t = cluster; t < total && !timed_out; t += nclusters, ++wave) {
            const PairTile p = decode_pair(args, t, vpref);
            if (args.cp_out) {
                // the visit's A rows are written by the copy warps of every
                // CTA: load them once all of them are in place
                bool ready = true;
                if (lane == 0) {
                    ready = wait_count(args.cp_ready + t / args.n_tiles, p.hi, abort_flag);
                    fence_proxy_async_global();
                }
                if (!__shfl_sync(0xFFFFFFFFu, ready, 0)) {
                    timed_out = true;
                    break;
                }
            }
            const bool rev = wave & 1;
            const int arow = p.m0 + BM * static_cast<int>(rank);
            const int brow = p.e * args.b_rows_per_expert + p.nb * BN + BH * static_cast<int>(rank);
            int grow[4] = {0, 0, 0, 0};
            if (GATHER) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int rr = BM * static_cast<int>(rank) + 4 * lane + j;  // row in the visit
                    // rows past the visit's valid rows are computed but never
                    // stored: any in-range token row will do
                    if (rr < p.hi) grow[j] = ld_dep(args.row_src + p.m0 + rr) / args.gather_k;
                }
            }
            const int n_steps = (args.k_blocks + KP - 1) / KP;
            for (int kb = 0; kb < n_steps; ++kb) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait(empty + s, ph ^ 1u, abort_flag);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (!ok) {
                    timed_out = true;
                    break;
                }
                const uint32_t full_leader = mapa_shared(smem_u32(full + s), 0);
                if (lane == 0) {
                    armed &= ~(1u << s);
                    if (leader) mbar_arrive_expect_tx(full + s, 2 * STAGE_BYTES);
                    const int kstep = rev ? n_steps - 1 - kb : kb;
                    if constexpr (!GATHER) {
                        tma_load_3d_pair(sA + s * A_BYTES, &tmA, 0, arow, kstep * KP, full_leader);
                        tma_load_3d_pair_hint(sB + s * B_BYTES, &tmB, 0, brow, kstep * KP, full_leader,
                                              keep);
                    } else {
                        tma_load_2d_pair_hint(sB + s * B_BYTES, &tmB, kstep * BK, brow, full_leader, keep);
                    }
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                }
                if (GATHER)
                    tma_gather4_pair(smem_u32(sA + s * A_BYTES) + lane * 512u, &tmA,
                                     (rev ? n_steps - 1 - kb : kb) * BK, grow[0],
                                     grow[1], grow[2], grow[3], full_leader);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (lane == 0 && (timed_out || *abort_flag) && leader) {
            *abort_flag = 1;
            for (int i = 0; i < S; ++i)
                if (armed & (1u << i)) {
                    volatile uint32_t never = 0;
                    (void)mbar_wait(full + i, (armed_par >> i) & 1u, &never);
                }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN);
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool issued = false;
            for (int t = cluster; t < total && !timed_out; t += nclusters) {
                if (!mbar_wait(tempty + acc, aph ^ 1u, abort_flag)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                const int n_steps = (args.k_blocks + KP - 1) / KP;
                for (int kb = 0; kb < n_steps; ++kb) {
                    if (!mbar_wait(full + s, ph, abort_flag)) {
                        timed_out = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + s * A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + s * B_BYTES);
#pragma unroll
                    for (int kp = 0; kp < KP; ++kp)
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            mma_bf16_pair(d_tmem, sdesc_sw128(a_addr + kp * A_TILE + kk * 32),
                                          sdesc_sw128(b_addr + kp * B_TILE + kk * 32), idesc,
                                          (kb | kp | kk) != 0 ? 1u : 0u);
                        }
                    issued = true;
                    mma_commit_pair(empty + s, 0x3);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (timed_out) break;
                mma_commit_pair(tfull + acc, 0x3);
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
            }
            if ((timed_out || *abort_flag) && issued) {
                *abort_flag = 1;
                mma_commit_pair(drain, 0x1);
                volatile uint32_t never = 0;
                (void)mbar_wait(drain, 0, &never);
            }
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;
        uint8_t* stage = sOut + (warp - 2) * 8192;
        int buf = 0;
        int acc = 0;
        uint32_t aph = 0;
        for (int t = cluster; t < total; t += nclusters) {
            const PairTile p = decode_pair(args, t, vpref);
            TileInfo ti;
            ti.e = p.e;
            ti.nb = p.nb;
            ti.m0 = p.m0 + BM * static_cast<int>(rank);
            ti.lo = max(0, p.lo - BM * static_cast<int>(rank));
            ti.hi = min(BM, p.hi - BM * static_cast<int>(rank));
            ti.skip = false;
            int pr[8];
            if constexpr (EPI == kEpiCombine) {
                // the token's routed rows, and their BN columns of this tile
                // fetched into L2 while the tile's MMAs run
                combine_rows_of(args, ti.m0 + row, row >= ti.lo && row < ti.hi, pr);
                const __nv_bfloat16* y = static_cast<const __nv_bfloat16*>(args.comb_y);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (pr[j] >= 0)
                        bulk_prefetch_l2(y + (int64_t)pr[j] * args.comb_ldy + (int64_t)ti.nb * BN, BN * 2);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) pr[j] = -1;
            }
            const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(tfull + acc, aph, abort_flag));
            if (!ok) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            epi_pair<BN, EPI>(args, ti, taddr, q, lane, stage, &tmOut, buf, pr);
            tc_fence_before();
            __syncwarp();
            // relaxed: the accumulator's reads are complete and the MMA warp
            // reads nothing this warp wrote (a release arrive would wait for
            // the tile's stores to land)
            if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(tempty + acc), 0));
            if constexpr (EPI == kEpiSwiGLU) {
                if (args.perm_out) permute_slice(args, ti, q, lane);
            }
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
        if (lane == 0) bulk_wait_all();  // staged stores done before shared memory goes
        if (timed_out) *abort_flag = 1;
    } else if (args.cp_out) {
        // --------------------------------------------------- copy warps
        // The permute ("MoE & MLA operators", sec. 2.3) for GEMM1's A
        // operand: padded row r <- token row row_src[r] / k, the rows dealt
        // out over the two copy warps of every CTA in ascending order (the
        // order the visits are loaded in), a warp per row with 16 vectors in
        // flight per lane.  After each row the warp publishes it (fence,
        // then a count per visit).  These warps wait on nothing.
        const int cw = warp - 6;
        const int R = ld_dep(args.padded_offsets + args.n_experts);
        const uint4* xs = static_cast<const uint4*>(args.cp_x);
        uint4* xd = static_cast<uint4*>(args.cp_out);
        const int nvec = args.cp_nvec;
        int e = 0, po0 = 0;
        int po1 = ld_dep(args.padded_offsets + 1);
        for (int r = static_cast<int>(blockIdx.x) * 2 + cw; r < R; r += 2 * static_cast<int>(gridDim.x)) {
            while (r >= po1) {  // the expert of row r (rows ascend)
                ++e;
                po0 = po1;
                po1 = ld_dep(args.padded_offsets + e + 1);
            }
            const int src = ld_dep(args.cp_row_src + r);
            if (src < 0) continue;  // a pad row: read by no stored output
            const uint4* s = xs + static_cast<int64_t>(src / args.cp_k) * nvec;
            uint4* d = xd + static_cast<int64_t>(r) * nvec;
            for (int v0 = lane; v0 < nvec; v0 += 32 * 16) {
                uint4 b[16];
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    if (v0 + 32 * u < nvec) b[u] = ld_dep(s + v0 + 32 * u);
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    if (v0 + 32 * u < nvec) d[v0 + 32 * u] = b[u];
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence();
                atomicAdd(args.cp_ready + vpref[e] + (r - po0) / 256, 1);
            }
        }
    }

    if (timed_out && args.status) atomicOr(args.status, kDevErrTimeout);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its pair may still touch its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host --

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled encode_fn() {
    static PFN_encodeTiled fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_encodeTiled>(p);
    }
    return fn;
}

// Row-major bf16 matrix [rows, cols] as a 2D tensor map with a
// {box_cols, box_rows} box and the 128-byte swizzle; out-of-range rows read
// as zero.
static bool make_tmap_box(CUtensorMap* tm, const void* ptr, int64_t rows, int64_t cols, int box_cols,
                          int box_rows) {
    PFN_encodeTiled enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tensor_map_2d(void* tmap, const void* ptr, int64_t rows, int64_t cols, int elem_bytes,
                        int dtype, int box_cols, int box_rows, int swizzle_bytes) {
    PFN_encodeTiled enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * static_cast<cuuint64_t>(elem_bytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(static_cast<CUtensorMap*>(tmap), static_cast<CUtensorMapDataType>(dtype), 2,
                     const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                     : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// K-major operand [rows, K]: {64, box_rows} boxes.
static bool make_tmap(CUtensorMap* tm, const void* ptr, int64_t rows, int64_t K, int box_rows) {
    return make_tmap_box(tm, ptr, rows, K, BK, box_rows);
}

// K-major operand [rows, K] seen as [K / 64][rows][64]: a {64, box_rows, 2}
// box carries two K blocks, landing as two 128-byte-swizzled tiles back to
// back.  K blocks past the last read as zero.
static bool make_tmap_kpair(CUtensorMap* tm, const void* ptr, int64_t rows, int64_t K, int box_rows) {
    PFN_encodeTiled enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(BK), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(K / BK)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(BK) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN, int EPI>
static cudaError_t launch_t(const CUtensorMap& tA, const CUtensorMap& tB, const GemmArgs& args,
                            int max_tiles, cudaStream_t stream) {
    using C = GemmCfg<BN>;
    static bool attr_done[64] = {};  // per device (small device counts)
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_grouped_gemm<BN, EPI>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    int grid = num_sms();
    if (max_tiles < grid) grid = max_tiles;
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(k_grouped_gemm<BN, EPI>, dim3(grid), dim3(kThreads), C::SMEM, stream, tA, tB,
                      args);
}

template <int BN>
static cudaError_t launch_router_cluster_t(const CUtensorMap& tA, const CUtensorMap& tB,
                                           const GemmArgs& args, int m_tiles, int slices,
                                           cudaStream_t stream) {
    const int smem = router_cluster_smem<BN>(slices);
    static int attr_smem[64] = {};  // per device: the largest size set so far
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64) return cudaErrorInvalidDevice;
    if (attr_smem[dev] < smem) {
        cudaError_t e = cudaFuncSetAttribute(k_router_cluster<BN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_smem[dev] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(m_tiles * slices, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = slices;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_router_cluster<BN>, tA, tB, args);
}

bool router_cluster_fits(int bn, int slices) {
    // up to 4 slices: with 8 the clustered launch (8 co-scheduled CTAs of up
    // to 206 KB each) measured slower than partial logits + a reduce kernel
    if (slices < 2 || slices > 4) return false;
    switch (bn) {
        case 16: return router_cluster_smem<16>(slices) <= 232448;
        case 32: return router_cluster_smem<32>(slices) <= 232448;
        case 64: return router_cluster_smem<64>(slices) <= 232448;
        default: return false;
    }
}

cudaError_t launch_router_cluster(int bn, const void* x, int64_t T, const void* Wg_t, int64_t E,
                                  int64_t K, const GemmArgs& args, int slices, cudaStream_t stream) {
    if (!router_cluster_fits(bn, slices)) return cudaErrorInvalidValue;
    CUtensorMap tA, tB;
    if (!make_tmap(&tA, x, T, K, BM) || !make_tmap(&tB, Wg_t, E, K, bn)) return cudaErrorInvalidValue;
    const int m_tiles = static_cast<int>((T + BM - 1) / BM);
    switch (bn) {
        case 16: return launch_router_cluster_t<16>(tA, tB, args, m_tiles, slices, stream);
        case 32: return launch_router_cluster_t<32>(tA, tB, args, m_tiles, slices, stream);
        case 64: return launch_router_cluster_t<64>(tA, tB, args, m_tiles, slices, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int BN, int EPI, bool GATHER>
static cudaError_t launch_pair_t(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tO,
                                 const GemmArgs& args, int max_visits, cudaStream_t stream) {
    constexpr int NT = kPairThreads;
    constexpr int STAGE_BYTES = (BM * BK * 2 + (BN / 2) * BK * 2) * (GATHER ? 1 : 2);
    constexpr int S = (196 * 1024) / STAGE_BYTES > 8 ? 8 : (196 * 1024) / STAGE_BYTES;
    constexpr int SMEM = 1024 + S * STAGE_BYTES + kOutStageBytes + 512 + 4 * 260;
    static_assert(SMEM <= 232448, "shared memory budget");
    static int max_clusters[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64) return cudaErrorInvalidDevice;
    if (!max_clusters[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_grouped_gemm_pair<BN, EPI, GATHER>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
        cfg.blockDim = dim3(NT, 1, 1);
        cfg.dynamicSmemBytes = SMEM;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, k_grouped_gemm_pair<BN, EPI, GATHER>, &cfg);
        if (e != cudaSuccess || n <= 0) n = num_sms() / 2;
        max_clusters[dev] = n;
    }
    int clusters = max_clusters[dev];
    if (max_visits < clusters) clusters = max_visits;
    if (clusters <= 0) return cudaSuccess;
    // the two copy warps only when GEMM1 does the permute
    const int nt = args.cp_out ? NT : kThreads;
    return launch_pdl(k_grouped_gemm_pair<BN, EPI, GATHER>, dim3(2 * clusters), dim3(nt), SMEM, stream,
                      tA, tB, tO, args);
}

cudaError_t launch_grouped_gemm(int epi, int bn, const void* A, int64_t rowsA, const void* B,
                                int64_t rowsB, int64_t K, const GemmArgs& args, int max_tiles,
                                cudaStream_t stream) {
    CUtensorMap tA, tB;
    const bool pair = epi != kEpiRouter && epi != kEpiPartial;
    const bool kpair = pair && epi != kEpiSwiGLUGather;
    const int a_box = epi == kEpiSwiGLUGather ? 1 : BM;  // gather4 reads one-row boxes
    if (kpair) {
        if (!make_tmap_kpair(&tA, A, rowsA, K, BM) || !make_tmap_kpair(&tB, B, rowsB, K, bn / 2))
            return cudaErrorInvalidValue;
    } else if (!make_tmap(&tA, A, rowsA, K, a_box) || !make_tmap(&tB, B, rowsB, K, pair ? bn / 2 : bn)) {
        return cudaErrorInvalidValue;
    }
    if (pair) {
        // the output as a [rows, ldo] bf16 tensor for the staged TMA stores
        CUtensorMap tO;
        if (!make_tmap_box(&tO, args.out, args.out_rows, args.ldo, 64, 32)) return cudaErrorInvalidValue;
        if (epi == kEpiCombine &&
            (args.comb_k < 1 || args.comb_k > 8 || !args.comb_y || !args.comb_perm))
            return cudaErrorInvalidValue;
        if (epi == kEpiSwiGLU && bn == 256)
            return launch_pair_t<256, kEpiSwiGLU, false>(tA, tB, tO, args, max_tiles, stream);
        if (epi == kEpiSwiGLUGather && bn == 256)
            return launch_pair_t<256, kEpiSwiGLU, true>(tA, tB, tO, args, max_tiles, stream);
        if (epi == kEpiGate && bn == 256)
            return launch_pair_t<256, kEpiGate, false>(tA, tB, tO, args, max_tiles, stream);
        if (epi == kEpiGate && bn == 128)
            return launch_pair_t<128, kEpiGate, false>(tA, tB, tO, args, max_tiles, stream);
        if (epi == kEpiCombine && bn == 256)
            return launch_pair_t<256, kEpiCombine, false>(tA, tB, tO, args, max_tiles, stream);
        if (epi == kEpiCombine && bn == 128)
            return launch_pair_t<128, kEpiCombine, false>(tA, tB, tO, args, max_tiles, stream);
        return cudaErrorInvalidValue;
    }
    if (epi == kEpiPartial) {
        switch (bn) {
            case 16: return launch_t<16, kEpiPartial>(tA, tB, args, max_tiles, stream);
            case 32: return launch_t<32, kEpiPartial>(tA, tB, args, max_tiles, stream);
            case 64: return launch_t<64, kEpiPartial>(tA, tB, args, max_tiles, stream);
            case 128: return launch_t<128, kEpiPartial>(tA, tB, args, max_tiles, stream);
            case 256: return launch_t<256, kEpiPartial>(tA, tB, args, max_tiles, stream);
            default: break;
        }
    } else if (epi == kEpiRouter) {
        switch (bn) {
            case 16: return launch_t<16, kEpiRouter>(tA, tB, args, max_tiles, stream);
            case 32: return launch_t<32, kEpiRouter>(tA, tB, args, max_tiles, stream);
            case 64: return launch_t<64, kEpiRouter>(tA, tB, args, max_tiles, stream);
            case 128: return launch_t<128, kEpiRouter>(tA, tB, args, max_tiles, stream);
            case 256: return launch_t<256, kEpiRouter>(tA, tB, args, max_tiles, stream);
            default: break;
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
