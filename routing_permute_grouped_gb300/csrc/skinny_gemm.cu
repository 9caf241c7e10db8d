// skinny_gemm.cu -- the grouped expert GEMMs for blocks with few token rows
// (decode-sized batches), with bf16 or e4m3 expert weights.
//
// With a handful of rows per expert the token rows cannot fill the MMA's
// M = 128, so the operands are swapped: a tile multiplies 256 rows of one
// expert's K-major weight matrix (two M = 128 halves) by the token rows of one
// block of the table, which become the MMA's N:
//     D^T[f, t] = sum_k W[f, k] X[t, k]
// and the epilogue writes D back into the row-major h / y.  The weights pass
// through the SM once per tile; at decode sizes every (expert, panel) is
// visited by one tile, so the kernel's time is the weight bytes over the HBM
// bandwidth ("Dropless and grouped GEMM", sec. 10: the small-M decode layout
// with valid rows per expert; the block table stays the work list).
//
// bf16 weights: stages of [256 weight rows | <= 128 token rows] x 64 K, bf16
// MMAs (kind::f16, K = 16).
//
// e4m3 weights ("MoE & MLA operators", sec. 6.1: one byte per weight;
// "Dropless and grouped GEMM", sec. 12: the scale multiplies the product when
// one scale covers the whole contraction): stages of [256 weight rows | 2 x
// <= 64 token rows] x 128 K, 8-bit MMAs (kind::f8f6f4, K = 32) straight from
// the staged codes.  An N = 16 MMA costs the tensor pipe about as much as a
// 128-column one, so at decode sizes the MMA count per weight byte sets the
// pace; 8-bit MMAs take half as many as widening the weights to 16 bits would.
// The token rows come as e4m3 pairs (hi, lo) with a power-of-two row scale
// (ptx.cuh), interleaved as rows 2r and 2r + 1, so the MMA computes both
// halves as neighbouring columns and the epilogue adds them: the product with
// the 16-bit activation is exact up to 2^-10 of the row's largest value.  The
// epilogue multiplies by the row scale and by the weights' per-output-channel
// scale.  Tiles hold at most 64 token rows; a block with more is split into
// chunks of 64, ordered chunk-major so that decode (one chunk) keeps a
// balanced round-robin.
//
// Tile list, built on the device from the block table: routed tile t is
// chunk t / (nb * n_panels) of panel (t % (nb * n_panels)) / nb of block
// t % nb, so neighbouring CTAs read the same weight panel for the blocks of
// one expert; the dense shared expert's tiles follow in the same launch.
//
// Warp roles, one CTA per SM (192 threads):
//   warp 0        TMA producer: weight panels and token rows
//   warp 1        TMEM allocation; one lane issues the MMAs
//   warps 2..5    epilogue
// Every wait is bounded; on a timeout the CTA flags the status word, lets its
// copies and MMAs in flight finish and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kWRows = 256;            // weight rows per tile (two M = 128 halves)
constexpr int kABytes = kWRows * 128;  // 256 rows x 128 bytes, swizzled
constexpr uint32_t kErrRange = 0x1u;   // expert id outside [0, E)
constexpr uint32_t kErrTimeout = 0x2u;

template <bool FP8>
struct SkCfg {
    static constexpr int NMAX = FP8 ? 64 : 128;      // token rows per tile
    static constexpr int BROWS = FP8 ? 2 * NMAX : NMAX;  // staged token rows (e4m3: hi and lo)
    static constexpr int KSTEP = FP8 ? 128 : 64;     // K per stage (128 bytes per row)
    static constexpr int STAGE = kABytes + BROWS * 128;
    static constexpr int S = 4;
    // TMEM: two accumulator buffers of two halves of BROWS columns
    static constexpr uint32_t HALF = BROWS;
    static constexpr uint32_t ACC_STRIDE = 2 * BROWS;
    static constexpr int BARS = 2 * S + 5;
    static constexpr int SMEM = 1024 + S * STAGE + BARS * 8 + 16;
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(2 * ACC_STRIDE <= 512, "tensor memory budget");
    static_assert(STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

struct SkTile {
    int e, m0, vm, p;
    bool shared, ok, skip;  // skip: an empty chunk of a block, not an error
};

template <int NMAX>
__device__ __forceinline__ SkTile sk_tile(const SkinnyArgs& a, int nb, int t) {
    SkTile x;
    x.skip = false;
    const int per_chunk = nb * a.n_panels;
    const int nr = per_chunk * a.n_chunks;
    if (t < nr) {
        const int c = t / per_chunk;
        const int rest = t - c * per_chunk;
        x.p = rest / nb;
        const int b = rest - x.p * nb;
        x.e = ld_dep(a.block_metadata + 3 * b);
        x.m0 = ld_dep(a.block_metadata + 3 * b + 1);
        x.vm = ld_dep(a.block_metadata + 3 * b + 2);
        x.shared = false;
        x.ok = x.e >= 0 && x.e < a.n_experts && x.m0 >= 0 && x.vm > 0 &&
               static_cast<int64_t>(x.m0) < a.out_rows;
        if (x.ok) {
            const int64_t room = a.out_rows - x.m0;
            x.vm = min(x.vm, 128);
            if (room < x.vm) x.vm = static_cast<int>(room);
            const int off = c * NMAX;
            if (x.vm <= off) {
                x.ok = false;
                x.skip = true;
            } else {
                x.m0 += off;
                x.vm = min(NMAX, x.vm - off);
            }
        }
    } else {
        const int ts = t - nr;
        const int nch = (a.s_rows + NMAX - 1) / NMAX;
        x.p = ts / nch;
        const int c = ts - x.p * nch;
        x.e = 0;
        x.m0 = c * NMAX;
        x.vm = min(NMAX, a.s_rows - x.m0);
        x.shared = true;
        x.ok = true;
    }
    return x;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

template <int EPI, bool FP8>
__global__ void __launch_bounds__(192, 1)
    k_grouped_gemm_skinny(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                          const __grid_constant__ CUtensorMap tAs, const __grid_constant__ CUtensorMap tBs,
                          const SkinnyArgs args) {
    using C = SkCfg<FP8>;
    constexpr int S = C::S;
    constexpr int STAGE = C::STAGE;
    constexpr int NMAX = C::NMAX;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * STAGE);
    uint64_t* full = bars;       // stage landed
    uint64_t* empty = full + S;  // stage consumed by the MMA
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_holder + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull + i, 1);
            mbar_init(tempty + i, 4);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tA);
        tma_prefetch_desc(&tB);
        if (args.s_rows > 0) {
            tma_prefetch_desc(&tAs);
            tma_prefetch_desc(&tBs);
        }
    }
    // The block table and the token rows are visible after pdl_wait().
    // Tensor memory is taken after the wait: every earlier kernel of the
    // stream has then released its own, and no later one holds any yet.
    pdl_wait();
    if (warp == 1) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    int nb = args.num_blocks ? ld_dep(args.num_blocks) : 0;  // null: shared-expert tiles only
    nb = nb < 0 ? 0 : (nb > args.nb_cap ? args.nb_cap : nb);
    const int total = nb * args.n_panels * args.n_chunks +
                      (args.s_rows > 0 ? ((args.s_rows + NMAX - 1) / NMAX) * args.s_panels : 0);
    bool timed_out = false;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;  // stages with copies not yet seen landed
            for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
                const SkTile x = sk_tile<NMAX>(args, nb, t);
                if (!x.ok) continue;
                const CUtensorMap* ta = x.shared ? &tAs : &tA;
                const CUtensorMap* tb = x.shared ? &tBs : &tB;
                const int arow = (x.shared ? 0 : x.e * args.rows_per_expert) + x.p * kWRows;
                const int kbs = x.shared ? args.s_k_blocks : args.k_blocks;
                // e4m3: token row r is the row pair (2r, 2r + 1) of the staged operand
                const int brow = FP8 ? 2 * x.m0 : x.m0;
                const int nbox = ((FP8 ? 2 * x.vm : x.vm) + 15) >> 4;
                for (int kb = 0; kb < kbs; ++kb) {
                    if (!mbar_wait(empty + s, ph ^ 1u, abort_flag)) {
                        timed_out = true;
                        break;
                    }
                    armed &= ~(1u << s);
                    uint8_t* st = smem + s * STAGE;
                    mbar_arrive_expect_tx(full + s, kABytes + nbox * 2048);
                    tma_load_2d(st, ta, kb * C::KSTEP, arow, full + s);
                    for (int j = 0; j < nbox; ++j)
                        tma_load_2d(st + kABytes + j * 2048, tb, kb * C::KSTEP, brow + 16 * j, full + s);
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
            const uint32_t idesc0 = FP8 ? idesc_e4m3_f32(128, 8) : idesc_bf16_f32(128, 8);
            const uint32_t idesc_base = idesc0 & ~(0x3Fu << 17);
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool issued = false;
            for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
                const SkTile x = sk_tile<NMAX>(args, nb, t);
                if (!x.ok) continue;
                const int kbs = x.shared ? args.s_k_blocks : args.k_blocks;
                const uint32_t n = static_cast<uint32_t>(((FP8 ? 2 * x.vm : x.vm) + 15) & ~15);
                const uint32_t idesc = idesc_base | ((n >> 3) << 17);
                if (!mbar_wait(tempty + acc, aph ^ 1u, abort_flag)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc) * C::ACC_STRIDE;
                for (int kb = 0; kb < kbs; ++kb) {
                    if (!mbar_wait(full + s, ph, abort_flag)) {
                        timed_out = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * STAGE);
                    const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {  // 4 x 32 bytes of each 128-byte row
                        const uint64_t bd = sdesc_sw128(b_addr + kk * 32);
                        const uint64_t a0 = sdesc_sw128(a_addr + kk * 32);
                        const uint64_t a1 = sdesc_sw128(a_addr + 16384 + kk * 32);
                        const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
                        if constexpr (FP8) {
                            mma_e4m3(d0, a0, bd, idesc, accum);
                            mma_e4m3(d0 + C::HALF, a1, bd, idesc, accum);
                        } else {
                            mma_bf16(d0, a0, bd, idesc, accum);
                            mma_bf16(d0 + C::HALF, a1, bd, idesc, accum);
                        }
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
            const SkTile x = sk_tile<NMAX>(args, nb, t);
            if (!x.ok) {
                if (!x.skip && warp == 2 && lane == 0 && args.status) atomicOr(args.status, kErrRange);
                continue;
            }
            const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(tfull + acc, aph, abort_flag));
            if (!ok) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            const uint32_t t0 = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                static_cast<uint32_t>(acc) * C::ACC_STRIDE;
            const int n = ((FP8 ? 2 * x.vm : x.vm) + 15) & ~15;  // accumulator columns
            const int rpe = x.shared ? args.s_rows_per_expert : args.rows_per_expert;
            const int64_t wrow = (x.shared ? 0 : static_cast<int64_t>(x.e) * rpe) +
                                 static_cast<int64_t>(x.p) * kWRows + row;
            const float* sc = x.shared ? args.s_scale : args.scale;
            const float* xsc = x.shared ? args.s_xscale : args.xscale;  // e4m3: token row scales
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(x.shared ? args.s_out : args.out);
            const int64_t ldo = x.shared ? args.s_ldo : args.ldo;
            __nv_bfloat16* gu = static_cast<__nv_bfloat16*>(x.shared ? args.s_gu_out : args.gu_out);
            const int64_t ld_gu = x.shared ? args.s_ld_gu : args.ld_gu;
            constexpr int TPC = FP8 ? 8 : 16;  // tokens per 16 accumulator columns
            const bool two = EPI == kEpiSwiGLU || x.p * kWRows + kWRows <= rpe;
            const float s0 = FP8 ? ld_dep(sc + wrow) : 1.0f;
            const float s1 = (FP8 && two) ? ld_dep(sc + wrow + 128) : 1.0f;
#pragma unroll 1
            for (int c0 = 0; c0 < n; c0 += 16) {
                uint32_t a0[16], a1[16];
                tmem_ld16(t0 + c0, a0);
                tmem_ld16(t0 + C::HALF + c0, a1);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < TPC; ++i) {
                    const int tt = (FP8 ? c0 / 2 : c0) + i;
                    if (tt < x.vm) {
                        float v0, v1;
                        if constexpr (FP8) {  // the hi and lo columns of the token
                            const float rs = ld_dep(xsc + x.m0 + tt);
                            v0 = (__uint_as_float(a0[2 * i]) + __uint_as_float(a0[2 * i + 1])) * rs;
                            v1 = (__uint_as_float(a1[2 * i]) + __uint_as_float(a1[2 * i + 1])) * rs;
                        } else {
                            v0 = __uint_as_float(a0[i]);
                            v1 = __uint_as_float(a1[i]);
                        }
                        if constexpr (EPI == kEpiSwiGLU) {
                            // gate half, up half of the 128 outputs p*128 + row
                            const float h = silu(v0 * s0) * (v1 * s1);
                            out[(x.m0 + tt) * ldo + static_cast<int64_t>(x.p) * 128 + row] =
                                __float2bfloat16_rn(h);
                            if (gu) {  // the gate/up values, packed order
                                __nv_bfloat16* gr = gu + (x.m0 + tt) * ld_gu +
                                                    static_cast<int64_t>(x.p) * kWRows + row;
                                gr[0] = __float2bfloat16_rn(v0 * s0);
                                gr[128] = __float2bfloat16_rn(v1 * s1);
                            }
                        } else {
                            const float gate = (!x.shared && args.row_gate)
                                                   ? ld_dep(args.row_gate + x.m0 + tt)
                                                   : 1.0f;
                            __nv_bfloat16* yr = out + (x.m0 + tt) * ldo +
                                                static_cast<int64_t>(x.p) * kWRows + row;
                            yr[0] = __float2bfloat16_rn(gate * (v0 * s0));
                            if (two) yr[128] = __float2bfloat16_rn(gate * (v1 * s1));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty + acc);
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
        if (timed_out) *abort_flag = 1;
    }

    if (timed_out && args.status) atomicOr(args.status, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

template <int EPI, bool FP8>
cudaError_t launch_sk(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tAs,
                      const CUtensorMap& tBs, const SkinnyArgs& args, int max_tiles,
                      cudaStream_t stream) {
    using C = SkCfg<FP8>;
    static bool attr_done[kMaxDevices] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_grouped_gemm_skinny<EPI, FP8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    int grid = num_sms();
    if (max_tiles < grid) grid = max_tiles;
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(k_grouped_gemm_skinny<EPI, FP8>, dim3(grid), dim3(192), C::SMEM, stream, tA,
                      tB, tAs, tBs, args);
}

}  // namespace

int skinny_tile_rows(bool fp8) { return fp8 ? SkCfg<true>::NMAX : SkCfg<false>::NMAX; }
int skinny_k_step(bool fp8) { return fp8 ? SkCfg<true>::KSTEP : SkCfg<false>::KSTEP; }

cudaError_t launch_grouped_gemm_skinny(int epi, bool fp8, const void* W, int64_t rowsW,
                                       const void* X, int64_t rowsX, int64_t K, const void* Ws,
                                       int64_t rowsWs, const void* Xs, int64_t rowsXs, int64_t Ks,
                                       const SkinnyArgs& args, int max_tiles, cudaStream_t stream) {
    CUtensorMap tA, tB, tAs, tBs;
    if (!args.num_blocks) {  // shared-expert tiles only: the routed maps are never used
        W = Ws;
        rowsW = rowsWs;
        X = Xs;
        rowsX = rowsXs;
        K = Ks;
    }
    // weights: {128-byte rows, 256}; token rows: {128-byte rows, 16}; e4m3
    // token operands are [2 * rows, K] (hi, lo row pairs)
    const int dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int eb = fp8 ? 1 : 2;
    const int bx = fp8 ? 128 : 64;
    const int64_t xr = fp8 ? 2 : 1;
    if (!make_tensor_map_2d(&tA, W, rowsW, K, eb, dt, bx, kWRows, 128) ||
        !make_tensor_map_2d(&tB, X, xr * rowsX, K, eb, dt, bx, 16, 128))
        return cudaErrorInvalidValue;
    if (args.s_rows > 0) {
        if (!make_tensor_map_2d(&tAs, Ws, rowsWs, Ks, eb, dt, bx, kWRows, 128) ||
            !make_tensor_map_2d(&tBs, Xs, xr * rowsXs, Ks, eb, dt, bx, 16, 128))
            return cudaErrorInvalidValue;
    } else {
        tAs = tA;
        tBs = tB;
    }
    if (epi == kEpiSwiGLU)
        return fp8 ? launch_sk<kEpiSwiGLU, true>(tA, tB, tAs, tBs, args, max_tiles, stream)
                   : launch_sk<kEpiSwiGLU, false>(tA, tB, tAs, tBs, args, max_tiles, stream);
    if (epi == kEpiGate)
        return fp8 ? launch_sk<kEpiGate, true>(tA, tB, tAs, tBs, args, max_tiles, stream)
                   : launch_sk<kEpiGate, false>(tA, tB, tAs, tBs, args, max_tiles, stream);
    return cudaErrorInvalidValue;
}

}  // namespace moe
