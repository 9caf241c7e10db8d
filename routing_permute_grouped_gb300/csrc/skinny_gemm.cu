// skinny_gemm.cu -- the grouped expert GEMMs for blocks with few token rows
// (decode-sized batches), with bf16 or e4m3 expert weights.
//
// With a handful of rows per expert the token rows cannot fill the MMA's
// M = 128, so the operands are swapped: a tile multiplies 256 rows of one
// expert's K-major weight matrix (two M = 128 halves) by the token rows of one
// block of the table, which become the MMA's N (valid rows rounded up to 16):
//     D^T[f, t] = sum_k W[f, k] X[t, k]
// and the epilogue writes D back into the row-major h / y.  The weights pass
// through the SM once per tile; at decode sizes every (expert, panel) is
// visited by one tile, so the kernel's time is the weight bytes over the HBM
// bandwidth ("Dropless and grouped GEMM", sec. 10: the small-M decode layout
// with valid rows per expert; the block table stays the work list).
//
// bf16 weights: S stages of [256 weight rows | <= 128 token rows] x 64 K,
// loaded by TMA with the 128-byte swizzle and read by the MMA from shared
// memory.
//
// e4m3 weights ("MoE & MLA operators", sec. 6.1: one byte per weight;
// "Dropless and grouped GEMM", sec. 12: the scale multiplies the product when
// one scale covers the whole contraction).  A kind::f16 MMA takes two operands
// of one type, so the panel is widened to f16, which is exact (every e4m3
// value is an f16 value), and the token rows arrive in f16 (exact copies of
// the bf16 values inside f16's range).  TMA stages R slots of [e4m3 panel
// (64-byte swizzle) | <= 64 token rows]; converter warps widen each weight row
// in registers and store it into one of four A slots in tensor memory with
// tcgen05.st; the MMA reads A from tensor memory and B from the staging slot.
// Keeping the widened panel out of shared memory leaves room for nine staging
// slots (144 KB of weights in flight per SM).  At decode sizes the e4m3 stream
// is then bound by the MMA issue rate rather than by HBM: each M = 128, N = 16,
// K = 16 MMA occupies the tensor pipe about as long as a 128-column one, and a
// 64-K step of a 256-row panel takes eight of them for 16 KB of weights.  The
// per-output-channel scale multiplies the fp32 accumulator in the epilogue,
// after the whole K sum.  Tiles hold at most 64 token rows; a block with more
// is split into chunks of 64, ordered chunk-major so that decode (one chunk)
// keeps a balanced round-robin.
//
// Tile list, built on the device from the block table: routed tile t is
// chunk t / (nb * n_panels) of panel (t % (nb * n_panels)) / nb of block
// t % nb, so neighbouring CTAs read the same weight panel for the blocks of
// one expert; the dense shared expert's tiles follow in the same launch.
//
// Warp roles, one CTA per SM:
//   warp 0        TMA producer: weight panels and token rows
//   warp 1        TMEM allocation; one lane issues the MMAs
//   warps 2..5    epilogue
//   warps 6..13   (e4m3 only) converters: warp w widens weight rows
//                 128 * ((w - 6) / 4) + 32 * (w % 4) + lane, the TMEM lanes
//                 it may write
// Every wait is bounded; on a timeout the CTA flags the status word, lets its
// copies and MMAs in flight finish and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kWRows = 256;                  // weight rows per tile (two M = 128 halves)
constexpr int kABytes = kWRows * 128;        // 256 rows x 64 K, 16-bit, swizzled
constexpr int kRawBytes = kWRows * 64;       // 256 rows x 64 K e4m3 codes
constexpr uint32_t kErrRange = 0x1u;         // expert id outside [0, E)
constexpr uint32_t kErrTimeout = 0x2u;
constexpr uint32_t kErrF16Range = 0x4u;      // an activation outside f16's range

template <bool FP8>
struct SkCfg {
    static constexpr int NMAX = FP8 ? 64 : 128;        // token rows per tile
    static constexpr int BBYTES = NMAX * 128;          // token rows x 64 K, 16-bit
    static constexpr int S = 4;                        // bf16: smem stages; e4m3: TMEM A slots
    static constexpr int R = FP8 ? 9 : 0;              // e4m3 staging slots
    static constexpr int STAGE = FP8 ? 0 : kABytes + BBYTES;
    static constexpr int RAW = FP8 ? kRawBytes + BBYTES : 0;
    static constexpr int THREADS = FP8 ? 448 : 192;
    // TMEM columns: two accumulator buffers of two halves, then (e4m3) the A
    // slots of 2 x 32 columns (64 f16 K-values per lane and half)
    static constexpr uint32_t ACC_STRIDE = 2 * NMAX;
    static constexpr uint32_t HALF = NMAX;
    static constexpr uint32_t A_TMEM = 4 * NMAX;
    static constexpr int BARS = 2 * S + 2 * R + 5;
    static constexpr int SMEM = 1024 + S * STAGE + R * RAW + BARS * 8 + 16;
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(!FP8 || A_TMEM + S * 64 <= 512, "tensor memory budget");
    static_assert(RAW % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
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

// bf16-rounded SwiGLU output stored as bf16, or (e4m3 path) as the f16 holding
// the same value; returns false when that value is outside f16's range.
template <bool FP8>
__device__ __forceinline__ bool store_h(void* out, int64_t idx, float v) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    if constexpr (FP8) {
        const float bv = __bfloat162float(b);
        static_cast<__half*>(out)[idx] = __float2half_rn(bv);
        return !(fabsf(bv) >= 65520.0f) || isinf(bv);  // finite bf16 past f16's largest
    } else {
        static_cast<__nv_bfloat16*>(out)[idx] = b;
        return true;
    }
}

// Sixteen e4m3 codes -> eight f16x2 words (element 2i in the low half).
__device__ __forceinline__ void widen16(const uint4& v, uint32_t* f) {
    f[0] = e4m3x2_to_f16x2(static_cast<uint16_t>(v.x));
    f[1] = e4m3x2_to_f16x2(static_cast<uint16_t>(v.x >> 16));
    f[2] = e4m3x2_to_f16x2(static_cast<uint16_t>(v.y));
    f[3] = e4m3x2_to_f16x2(static_cast<uint16_t>(v.y >> 16));
    f[4] = e4m3x2_to_f16x2(static_cast<uint16_t>(v.z));
    f[5] = e4m3x2_to_f16x2(static_cast<uint16_t>(v.z >> 16));
    f[6] = e4m3x2_to_f16x2(static_cast<uint16_t>(v.w));
    f[7] = e4m3x2_to_f16x2(static_cast<uint16_t>(v.w >> 16));
}

template <int EPI, bool FP8>
__global__ void __launch_bounds__(SkCfg<FP8>::THREADS, 1)
    k_grouped_gemm_skinny(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                          const __grid_constant__ CUtensorMap tAs, const __grid_constant__ CUtensorMap tBs,
                          const SkinnyArgs args) {
    using C = SkCfg<FP8>;
    constexpr int S = C::S;
    constexpr int R = C::R;
    constexpr int STAGE = C::STAGE;
    constexpr int RAW = C::RAW;
    constexpr int NMAX = C::NMAX;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sStage = smem;                  // bf16: S x [weights 32 KB | tokens]
    uint8_t* sRaw = smem + S * STAGE;        // e4m3: R x [e4m3 panel 16 KB | tokens]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRaw + R * RAW);
    uint64_t* full = bars;           // bf16: stage landed; e4m3: A slot written
    uint64_t* empty = full + S;      // stage / A slot consumed by the MMA
    uint64_t* rfull = empty + S;     // (e4m3) staging slot landed
    uint64_t* rempty = rfull + R;    // (e4m3) staging slot consumed by the MMA
    uint64_t* tfull = rempty + R;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_holder + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full + i, FP8 ? 8 : 1);  // e4m3: one arrival per converter warp
            mbar_init(empty + i, 1);
        }
        for (int i = 0; i < R; ++i) {
            mbar_init(rfull + i, 1);
            mbar_init(rempty + i, 1);
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
    if (warp == 1) tmem_alloc(tmem_holder, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_wait();  // the block table and the token rows are visible from here on

    int nb = args.num_blocks ? ld_dep(args.num_blocks) : 0;  // null: shared-expert tiles only
    nb = nb < 0 ? 0 : (nb > args.nb_cap ? args.nb_cap : nb);
    const int total = nb * args.n_panels * args.n_chunks +
                      (args.s_rows > 0 ? ((args.s_rows + NMAX - 1) / NMAX) * args.s_panels : 0);
    bool timed_out = false;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            constexpr int NSLOT = FP8 ? R : S;
            uint64_t* ring_full = FP8 ? rfull : full;
            uint64_t* ring_empty = FP8 ? rempty : empty;
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;  // slots with copies not yet seen landed
            for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
                const SkTile x = sk_tile<NMAX>(args, nb, t);
                if (!x.ok) continue;
                const CUtensorMap* ta = x.shared ? &tAs : &tA;
                const CUtensorMap* tb = x.shared ? &tBs : &tB;
                const int arow = (x.shared ? 0 : x.e * args.rows_per_expert) + x.p * kWRows;
                const int kbs = x.shared ? args.s_k_blocks : args.k_blocks;
                const int nbox = (x.vm + 15) >> 4;
                for (int kb = 0; kb < kbs; ++kb) {
                    if (!mbar_wait(ring_empty + s, ph ^ 1u, abort_flag)) {
                        timed_out = true;
                        break;
                    }
                    armed &= ~(1u << s);
                    uint8_t* slot = FP8 ? sRaw + s * RAW : sStage + s * STAGE;
                    uint8_t* btile = slot + (FP8 ? kRawBytes : kABytes);
                    mbar_arrive_expect_tx(ring_full + s, (FP8 ? kRawBytes : kABytes) + nbox * 2048);
                    tma_load_2d(slot, ta, kb * 64, arow, ring_full + s);
                    for (int j = 0; j < nbox; ++j)
                        tma_load_2d(btile + j * 2048, tb, kb * 64, x.m0 + 16 * j, ring_full + s);
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == NSLOT) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (timed_out || *abort_flag) {
                *abort_flag = 1;
                for (int i = 0; i < NSLOT; ++i)
                    if (armed & (1u << i)) {
                        volatile uint32_t never = 0;
                        (void)mbar_wait(ring_full + i, (armed_par >> i) & 1u, &never);
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer
            const uint32_t idesc0 = FP8 ? idesc_f16_f32(128, 8) : idesc_bf16_f32(128, 8);
            const uint32_t idesc_base = idesc0 & ~(0x3Fu << 17);
            int s = 0, r = 0;
            uint32_t ph = 0, rph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool issued = false;
            for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
                const SkTile x = sk_tile<NMAX>(args, nb, t);
                if (!x.ok) continue;
                const int kbs = x.shared ? args.s_k_blocks : args.k_blocks;
                const uint32_t n = static_cast<uint32_t>((x.vm + 15) & ~15);
                const uint32_t idesc = idesc_base | ((n >> 3) << 17);
                if (!mbar_wait(tempty + acc, aph ^ 1u, abort_flag)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc) * C::ACC_STRIDE;
                for (int kb = 0; kb < kbs; ++kb) {
                    bool ok = mbar_wait(full + s, ph, abort_flag);
                    // e4m3: the token rows sit in the staging slot, whose phase
                    // has completed already (the converters waited on it)
                    if (FP8 && ok) ok = mbar_wait(rfull + r, rph, abort_flag);
                    if (!ok) {
                        timed_out = true;
                        break;
                    }
                    tc_fence_after();
                    if constexpr (FP8) {
                        const uint32_t a_t = tmem_base + C::A_TMEM + static_cast<uint32_t>(s) * 64;
                        const uint32_t b_addr = smem_u32(sRaw + r * RAW + kRawBytes);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t bd = sdesc_sw128(b_addr + kk * 32);
                            const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
                            mma_f16_tmem_a(d0, a_t + kk * 8, bd, idesc, accum);
                            mma_f16_tmem_a(d0 + C::HALF, a_t + 32 + kk * 8, bd, idesc, accum);
                        }
                    } else {
                        const uint32_t a_addr = smem_u32(sStage + s * STAGE);
                        const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t bd = sdesc_sw128(b_addr + kk * 32);
                            const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
                            mma_bf16(d0, sdesc_sw128(a_addr + kk * 32), bd, idesc, accum);
                            mma_bf16(d0 + C::HALF, sdesc_sw128(a_addr + 16384 + kk * 32), bd, idesc,
                                     accum);
                        }
                    }
                    issued = true;
                    mma_commit(empty + s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if constexpr (FP8) {
                        mma_commit(rempty + r);
                        if (++r == R) {
                            r = 0;
                            rph ^= 1u;
                        }
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
    } else if (warp <= 5) {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t aph = 0;
        bool range_ok = true;
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
            const int n = (x.vm + 15) & ~15;
            const int rpe = x.shared ? args.s_rows_per_expert : args.rows_per_expert;
            const int64_t wrow = (x.shared ? 0 : static_cast<int64_t>(x.e) * rpe) +
                                 static_cast<int64_t>(x.p) * kWRows + row;
            const float* sc = x.shared ? args.s_scale : args.scale;
            void* out = x.shared ? args.s_out : args.out;
            const int64_t ldo = x.shared ? args.s_ldo : args.ldo;
            if constexpr (EPI == kEpiSwiGLU) {
                const float sg = FP8 ? ld_dep(sc + wrow) : 1.0f;
                const float su = FP8 ? ld_dep(sc + wrow + 128) : 1.0f;
                const int64_t col = static_cast<int64_t>(x.p) * 128 + row;
#pragma unroll 1
                for (int c0 = 0; c0 < n; c0 += 16) {
                    uint32_t g[16], u[16];
                    tmem_ld16(t0 + c0, g);
                    tmem_ld16(t0 + C::HALF + c0, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int tt = c0 + i;
                        if (tt < x.vm) {
                            const float gv = __uint_as_float(g[i]) * sg;
                            const float uv = __uint_as_float(u[i]) * su;
                            range_ok &= store_h<FP8>(out, (x.m0 + tt) * ldo + col, silu(gv) * uv);
                        }
                    }
                }
            } else {
                const bool two = x.p * kWRows + kWRows <= rpe;
                const float s0 = FP8 ? ld_dep(sc + wrow) : 1.0f;
                const float s1 = (FP8 && two) ? ld_dep(sc + wrow + 128) : 1.0f;
                const int64_t col = static_cast<int64_t>(x.p) * kWRows + row;
                __nv_bfloat16* y = static_cast<__nv_bfloat16*>(out);
#pragma unroll 1
                for (int c0 = 0; c0 < n; c0 += 16) {
                    uint32_t a0[16], a1[16];
                    tmem_ld16(t0 + c0, a0);
                    tmem_ld16(t0 + C::HALF + c0, a1);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int tt = c0 + i;
                        if (tt < x.vm) {
                            const float gate = (!x.shared && args.row_gate) ? ld_dep(args.row_gate + x.m0 + tt)
                                                                            : 1.0f;
                            __nv_bfloat16* yr = y + (x.m0 + tt) * ldo + col;
                            yr[0] = __float2bfloat16_rn(gate * (__uint_as_float(a0[i]) * s0));
                            if (two) yr[128] = __float2bfloat16_rn(gate * (__uint_as_float(a1[i]) * s1));
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
        if (!range_ok && args.status) atomicOr(args.status, kErrF16Range);
    } else if constexpr (FP8) {
        // ------------------------------------- e4m3 -> f16 into tensor memory
        const int half = (warp - 6) >> 2;           // weight rows [128 half, 128 half + 128)
        const int q = warp & 3;                     // TMEM lane quarter
        const int wr = half * 128 + q * 32 + lane;  // the weight row this thread widens
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + C::A_TMEM +
                                   static_cast<uint32_t>(half) * 32;
        const int sw = (wr >> 1) & 3;  // 64-byte swizzle: 16-byte chunk c of row wr sits at c ^ sw
        int s = 0, r = 0;
        uint32_t ph = 0, rph = 0;
        for (int t = blockIdx.x; t < total && !timed_out; t += gridDim.x) {
            const SkTile x = sk_tile<NMAX>(args, nb, t);
            if (!x.ok) continue;
            const int kbs = x.shared ? args.s_k_blocks : args.k_blocks;
            for (int kb = 0; kb < kbs; ++kb) {
                bool ok = true;
                if (lane == 0) ok = mbar_wait(empty + s, ph ^ 1u, abort_flag);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (ok && lane == 0) ok = mbar_wait(rfull + r, rph, abort_flag);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
                if (!ok) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint8_t* src = sRaw + r * RAW + wr * 64;
                uint32_t f[32];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    widen16(*reinterpret_cast<const uint4*>(src + ((c ^ sw) << 4)), f + 8 * c);
                tmem_st32(lane_base + static_cast<uint32_t>(s) * 64, f);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(full + s);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
                if (++r == R) {
                    r = 0;
                    rph ^= 1u;
                }
            }
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
    return launch_pdl(k_grouped_gemm_skinny<EPI, FP8>, dim3(grid), dim3(C::THREADS), C::SMEM, stream,
                      tA, tB, tAs, tBs, args);
}

}  // namespace

int skinny_tile_rows(bool fp8) { return fp8 ? SkCfg<true>::NMAX : SkCfg<false>::NMAX; }

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
    const int wdt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int wbytes = fp8 ? 1 : 2;
    const int wswz = fp8 ? 64 : 128;  // e4m3: 64-byte rows for the converters; bf16: as the MMA reads
    const int xdt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // weights: {64, 256} boxes; tokens: {64, 16}
    if (!make_tensor_map_2d(&tA, W, rowsW, K, wbytes, wdt, 64, kWRows, wswz) ||
        !make_tensor_map_2d(&tB, X, rowsX, K, 2, xdt, 64, 16, 128))
        return cudaErrorInvalidValue;
    if (args.s_rows > 0) {
        if (!make_tensor_map_2d(&tAs, Ws, rowsWs, Ks, wbytes, wdt, 64, kWRows, wswz) ||
            !make_tensor_map_2d(&tBs, Xs, rowsXs, Ks, 2, xdt, 64, 16, 128))
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
