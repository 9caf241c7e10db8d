// wgrad_gemm.cu -- weight gradients of the grouped expert GEMMs.
//
//   C[e][m][n] = sum over the rows r of expert e's segment of A[r][m] * B[r][n]
//
// A [rows, M] and B [rows, N] are the row-major activations of the padded
// layout as the backward produces them (pad rows hold zeros), and expert e
// owns rows [seg[e], seg[e+1]).  For the down projection A = p h, B = dz give
// dW2[e] = (p h)_e^T dz_e; for gate/up A = x_perm, B = dgu give the gradient
// of the packed gate/up weights.  ("Dropless and grouped GEMM", sec. 5: a
// tile reads exactly one expert's rows; here the reduction, not the output,
// runs over them.)
//
// The reduction runs along the rows, so both operands are MN-major: TMA
// copies boxes of 64 rows x 64 columns (128-byte swizzle, one 128-byte row
// per k) and the MMA reads them through MN-major shared-memory descriptors,
// no transposed copy.  Tiles are (expert, 256 rows of M over the CTA pair
// (cta_group::2), BN columns split over the pair), the K loop over the
// expert's segment in 64-row steps.  An expert without rows gets a zero
// gradient.  For the packed gate/up operand the epilogue splits every
// 256-column tile (128 gate, 128 up columns) straight into the two gradients;
// the router's gradient (N = the expert count rounded up to 128) is written
// as fp32 for its first E columns.  Warp roles: warp 0 TMA producer, warp 1
// TMEM allocation and MMA issue (even CTA), warps 2..9 epilogue (two per
// TMEM lane quarter, each half of the columns; bf16 stores of the fp32
// accumulators).  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "backward.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;  // rows of A per CTA
constexpr int kBK = 64;
constexpr uint32_t kTimeout = 0x2u;
// bits [15] and [16] of the instruction descriptor: A and B are MN-major
constexpr uint32_t kIdescMnMajorAB = (1u << 15) | (1u << 16);
// warps: TMA producer, MMA issuer, then two epilogue warps per TMEM lane
// quarter (each takes half of the tile's columns)
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
// output staging: epilogue warps x 2 buffers x (32 rows x 128 bytes)
constexpr int kOutStage = kEpiWarps * 2 * 4096;

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzle:
// rows of 128 bytes (64 bf16 along M or N) per k, 8-row groups 1024 bytes
// apart (stride byte offset), 64-column chunks `chunk_bytes` apart (leading
// byte offset).
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t chunk_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((chunk_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}
constexpr uint32_t kBadSegment = 0x4u;

struct WTile {
    int e, mt, nt, kb0, kb1;
    bool bad;  // the segment lies outside [0, rows): skipped as empty and flagged
};

__device__ __forceinline__ WTile wg_tile(const WgradArgs& a, int t) {
    WTile w;
    w.nt = t % a.n_tiles;
    const int r = t / a.n_tiles;
    w.mt = r % a.m_tiles;
    w.e = r / a.m_tiles;
    const int s0 = a.seg ? ld_dep(a.seg + w.e) : 0;
    int s1 = a.seg ? ld_dep(a.seg + w.e + 1) : a.dense_rows;
    w.bad = s0 < 0 || s1 < s0 || s1 > a.rows;
    if (a.seg && a.valid && !w.bad) {
        // rows past the valid ones are zero: stop at the last 64-row step
        // that holds data (at decode sizes that halves a tile's K loop)
        const int v = ld_dep(a.valid + w.e);
        w.bad = v < 0 || v > s1 - s0;
        s1 = s0 + v;
    }
    w.kb0 = w.bad ? 0 : s0 / kBK;
    w.kb1 = (!w.bad && s1 > s0) ? (s1 + kBK - 1) / kBK : w.kb0;
    return w;
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_wgrad_pair(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                 const __grid_constant__ CUtensorMap tO, const __grid_constant__ CUtensorMap tO2,
                 const WgradArgs args) {
    constexpr int BH = BN / 2;
    constexpr int BOX = 64 * kBK * 2;  // one TMA box: 64 columns x 64 rows, 8 KB
    constexpr int A_BYTES = kBM * kBK * 2;
    constexpr int B_BYTES = BH * kBK * 2;
    constexpr int STAGE = A_BYTES + B_BYTES;
    constexpr int S = (160 * 1024) / STAGE > 8 ? 8 : (160 * 1024) / STAGE;
    constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * A_BYTES;
    uint8_t* sOut = sB + S * B_BYTES;  // epilogue warps x 2 x 4 KB staging
    uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + kOutStage);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* tfull = bars + 2 * S;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_holder + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull + i, 1);
            mbar_init(tempty + i, 2 * kEpiWarps);  // one arrival per epilogue warp of both CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tA);
        tma_prefetch_desc(&tB);
    }
    // tensor memory is taken only once the kernels before this one have
    // finished (and released theirs)
    pdl_wait();
    if (warp == 1) tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers are initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int total = args.n_experts * args.m_tiles * args.n_tiles;
    const int cluster = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;
    bool timed_out = false;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;
            for (int t = cluster; t < total && !timed_out; t += nclusters) {
                const WTile w = wg_tile(args, t);
                const int acol = w.mt * 256 + kBM * static_cast<int>(rank);
                const int bcol = w.nt * BN + BH * static_cast<int>(rank);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(empty + s, ph ^ 1u, abort_flag)) {
                        timed_out = true;
                        break;
                    }
                    const uint32_t full_leader = mapa_shared(smem_u32(full + s), 0);
                    armed &= ~(1u << s);
                    if (leader) mbar_arrive_expect_tx(full + s, 2 * STAGE);
#pragma unroll
                    for (int i = 0; i < kBM / 64; ++i)
                        tma_load_2d_pair(sA + s * A_BYTES + i * BOX, &tA, acol + 64 * i, kb * kBK,
                                         full_leader);
#pragma unroll
                    for (int i = 0; i < BH / 64; ++i)
                        tma_load_2d_pair(sB + s * B_BYTES + i * BOX, &tB, bcol + 64 * i, kb * kBK,
                                         full_leader);
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if ((timed_out || *abort_flag) && leader) {
                *abort_flag = 1;
                for (int i = 0; i < S; ++i)
                    if (armed & (1u << i)) {
                        volatile uint32_t never = 0;
                        (void)mbar_wait(full + i, (armed_par >> i) & 1u, &never);
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ----------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, BN) | kIdescMnMajorAB;
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool issued = false;
            for (int t = cluster; t < total && !timed_out; t += nclusters) {
                const WTile w = wg_tile(args, t);
                if (w.kb1 <= w.kb0) continue;  // no rows: the epilogue writes zeros
                if (!mbar_wait(tempty + acc, aph ^ 1u, abort_flag)) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(full + s, ph, abort_flag)) {
                        timed_out = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + s * A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + s * B_BYTES);
                    // K = 16 rows per MMA: two 8-row groups of 1024 bytes
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16_pair(d_tmem, sdesc_sw128_mn(a_addr + kk * 2048, BOX),
                                      sdesc_sw128_mn(b_addr + kk * 2048, BOX), idesc,
                                      (kb != w.kb0 || kk != 0) ? 1u : 0u);
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
    } else if (warp >= 2) {
        // ---------------------------------------------------------- epilogue
        // Each warp owns 32 rows of M (its TMEM lane quarter) and half of the
        // tile's columns.  bf16 outputs leave through TMA bulk stores of
        // 32 x 64 boxes staged in shared memory (128-byte swizzle, two 4 KB
        // buffers per warp); the fp32 router gradient (a few columns) is
        // stored per thread.
        const int q = warp & 3;
        const int ew = warp - 2;            // epilogue warp 0 .. kEpiWarps - 1
        const int c_lo = (ew >> 2) * (BN / 2), c_hi = c_lo + BN / 2;
        int acc = 0;
        uint32_t aph = 0;
        int buf = 0;
        uint8_t* stage = sOut + ew * 2 * 4096;
        float* outf = static_cast<float*>(args.out);
        const bool split = args.out2 != nullptr;
        for (int t = cluster; t < total; t += nclusters) {
            const WTile w = wg_tile(args, t);
            const int mb = w.mt * 256 + kBM * static_cast<int>(rank) + q * 32;  // warp's first row
            const int m = mb + lane;
            const int col0 = w.nt * BN;
            const int64_t orow = static_cast<int64_t>(w.e) * args.M + mb;  // row in the output map
            const bool empty_tile = w.kb1 <= w.kb0;
            if (empty_tile && w.bad && ew == 0 && lane == 0 && args.status)
                atomicOr(args.status, kBadSegment);
            uint32_t taddr = 0;
            if (!empty_tile) {
                const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(tfull + acc, aph, abort_flag));
                if (!ok) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            }
            if (args.f32) {
                const int64_t row_off = (static_cast<int64_t>(w.e) * args.M + m) * args.n_valid;
#pragma unroll 1
                for (int c = c_lo; c < c_hi; c += 32) {
                    uint32_t v[32];
                    if (!empty_tile) {
                        tmem_ld32(taddr + c, v);
                        tmem_ld_wait();
                    }
                    if (m < args.M) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (col0 + c + i < args.n_valid)
                                outf[row_off + col0 + c + i] = empty_tile ? 0.0f : __uint_as_float(v[i]);
                    }
                }
            } else {
                // The warp's BN / 2 columns are read out of tensor memory and
                // packed to bf16 pairs first, and the accumulator is handed
                // back before any store of this tile is issued, with a
                // relaxed arrive: the reads are complete (wait::ld) and the
                // MMA side reads nothing this warp wrote.  A release arrive
                // waits for the warp's earlier stores to land, which at
                // decode sizes (a K loop of two steps per tile) paced the
                // whole kernel at 1.7x its store-bound time.
                uint32_t pk[BN / 4];
                if (!empty_tile) {
#pragma unroll
                    for (int c = 0; c < BN / 2; c += 64) {
                        uint32_t v[2][32];
                        tmem_ld32(taddr + c_lo + c, v[0]);
                        tmem_ld32(taddr + c_lo + c + 32, v[1]);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            pk[c / 2 + i] = pack_bf16x2(__uint_as_float(v[i >> 4][2 * (i & 15)]),
                                                        __uint_as_float(v[i >> 4][2 * (i & 15) + 1]));
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(tempty + acc), 0));
                    acc ^= 1;
                    if (acc == 0) aph ^= 1u;
                } else {
#pragma unroll
                    for (int i = 0; i < BN / 4; ++i) pk[i] = 0u;
                }
#pragma unroll
                for (int c = 0; c < BN / 2; c += 64) {
                    if (lane == 0) bulk_wait_read<1>();  // this buffer's previous store has read it
                    __syncwarp();
                    uint8_t* sb = stage + buf * 4096 + lane * 128;
#pragma unroll
                    for (int chunk = 0; chunk < 8; ++chunk) {  // 16-byte chunks of the 128-byte row
                        const uint32_t* u = pk + c / 2 + 4 * chunk;
                        *reinterpret_cast<uint4*>(sb + ((chunk ^ (lane & 7)) << 4)) =
                            make_uint4(u[0], u[1], u[2], u[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && mb < args.M) {
                        // split: tile columns [0, 128) are gate, [128, 256) up
                        const int cc = c_lo + c;
                        const bool up = split && cc >= 128;
                        const int x = split ? w.nt * 128 + (cc & 127) : col0 + cc;
                        tma_store_2d(up ? &tO2 : &tO, stage + buf * 4096, x, static_cast<int32_t>(orow));
                        bulk_commit();
                    }
                    buf ^= 1;
                }
                continue;  // the accumulator went back above
            }
            if (!empty_tile) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(tempty + acc), 0));
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_all();  // the stores have left shared memory and landed
        if (timed_out) *abort_flag = 1;
    }

    if (timed_out && args.status) atomicOr(args.status, kTimeout);
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <int BN>
cudaError_t launch_wg(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tO,
                      const CUtensorMap& tO2, const WgradArgs& args, cudaStream_t stream) {
    constexpr int STAGE = kBM * kBK * 2 + (BN / 2) * kBK * 2;
    constexpr int S = (160 * 1024) / STAGE > 8 ? 8 : (160 * 1024) / STAGE;
    constexpr int SMEM = 1024 + S * STAGE + kOutStage + 512;
    static_assert(SMEM <= 232448, "shared memory budget");
    static bool attr_done[kMaxDevices] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_wgrad_pair<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const int total = args.n_experts * args.m_tiles * args.n_tiles;
    int clusters = num_sms() / 2;
    if (total < clusters) clusters = total;
    if (clusters <= 0) return cudaSuccess;
    return launch_pdl(k_wgrad_pair<BN>, dim3(2 * clusters), dim3(kThreads), SMEM, stream, tA, tB, tO, tO2,
                      args);
}

}  // namespace

cudaError_t launch_wgrad(const void* A, int64_t M, const void* B, int64_t N, int64_t rows,
                         const int32_t* seg, int n_experts, int dense_rows, void* out, void* out2,
                         uint32_t* status, cudaStream_t stream, int f32_cols, const int32_t* valid) {
    if (N % 128 || M % 64 || M <= 0 || rows <= 0 || f32_cols < 0 || f32_cols > N)
        return cudaErrorInvalidValue;
    if (n_experts <= 0) return cudaErrorInvalidValue;
    const int bn = N % 256 == 0 ? 256 : 128;
    if (out2 && (bn != 256 || f32_cols)) return cudaErrorInvalidValue;  // split: 256-column tiles
    CUtensorMap tA, tB;
    if (!make_tensor_map_2d(&tA, A, rows, M, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64, kBK, 128) ||
        !make_tensor_map_2d(&tB, B, rows, N, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64, kBK, 128))
        return cudaErrorInvalidValue;
    WgradArgs a{};
    a.seg = seg;
    a.dense_rows = dense_rows;
    a.rows = static_cast<int32_t>(rows);
    a.n_experts = n_experts;
    a.M = static_cast<int32_t>(M);
    a.N = static_cast<int32_t>(N);
    a.m_tiles = static_cast<int32_t>((M + 255) / 256);
    a.n_tiles = static_cast<int32_t>(N / bn);
    a.out = out;
    a.out2 = out2;
    a.f32 = f32_cols > 0;
    a.n_valid = f32_cols > 0 ? f32_cols : static_cast<int32_t>(N);
    a.status = status;
    a.valid = valid;
    // bf16 outputs as [n_experts * M, ldo] maps stored in 64 x 32 boxes (the
    // fp32 output is stored per thread and needs none)
    CUtensorMap tO, tO2;
    const int64_t ldo = out2 ? N / 2 : N;
    const int64_t orows = static_cast<int64_t>(n_experts) * M;
    if (f32_cols) {
        tO = tA;
        tO2 = tA;
    } else if (!make_tensor_map_2d(&tO, out, orows, ldo, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64, 32,
                                   128) ||
               !make_tensor_map_2d(&tO2, out2 ? out2 : out, orows, ldo, 2,
                                   CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64, 32, 128)) {
        return cudaErrorInvalidValue;
    }
    return bn == 256 ? launch_wg<256>(tA, tB, tO, tO2, a, stream)
                     : launch_wg<128>(tA, tB, tO, tO2, a, stream);
}

}  // namespace moe
