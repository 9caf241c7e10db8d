// wgrad_gemm.cu -- weight gradients of the grouped expert GEMMs.
//
//   C[e][m][n] = sum over the rows r of expert e's segment of A[m][r] * B[n][r]
//
// A [M, Rtot] and B [N, Rtot] are K-major copies of two activation matrices
// transposed so that the padded rows run along K (pad rows hold zeros), and
// expert e owns rows [seg[e], seg[e+1]) of the padded layout.  For the down
// projection A = h^T, B = dz^T give dW2[e] = h_e^T dz_e; for gate/up A = x^T,
// B = dgu^T give the gradient of the packed gate/up weights.  ("Dropless and
// grouped GEMM", sec. 5: a tile reads exactly one expert's rows; here the
// reduction, not the output, runs over them.)
//
// Tiles are (expert, 256-row block of M, BN-column block of N) on CTA pairs
// (cta_group::2, M = 256 split over the pair, B split along N), the K loop
// over the expert's rows in 64-row steps.  An expert without rows gets a zero
// gradient.  Warp roles as in the forward kernels: warp 0 TMA producer,
// warp 1 TMEM allocation and MMA issue (even CTA), warps 2..5 epilogue
// (bf16 stores of the fp32 accumulators).  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;  // rows of A per CTA
constexpr int kBK = 64;
constexpr uint32_t kTimeout = 0x2u;

struct WTile {
    int e, mt, nt, kb0, kb1;
};

__device__ __forceinline__ WTile wg_tile(const WgradArgs& a, int t) {
    WTile w;
    w.nt = t % a.n_tiles;
    const int r = t / a.n_tiles;
    w.mt = r % a.m_tiles;
    w.e = r / a.m_tiles;
    const int s0 = a.seg ? ld_dep(a.seg + w.e) : 0;
    const int s1 = a.seg ? ld_dep(a.seg + w.e + 1) : a.dense_rows;
    w.kb0 = s0 / kBK;
    w.kb1 = s1 > s0 ? (s1 + kBK - 1) / kBK : w.kb0;
    return w;
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    k_wgrad_pair(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                 const WgradArgs args) {
    constexpr int BH = BN / 2;
    constexpr int A_BYTES = kBM * kBK * 2;
    constexpr int B_BYTES = BH * kBK * 2;
    constexpr int STAGE = A_BYTES + B_BYTES;
    constexpr int S = (192 * 1024) / STAGE > 8 ? 8 : (192 * 1024) / STAGE;
    constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S * B_BYTES);
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
            mbar_init(tempty + i, 8);  // one arrival per epilogue warp of both CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tA);
        tma_prefetch_desc(&tB);
    }
    if (warp == 1) tmem_alloc_pair(tmem_holder, TMEM_COLS);
    pdl_wait();
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
                const int arow = w.mt * 256 + kBM * static_cast<int>(rank);
                const int brow = w.nt * BN + BH * static_cast<int>(rank);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(empty + s, ph ^ 1u, abort_flag)) {
                        timed_out = true;
                        break;
                    }
                    const uint32_t full_leader = mapa_shared(smem_u32(full + s), 0);
                    armed &= ~(1u << s);
                    if (leader) mbar_arrive_expect_tx(full + s, 2 * STAGE);
                    tma_load_2d_pair(sA + s * A_BYTES, &tA, kb * kBK, arow, full_leader);
                    tma_load_2d_pair(sB + s * B_BYTES, &tB, kb * kBK, brow, full_leader);
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
            constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, BN);
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
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16_pair(d_tmem, sdesc_sw128(a_addr + kk * 32), sdesc_sw128(b_addr + kk * 32),
                                      idesc, (kb != w.kb0 || kk != 0) ? 1u : 0u);
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
        const int q = warp & 3;
        int acc = 0;
        uint32_t aph = 0;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
        for (int t = cluster; t < total; t += nclusters) {
            const WTile w = wg_tile(args, t);
            const int m = w.mt * 256 + kBM * static_cast<int>(rank) + q * 32 + lane;
            __nv_bfloat16* dst = out + (static_cast<int64_t>(w.e) * args.M + m) * args.N +
                                 static_cast<int64_t>(w.nt) * BN;
            if (w.kb1 <= w.kb0) {  // an expert without rows: zero gradient
                if (m < args.M)
                    for (int c = 0; c < BN; c += 8) *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
                continue;
            }
            const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(tfull + acc, aph, abort_flag));
            if (!ok) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t v[32];
                tmem_ld32(taddr + c, v);
                tmem_ld_wait();
                if (m < args.M) {
                    uint32_t p[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        p[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        d4[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(tempty + acc), 0));
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
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
cudaError_t launch_wg(const CUtensorMap& tA, const CUtensorMap& tB, const WgradArgs& args,
                      cudaStream_t stream) {
    constexpr int STAGE = kBM * kBK * 2 + (BN / 2) * kBK * 2;
    constexpr int S = (192 * 1024) / STAGE > 8 ? 8 : (192 * 1024) / STAGE;
    constexpr int SMEM = 1024 + S * STAGE + 512;
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
    return launch_pdl(k_wgrad_pair<BN>, dim3(2 * clusters), dim3(192), SMEM, stream, tA, tB, args);
}

}  // namespace

cudaError_t launch_wgrad(const void* A, int64_t M, const void* B, int64_t N, int64_t ldk,
                         const int32_t* seg, int n_experts, int dense_rows, void* out,
                         uint32_t* status, cudaStream_t stream) {
    if (N % 128 || M <= 0 || ldk % 8) return cudaErrorInvalidValue;
    const int bn = N % 256 == 0 ? 256 : 128;
    CUtensorMap tA, tB;
    if (!make_tensor_map_2d(&tA, A, M, ldk, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kBK, kBM, 128) ||
        !make_tensor_map_2d(&tB, B, N, ldk, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kBK, bn / 2, 128))
        return cudaErrorInvalidValue;
    WgradArgs a{};
    a.seg = seg;
    a.dense_rows = dense_rows;
    a.n_experts = n_experts;
    a.M = static_cast<int32_t>(M);
    a.N = static_cast<int32_t>(N);
    a.m_tiles = static_cast<int32_t>((M + 255) / 256);
    a.n_tiles = static_cast<int32_t>(N / bn);
    a.out = out;
    a.status = status;
    return bn == 256 ? launch_wg<256>(tA, tB, a, stream) : launch_wg<128>(tA, tB, a, stream);
}

}  // namespace moe
