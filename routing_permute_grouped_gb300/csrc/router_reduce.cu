// router_reduce.cu -- second half of the split-K router ("MoE & MLA
// operators", sec. 2.2: softmax + top-k after logits = x W_g).  When a
// batch has too few 128-token tiles to occupy the GPU (decode), the router
// GEMM splits K and writes fp32 partial logits per K slice; this kernel sums
// the slices in slice order, adds the bias and picks the experts.
//
// One warp per token; lane l holds experts l, l + 32, ... (E <= 256).
//   group limit: the group's score is its largest logit; the topk_groups
//                best groups stay eligible (ties to the lower group)
//   top-k:       k rounds of a warp argmax over the eligible experts, ties
//                to the lower index, output in descending logit order
//   gates:       softmax over the k chosen logits
#include <cuda_runtime.h>

#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

constexpr int kReduceWarps = 8;
constexpr int kMaxSlices = 16;

// (value, index) maximum over the warp; the lower index wins a tie
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}

__global__ void __launch_bounds__(kReduceWarps * 32)
    k_router_reduce(const float* __restrict__ partial, int S, int T, int E, int k, int n_groups,
                    int topk_groups, const float* __restrict__ bias, int32_t* __restrict__ topk_idx,
                    float* __restrict__ topk_w) {
    __shared__ float s_logit[kReduceWarps][256];
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kReduceWarps + warp;
    if (t >= T) return;
    float l[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        l[i] = -FLT_MAX;
        if (e < E) {
            // every slice's load issued before the first add (a loop of
            // dependent load-add steps would pay one memory latency per
            // slice); the sum still runs in slice order
            float p[kMaxSlices];
#pragma unroll
            for (int sl = 0; sl < kMaxSlices; ++sl)
                p[sl] = sl < S ? ld_dep(partial + (static_cast<int64_t>(sl) * T + t) * E + e) : 0.0f;
            float v = 0.0f;
#pragma unroll
            for (int sl = 0; sl < kMaxSlices; ++sl)
                if (sl < S) v += p[sl];
            if (bias) v += ld_dep(bias + e);
            l[i] = v;
            s_logit[warp][e] = v;
        }
    }
    __syncwarp();
    // eligibility: bit i of elig set when expert lane + 32 i may be chosen
    uint32_t elig = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (lane + 32 * i < E) elig |= 1u << i;
    if (n_groups > 0) {
        const int gsz = E / n_groups;
        float gs = -FLT_MAX;
        if (lane < n_groups)
            for (int e = lane * gsz; e < (lane + 1) * gsz; ++e) gs = fmaxf(gs, s_logit[warp][e]);
        uint32_t kept = 0;  // bit g set when group g is kept (same in every lane)
        float cand = lane < n_groups ? gs : -FLT_MAX;
        for (int r = 0; r < topk_groups; ++r) {
            float v = cand;
            int g = lane < n_groups ? lane : 1 << 30;
            warp_argmax(v, g);
            kept |= 1u << g;
            if (lane == g) cand = -FLT_MAX;
        }
        // a chosen group's candidate is retired by setting it to -FLT_MAX, so a
        // later round can only pick it again if every score is -FLT_MAX; the
        // logits here are finite, so that does not happen
        elig = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            if (e < E && ((kept >> (e / gsz)) & 1u)) elig |= 1u << i;
        }
    }
    float chosen_v[8];
    int chosen_e[8];
    for (int r = 0; r < k; ++r) {
        float v = -FLT_MAX;
        int e = 1 << 30;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if ((elig >> i) & 1u) {
                const int ei = lane + 32 * i;
                if (l[i] > v || (l[i] == v && ei < e)) {
                    v = l[i];
                    e = ei;
                }
            }
        }
        warp_argmax(v, e);
        chosen_v[r < 8 ? r : 7] = v;
        chosen_e[r < 8 ? r : 7] = e;
        if ((e & 31) == lane) elig &= ~(1u << (e >> 5));
    }
    if (lane == 0) {
        float sum = 0.0f;
        for (int r = 0; r < k; ++r) sum += expf(chosen_v[r] - chosen_v[0]);
        const float inv = 1.0f / sum;
        for (int r = 0; r < k; ++r) {
            topk_idx[static_cast<int64_t>(t) * k + r] = chosen_e[r];
            topk_w[static_cast<int64_t>(t) * k + r] = expf(chosen_v[r] - chosen_v[0]) * inv;
        }
    }
}

cudaError_t launch_router_reduce(const float* partial, int S, int T, int E, int k, int n_groups,
                                 int topk_groups, const float* bias, int32_t* topk_idx,
                                 float* topk_w, cudaStream_t stream) {
    if (E > 256 || k > 8 || n_groups > 32 || S < 1 || S > kMaxSlices) return cudaErrorInvalidValue;
    const int grid = (T + kReduceWarps - 1) / kReduceWarps;
    return launch_pdl(k_router_reduce, dim3(grid), dim3(kReduceWarps * 32), 0, stream, partial, S, T,
                      E, k, n_groups, topk_groups, bias, topk_idx, topk_w);
}

}  // namespace moe
