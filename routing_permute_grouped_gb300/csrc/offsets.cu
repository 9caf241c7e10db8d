// offsets.cu -- counts, padded offsets, block table and the permutation,
// built entirely on the device (no host round trip of the per-expert sizes:
// "Dropless and grouped GEMM", sec. 5 and 7).
//
// Three launches over fixed-size chunks of the A = T*k assignments:
//   k_chunk_hist     per-chunk expert histograms (shared-memory counters)
//   k_scan           one CTA: per-expert totals, ceil(c/P)*P sizes, exclusive
//                    prefix sums (padded_offsets, block starts), the block
//                    table [expert, m_start, valid_m] ("MoE & MLA operators",
//                    sec. 2.3), pad-row markers, and each chunk's first row
//                    inside every segment
//   k_chunk_scatter  stable ranks inside each chunk (warp match + ballot
//                    prefix, then a prefix over the warps of the CTA) ->
//                    perm_row, row_src, row_gate
// Ranks depend only on the assignment order, never on atomic ordering, so the
// permutation is deterministic and rows of a segment stay in ascending
// assignment order.  Batches of at most 4096 assignments run all three steps
// in one CTA (one launch).
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

constexpr int kChunk = 2048;     // assignments per chunk
constexpr int kScatterThreads = 256;
constexpr int kScanThreads = 1024;
constexpr int kMaxE = 256;
constexpr uint32_t kDevErrExpert = 0x1u;

int64_t offsets_num_chunks(int64_t A) { return (A + kChunk - 1) / kChunk; }

__global__ void __launch_bounds__(kScatterThreads)
    k_chunk_hist(const int32_t* __restrict__ idx, int64_t A, int E, int32_t* __restrict__ chunk_counts,
                 uint32_t* status) {
    pdl_trigger();
    pdl_wait();
    __shared__ int hist[kMaxE];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t a0 = (int64_t)blockIdx.x * kChunk;
    const int64_t a1 = min(A, a0 + kChunk);
    bool bad = false;
    for (int64_t a = a0 + threadIdx.x; a < a1; a += blockDim.x) {
        const int e = ld_dep(idx + a);
        if (e >= 0 && e < E)
            atomicAdd(&hist[e], 1);
        else
            bad = true;
    }
    if (bad && status) atomicOr(status, kDevErrExpert);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// The pad rows of every segment, [offset + count, offset + padded size):
// row_src = -1, row_gate = 0.  A warp per expert, its lanes over the rows,
// so that the stores are coalesced.  s_incl holds the inclusive scan of the
// padded sizes and cnt the counts (both in shared memory, final).
__device__ __forceinline__ void fill_pad_rows(const int* s_incl, const int* cnt, int E, int P,
                                              int32_t* __restrict__ row_src,
                                              float* __restrict__ row_gate) {
    const int lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    for (int e = threadIdx.x >> 5; e < E; e += nw) {
        const int c = cnt[e];
        const int size = ((c + P - 1) / P) * P;
        const int po = s_incl[e] - size;
        for (int r = po + c + lane; r < po + size; r += 32) {
            row_src[r] = -1;
            row_gate[r] = 0.0f;
        }
    }
}

__global__ void __launch_bounds__(kScanThreads)
    k_scan(int n_chunks, int E, int P, int64_t R_max, int32_t* __restrict__ chunk_counts,
           int32_t* __restrict__ counts, int32_t* __restrict__ padded_offsets,
           int32_t* __restrict__ block_metadata, int32_t* __restrict__ num_blocks,
           int32_t* __restrict__ row_src, float* __restrict__ row_gate) {
    pdl_trigger();
    pdl_wait();
    __shared__ int s_size[kMaxE];
    __shared__ int s_nblk[kMaxE];
    __shared__ int s_cnt[kMaxE];
    __shared__ int s_total[2];
    const int e = threadIdx.x;
    int cnt = 0;
    if (e < E) {
        // exclusive prefix over the chunks, in place: chunk c's first rank
        for (int c = 0; c < n_chunks; ++c) {
            const int v = chunk_counts[(int64_t)c * E + e];
            chunk_counts[(int64_t)c * E + e] = cnt;
            cnt += v;
        }
        s_size[e] = ((cnt + P - 1) / P) * P;  // ceil(c/P)*P, 0 for an empty expert
        s_nblk[e] = (cnt + P - 1) / P;
        s_cnt[e] = cnt;
    }
    __syncthreads();
    // inclusive Hillis-Steele scans of sizes and block counts over E <= 256
    for (int off = 1; off < E; off <<= 1) {
        int vs = 0, vb = 0;
        if (e < E && e >= off) {
            vs = s_size[e - off];
            vb = s_nblk[e - off];
        }
        __syncthreads();
        if (e < E && e >= off) {
            s_size[e] += vs;
            s_nblk[e] += vb;
        }
        __syncthreads();
    }
    if (e == E - 1) {
        s_total[0] = s_size[e];
        s_total[1] = s_nblk[e];
    }
    __syncthreads();
    if (e < E) {
        const int size = ((cnt + P - 1) / P) * P;
        const int nblk = (cnt + P - 1) / P;
        const int po = s_size[e] - size;   // exclusive
        const int b0 = s_nblk[e] - nblk;   // exclusive
        counts[e] = cnt;
        padded_offsets[e] = po;
        if (e == E - 1) padded_offsets[E] = s_total[0];
        for (int c = 0; c < n_chunks; ++c) chunk_counts[(int64_t)c * E + e] += po;
        for (int i = 0; i < nblk; ++i) {
            block_metadata[3 * (b0 + i) + 0] = e;
            block_metadata[3 * (b0 + i) + 1] = po + i * P;
            block_metadata[3 * (b0 + i) + 2] = min(P, cnt - i * P);
        }
    }
    if (e == 0) *num_blocks = s_total[1];
    fill_pad_rows(s_size, s_cnt, E, P, row_src, row_gate);
    for (int64_t r = s_total[0] + threadIdx.x; r < R_max; r += blockDim.x) {
        row_src[r] = -1;
        row_gate[r] = 0.0f;
    }
}

__global__ void __launch_bounds__(kScatterThreads)
    k_chunk_scatter(const int32_t* __restrict__ idx, const float* __restrict__ w, int64_t A, int E,
                    const int32_t* __restrict__ chunk_base, int32_t* __restrict__ perm_row,
                    int32_t* __restrict__ row_src, float* __restrict__ row_gate) {
    pdl_trigger();
    pdl_wait();
    constexpr int W = kScatterThreads / 32;
    __shared__ int running[kMaxE];
    __shared__ int wcnt[W][kMaxE];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        running[e] = chunk_base[(int64_t)blockIdx.x * E + e];
#pragma unroll
        for (int i = 0; i < W; ++i) wcnt[i][e] = 0;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int64_t a0 = (int64_t)blockIdx.x * kChunk;
    const int64_t a1 = min(A, a0 + kChunk);
    for (int64_t base = a0; base < a1; base += kScatterThreads) {
        const int64_t a = base + threadIdx.x;
        int e = -1;
        if (a < a1) {
            e = ld_dep(idx + a);
            if (e < 0 || e >= E) {
                perm_row[a] = -1;  // flagged by the histogram pass
                e = -1;
            }
        }
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
        const int rank = __popc(peers & lt_mask);
        const bool leader = rank == 0;
        if (e >= 0 && leader) wcnt[warp][e] = __popc(peers);
        __syncthreads();
        if (e >= 0) {
            int off = 0;
            for (int i = 0; i < warp; ++i) off += wcnt[i][e];
            const int r = running[e] + off + rank;
            perm_row[a] = r;
            row_src[r] = static_cast<int32_t>(a);
            row_gate[r] = w ? ld_dep(w + a) : 1.0f;
        }
        __syncthreads();
        if (e >= 0 && leader) {
            atomicAdd(&running[e], __popc(peers));  // integer sum: order-independent
            wcnt[warp][e] = 0;
        }
        __syncthreads();
    }
}

// Small batches (A <= kSmallA): the three steps above in one CTA of 1024
// threads, so a decode step pays one launch instead of three.
constexpr int kSmallA = 4096;
constexpr int kSmallThreads = 1024;

__global__ void __launch_bounds__(kSmallThreads)
    k_offsets_small(const int32_t* __restrict__ idx, const float* __restrict__ w, int A, int E, int P,
                    int64_t R_max, int32_t* __restrict__ counts, int32_t* __restrict__ padded_offsets,
                    int32_t* __restrict__ block_metadata, int32_t* __restrict__ num_blocks,
                    int32_t* __restrict__ perm_row, int32_t* __restrict__ row_src,
                    float* __restrict__ row_gate, uint32_t* status) {
    pdl_trigger();
    pdl_wait();
    constexpr int W = kSmallThreads / 32;
    __shared__ int hist[kMaxE];
    __shared__ int s_size[kMaxE];
    __shared__ int s_nblk[kMaxE];
    __shared__ int running[kMaxE];
    __shared__ int wcnt[W][kMaxE];
    __shared__ int s_total[2];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = tid; e < E; e += blockDim.x) {
        hist[e] = 0;
        for (int i = 0; i < W; ++i) wcnt[i][e] = 0;
    }
    __syncthreads();
    bool bad = false;
    for (int a = tid; a < A; a += blockDim.x) {
        const int e = ld_dep(idx + a);
        if (e >= 0 && e < E)
            atomicAdd(&hist[e], 1);
        else
            bad = true;
    }
    if (bad && status) atomicOr(status, kDevErrExpert);
    __syncthreads();
    int cnt = 0;
    if (tid < E) {
        cnt = hist[tid];
        s_size[tid] = ((cnt + P - 1) / P) * P;
        s_nblk[tid] = (cnt + P - 1) / P;
    }
    __syncthreads();
    for (int off = 1; off < E; off <<= 1) {
        int vs = 0, vb = 0;
        if (tid < E && tid >= off) {
            vs = s_size[tid - off];
            vb = s_nblk[tid - off];
        }
        __syncthreads();
        if (tid < E && tid >= off) {
            s_size[tid] += vs;
            s_nblk[tid] += vb;
        }
        __syncthreads();
    }
    if (tid == E - 1) {
        s_total[0] = s_size[tid];
        s_total[1] = s_nblk[tid];
    }
    __syncthreads();
    if (tid < E) {
        const int size = ((cnt + P - 1) / P) * P;
        const int nblk = (cnt + P - 1) / P;
        const int po = s_size[tid] - size;
        const int b0 = s_nblk[tid] - nblk;
        counts[tid] = cnt;
        padded_offsets[tid] = po;
        if (tid == E - 1) padded_offsets[E] = s_total[0];
        running[tid] = po;
        for (int i = 0; i < nblk; ++i) {
            block_metadata[3 * (b0 + i) + 0] = tid;
            block_metadata[3 * (b0 + i) + 1] = po + i * P;
            block_metadata[3 * (b0 + i) + 2] = min(P, cnt - i * P);
        }
    }
    if (tid == 0) *num_blocks = s_total[1];
    fill_pad_rows(s_size, hist, E, P, row_src, row_gate);
    for (int64_t r = s_total[0] + tid; r < R_max; r += blockDim.x) {
        row_src[r] = -1;
        row_gate[r] = 0.0f;
    }
    __syncthreads();
    // stable ranks, 1024 assignments at a time in assignment order
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = 0; base < A; base += kSmallThreads) {
        const int a = base + tid;
        int e = -1;
        if (a < A) {
            e = ld_dep(idx + a);
            if (e < 0 || e >= E) {
                perm_row[a] = -1;
                e = -1;
            }
        }
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
        const int rank = __popc(peers & lt_mask);
        const bool leader = rank == 0;
        if (e >= 0 && leader) wcnt[warp][e] = __popc(peers);
        __syncthreads();
        if (e >= 0) {
            int off = 0;
            for (int i = 0; i < warp; ++i) off += wcnt[i][e];
            const int r = running[e] + off + rank;
            perm_row[a] = r;
            row_src[r] = a;
            row_gate[r] = w ? ld_dep(w + a) : 1.0f;
        }
        __syncthreads();
        if (e >= 0 && leader) {
            atomicAdd(&running[e], __popc(peers));
            wcnt[warp][e] = 0;
        }
        __syncthreads();
    }
}

cudaError_t launch_offsets(const int32_t* topk_idx, const float* topk_w, int64_t A, int E, int P,
                           int64_t R_max, int32_t* counts, int32_t* padded_offsets,
                           int32_t* block_metadata, int32_t* num_blocks, int32_t* perm_row,
                           int32_t* row_src, float* row_gate, uint32_t* status,
                           int32_t* chunk_scratch, cudaStream_t stream) {
    if (A <= kSmallA) {
        return launch_pdl(k_offsets_small, dim3(1), dim3(kSmallThreads), 0, stream, topk_idx, topk_w,
                          static_cast<int>(A), E, P, R_max, counts, padded_offsets, block_metadata,
                          num_blocks, perm_row, row_src, row_gate, status);
    }
    const int n_chunks = static_cast<int>(offsets_num_chunks(A));
    if (n_chunks > 0) {
        cudaError_t e = launch_pdl(k_chunk_hist, dim3(n_chunks), dim3(kScatterThreads), 0, stream,
                                   topk_idx, A, E, chunk_scratch, status);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_pdl(k_scan, dim3(1), dim3(kScanThreads), 0, stream, n_chunks, E, P,
                               R_max, chunk_scratch, counts, padded_offsets, block_metadata,
                               num_blocks, row_src, row_gate);
    if (e != cudaSuccess) return e;
    if (n_chunks > 0) {
        e = launch_pdl(k_chunk_scatter, dim3(n_chunks), dim3(kScatterThreads), 0, stream, topk_idx,
                       topk_w, A, E, static_cast<const int32_t*>(chunk_scratch), perm_row, row_src,
                       row_gate);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace moe
