// offsets.cu -- counts, padded offsets, block table and the permutation,
// built entirely on the device (no host round trip of the per-expert sizes:
// "Dropless and grouped GEMM", sec. 5 and 7).
//
// Up to three launches over fixed-size chunks of the A = T*k assignments:
//   k_chunk_hist     per-chunk expert histograms (shared-memory counters)
//   k_scan           one CTA: per-expert totals, ceil(c/P)*P sizes, exclusive
//                    prefix sums (padded_offsets, block starts), the block
//                    table [expert, m_start, valid_m] ("MoE & MLA operators",
//                    sec. 2.3), pad-row markers, and each chunk's first row
//                    inside every segment
//   k_chunk_scatter  stable ranks inside each chunk (warp match + ballot
//                    prefix, then a prefix over the warps of the CTA) ->
//                    perm_row, row_src, row_gate
// When the chunk histograms are small (chunks x experts <= 8192) the scan
// runs inside the scatter launch instead (k_scan_scatter): each CTA sums
// the histogram entries it needs, and CTA 0 writes the tables.
// Ranks depend only on the assignment order, never on atomic ordering, so the
// permutation is deterministic and rows of a segment stay in ascending
// assignment order.  Batches of at most 4096 assignments run all three steps
// in one CTA (one launch).
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

constexpr int kChunk = 2048;     // assignments per chunk
constexpr int kScatterThreads = 1024;  // two passes over a chunk
constexpr int kScanThreads = 1024;
constexpr int kMaxE = 256;
constexpr int kScanStaged = 8192;  // chunk counts k_scan stages in shared memory (32 KB)
constexpr uint32_t kDevErrExpert = 0x1u;
constexpr uint32_t kDevErrSegment = 0x4u;  // counts that do not fit the layout

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
    __shared__ int s_po[kMaxE];
    __shared__ int s_total[2];
    extern __shared__ int s_cc[];  // [n_chunks][E] when it fits (staged), else unused
    const bool staged = static_cast<int64_t>(n_chunks) * E <= kScanStaged;
    const int e = threadIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (staged) {
        // exclusive prefix over the chunks of every expert: the counts come in
        // with one coalesced pass, a warp scans an expert's column 32 chunks
        // at a time, the first ranks go back out with one coalesced pass
        const int n = n_chunks * E;
        for (int i = threadIdx.x; i < n; i += blockDim.x) s_cc[i] = chunk_counts[i];
        __syncthreads();
        for (int ex = warp; ex < E; ex += blockDim.x >> 5) {
            int running = 0;
            for (int base = 0; base < n_chunks; base += 32) {
                const int c = base + lane;
                const int v = c < n_chunks ? s_cc[c * E + ex] : 0;
                int x = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                    if (lane >= o) x += y;
                }
                if (c < n_chunks) s_cc[c * E + ex] = running + x - v;
                running += __shfl_sync(0xFFFFFFFFu, x, 31);
            }
            if (lane == 0) s_cnt[ex] = running;
        }
        __syncthreads();
    }
    int cnt = 0;
    if (e < E) {
        if (staged) {
            cnt = s_cnt[e];
        } else {
            // exclusive prefix over the chunks, in place: chunk c's first rank
            for (int c = 0; c < n_chunks; ++c) {
                const int v = chunk_counts[(int64_t)c * E + e];
                chunk_counts[(int64_t)c * E + e] = cnt;
                cnt += v;
            }
        }
        s_size[e] = ((cnt + P - 1) / P) * P;  // ceil(c/P)*P, 0 for an empty expert
        s_nblk[e] = (cnt + P - 1) / P;
    }
    __syncthreads();
    if (e < E) s_cnt[e] = cnt;
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
        s_po[e] = po;
        if (e == E - 1) padded_offsets[E] = s_total[0];
        if (!staged)
            for (int c = 0; c < n_chunks; ++c) chunk_counts[(int64_t)c * E + e] += po;
        if (block_metadata)  // null: the unpadded layout, which has no block table
            for (int i = 0; i < nblk; ++i) {
                block_metadata[3 * (b0 + i) + 0] = e;
                block_metadata[3 * (b0 + i) + 1] = po + i * P;
                block_metadata[3 * (b0 + i) + 2] = min(P, cnt - i * P);
            }
    }
    if (e == 0 && num_blocks) *num_blocks = s_total[1];
    if (staged) {
        __syncthreads();
        const int n = n_chunks * E;
        for (int i = threadIdx.x; i < n; i += blockDim.x) chunk_counts[i] = s_cc[i] + s_po[i % E];
    }
    fill_pad_rows(s_size, s_cnt, E, P, row_src, row_gate);
    for (int64_t r = s_total[0] + threadIdx.x; r < R_max; r += blockDim.x) {
        row_src[r] = -1;
        row_gate[r] = 0.0f;
    }
}

// Stable ranks of the assignments of this CTA's chunk (blockIdx.x) inside
// their segments, from running[e] = the chunk's first row in segment e:
// writes perm_row, row_src and row_gate.  wcnt must start at zero.
__device__ __forceinline__ void scatter_chunk(const int32_t* __restrict__ idx,
                                              const float* __restrict__ w, int64_t A, int E,
                                              int* running, int (*wcnt)[kMaxE],
                                              int32_t* __restrict__ perm_row,
                                              int32_t* __restrict__ row_src,
                                              float* __restrict__ row_gate) {
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
    scatter_chunk(idx, w, A, E, running, wcnt, perm_row, row_src, row_gate);
}

// The scan and the scatter in one launch, for up to kScanStaged chunk
// counts.  Every CTA derives what it needs from the chunk histograms itself
// (the expert totals, and its own chunk's first row in every segment), so
// no CTA waits for another.  CTA 0 also writes the tables k_scan writes:
// counts, padded offsets, the block table, the block count and the pad-row
// markers.  The results are those of k_scan + k_chunk_scatter.
__global__ void __launch_bounds__(kScatterThreads)
    k_scan_scatter(const int32_t* __restrict__ idx, const float* __restrict__ w, int64_t A,
                   int n_chunks, int E, int P, int64_t R_max,
                   const int32_t* __restrict__ chunk_counts, int32_t* __restrict__ counts,
                   int32_t* __restrict__ padded_offsets, int32_t* __restrict__ block_metadata,
                   int32_t* __restrict__ num_blocks, int32_t* __restrict__ perm_row,
                   int32_t* __restrict__ row_src, float* __restrict__ row_gate) {
    pdl_trigger();
    pdl_wait();
    constexpr int W = kScatterThreads / 32;
    __shared__ int s_cnt[kMaxE];
    __shared__ int s_pre[kMaxE];
    __shared__ int s_size[kMaxE];
    __shared__ int s_nblk[kMaxE];
    __shared__ int running[kMaxE];
    __shared__ int wcnt[W][kMaxE];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int me = blockIdx.x;
    // a warp per expert, its lanes over the chunks: the expert's total and
    // the counts of the chunks before this one
    for (int ex = warp; ex < E; ex += W) {
        int tot = 0, pre = 0;
        for (int c = lane; c < n_chunks; c += 32) {
            const int v = ld_dep(chunk_counts + (int64_t)c * E + ex);
            tot += v;
            if (c < me) pre += v;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
            pre += __shfl_xor_sync(0xFFFFFFFFu, pre, o);
        }
        if (lane == 0) {
            s_cnt[ex] = tot;
            s_pre[ex] = pre;
        }
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x)
#pragma unroll
        for (int i = 0; i < W; ++i) wcnt[i][e] = 0;
    __syncthreads();
    const int e = threadIdx.x;
    const int cnt = e < E ? s_cnt[e] : 0;
    const int size = ((cnt + P - 1) / P) * P;  // ceil(c/P)*P, 0 for an empty expert
    const int nblk = (cnt + P - 1) / P;
    if (e < E) {
        s_size[e] = size;
        s_nblk[e] = nblk;
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
    if (e < E) {
        const int po = s_size[e] - size;  // exclusive
        running[e] = po + s_pre[e];
        if (me == 0) {
            const int b0 = s_nblk[e] - nblk;  // exclusive
            counts[e] = cnt;
            padded_offsets[e] = po;
            if (e == E - 1) padded_offsets[E] = s_size[e];
            if (block_metadata)  // null: the unpadded layout, which has no block table
                for (int i = 0; i < nblk; ++i) {
                    block_metadata[3 * (b0 + i) + 0] = e;
                    block_metadata[3 * (b0 + i) + 1] = po + i * P;
                    block_metadata[3 * (b0 + i) + 2] = min(P, cnt - i * P);
                }
        }
    }
    if (me == 0 && e == 0 && num_blocks) *num_blocks = s_nblk[E - 1];
    __syncthreads();
    if (me == 0) {
        fill_pad_rows(s_size, s_cnt, E, P, row_src, row_gate);
        for (int64_t r = s_size[E - 1] + threadIdx.x; r < R_max; r += blockDim.x) {
            row_src[r] = -1;
            row_gate[r] = 0.0f;
        }
    }
    scatter_chunk(idx, w, A, E, running, wcnt, perm_row, row_src, row_gate);
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
        if (block_metadata)
            for (int i = 0; i < nblk; ++i) {
                block_metadata[3 * (b0 + i) + 0] = tid;
                block_metadata[3 * (b0 + i) + 1] = po + i * P;
                block_metadata[3 * (b0 + i) + 2] = min(P, cnt - i * P);
            }
    }
    if (tid == 0 && num_blocks) *num_blocks = s_total[1];
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

// The receiving side of an expert-parallel dispatch: from counts [n_src, E]
// (rows of sender s for local expert e) the padded offsets, the block table
// and piece_row [n_src, E] (where sender s's rows for e begin).  Expert e's
// segment holds the senders' rows back to back in sender order and is
// padded to a multiple of P, so its valid rows form a prefix, as in the
// single-GPU layout.  One CTA, a thread per expert.
__global__ void __launch_bounds__(kScanThreads)
    k_blocks_from_counts(const int32_t* __restrict__ counts, int n_src, int E, int P,
                         int32_t* __restrict__ padded_offsets, int32_t* __restrict__ block_metadata,
                         int32_t* __restrict__ num_blocks, int nb_cap,
                         int32_t* __restrict__ piece_row, uint32_t* status) {
    pdl_trigger();
    pdl_wait();
    __shared__ int s_size[kMaxE];
    __shared__ int s_nblk[kMaxE];
    __shared__ int s_total[2];
    const int e = threadIdx.x;
    int cnt = 0;
    bool bad = false;
    if (e < E) {
        for (int s = 0; s < n_src; ++s) {
            const int v = ld_dep(counts + static_cast<int64_t>(s) * E + e);
            if (v < 0) bad = true;
            cnt += v > 0 ? v : 0;
        }
        s_size[e] = ((cnt + P - 1) / P) * P;
        s_nblk[e] = (cnt + P - 1) / P;
    }
    __syncthreads();
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
        const int po = s_size[e] - size;
        const int b0 = s_nblk[e] - nblk;
        padded_offsets[e] = po;
        if (e == E - 1) padded_offsets[E] = s_total[0];
        if (piece_row) {
            int row = po;
            for (int s = 0; s < n_src; ++s) {
                piece_row[static_cast<int64_t>(s) * E + e] = row;
                const int v = ld_dep(counts + static_cast<int64_t>(s) * E + e);
                row += v > 0 ? v : 0;
            }
        }
        for (int i = 0; i < nblk; ++i) {
            if (b0 + i >= nb_cap) {
                bad = true;
                break;
            }
            block_metadata[3 * (b0 + i) + 0] = e;
            block_metadata[3 * (b0 + i) + 1] = po + i * P;
            block_metadata[3 * (b0 + i) + 2] = min(P, cnt - i * P);
        }
    }
    if (e == 0) *num_blocks = min(s_total[1], nb_cap);
    if (bad && status) atomicOr(status, kDevErrSegment);
}

cudaError_t launch_blocks_from_counts(const int32_t* counts, int n_src, int E, int P,
                                      int32_t* padded_offsets, int32_t* block_metadata,
                                      int32_t* num_blocks, int nb_cap, int32_t* piece_row,
                                      uint32_t* status, cudaStream_t stream) {
    return launch_pdl(k_blocks_from_counts, dim3(1), dim3(kScanThreads), 0, stream, counts, n_src, E,
                      P, padded_offsets, block_metadata, num_blocks, nb_cap, piece_row, status);
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
    if (n_chunks > 0 && static_cast<int64_t>(n_chunks) * E <= kScanStaged) {
        cudaError_t e = launch_pdl(k_scan_scatter, dim3(n_chunks), dim3(kScatterThreads), 0, stream,
                                   topk_idx, topk_w, A, n_chunks, E, P, R_max,
                                   static_cast<const int32_t*>(chunk_scratch), counts,
                                   padded_offsets, block_metadata, num_blocks, perm_row, row_src,
                                   row_gate);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const size_t scan_smem = static_cast<int64_t>(n_chunks) * E <= kScanStaged
                                 ? static_cast<size_t>(n_chunks) * E * 4 : 0;
    cudaError_t e = launch_pdl(k_scan, dim3(1), dim3(kScanThreads), scan_smem, stream, n_chunks, E, P,
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
