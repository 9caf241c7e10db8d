// internal.h -- declarations shared by the translation units of the library
// (launchers and the GEMM problem description).  Not part of the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <utility>

namespace moe {

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while the previous kernel on the stream finishes; every kernel of
// the library calls pdl_wait() before it reads anything an earlier kernel
// wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Device-side description of one grouped-GEMM launch.  The tile list is
// either the block table written by the offsets stage (block_metadata +
// num_blocks, both in device memory) or, when block_metadata is null, a
// dense list of ceil(dense_rows / 128) blocks of expert 0.
struct GemmArgs {
    const int32_t* block_metadata;  // [nb_cap, 3] or null
    const int32_t* num_blocks;      // [1] or null
    int32_t nb_cap;                 // capacity of the block table
    const int32_t* padded_offsets;  // [E + 1] segment starts (CTA-pair kernel)
    int32_t block_rows;             // rows per block of the table (P)
    int32_t n_experts;              // E (CTA-pair kernel)
    // CTA-pair kernel on the unpadded layout: padded_offsets holds the plain
    // group offsets, no block table; visits are the 256-row windows of each
    // expert's rows (a window cut by a boundary is visited once per expert)
    int32_t unpadded;
    // A rows gathered from token rows (permute fused into GEMM1's A load):
    // padded row r reads gather_x[row_src[r] / gather_k], pad rows read zeros
    const void* gather_x;
    const int32_t* row_src;
    int32_t gather_k;
    // split-K router (kEpiPartial): tile nb covers k-blocks
    // [nb * k_per_split, (nb + 1) * k_per_split); fp32 partial logits go to
    // partial[(nb * dense_rows + row) * E + e]
    int32_t k_per_split;
    float* partial;
    int32_t dense_rows;             // rows when block_metadata is null
    int32_t n_tiles;                // N / BN
    int32_t k_blocks;               // K / 64
    int32_t b_rows_per_expert;      // rows of the packed B operand per expert
    void* out;                      // bf16 output
    int64_t ldo;                    // output row stride (elements)
    int64_t out_rows;               // rows of the output tensor
    const float* row_gate;          // per padded row (gate epilogue), may be null
    // SwiGLU epilogue only: also store the gate/up values (bf16) of the tile,
    // in the packed interleaved column order, at gu_out[row * ld_gu + col]
    void* gu_out;
    int64_t ld_gu;
    // per-column scale of the accumulators (e4m3 weights widened to bf16:
    // the weights' per-output-channel scales), indexed like the B rows:
    // col_scale[e * b_rows_per_expert + packed row]; null = 1
    const float* col_scale;
    uint32_t* status;               // device error word, may be null
    // combine epilogue (the shared expert's GEMM2 over token rows): output row
    // t = sum over j of comb_y[comb_perm[t * comb_k + j]] (fp32, j ascending,
    // rows < 0 skipped) + the tile's own bf16 result, rounded once to bf16
    const void* comb_y;             // routed GEMM2 output [rows, comb_ldy] bf16
    const int32_t* comb_perm;       // [T, comb_k]
    int32_t comb_k;                 // 1..8
    int64_t comb_ldy;
    // permute in the SwiGLU epilogue (the shared expert's GEMM1 over token
    // rows): after its tile, the epilogue copies columns
    // [nb * nvec / n_tiles, (nb + 1) * nvec / n_tiles) (16-byte vectors) of
    // its token rows perm_x[t] to perm_out[perm_rows[t * perm_k + j]], j < perm_k
    const void* perm_x;             // token rows [T, perm_nvec * 8] bf16
    const int32_t* perm_rows;       // [T, perm_k]
    void* perm_out;                 // permuted rows (null: no permute)
    int32_t perm_k;
    int32_t perm_nvec;
    // permute by copy warps of the routed GEMM1 (CTA-pair kernel, padded
    // layout): padded row r of cp_out (GEMM1's A operand) is token row
    // cp_x[cp_row_src[r] / cp_k] (cp_nvec 16-byte vectors); every copied row
    // adds 1 to cp_ready[its visit], and the producer loads a visit's rows
    // once its count reaches the visit's valid rows.  cp_ready must start at
    // zero.
    const void* cp_x;
    const int32_t* cp_row_src;
    void* cp_out;
    int32_t* cp_ready;
    int32_t cp_k;
    int32_t cp_nvec;
    // router epilogue
    const float* bias;
    int32_t E, k, n_groups, topk_groups;
    int32_t* topk_idx;
    float* topk_w;
};

// The split-K router on clusters of `slices` CTAs (one per K slice of a
// 128-token tile; top-k fused after a distributed-shared-memory reduction).
// router_cluster_fits says whether a router of tile width bn with that many
// slices takes the kernel (2..4 slices, bn <= 64, shared-memory budget).
bool router_cluster_fits(int bn, int slices);
cudaError_t launch_router_cluster(int bn, const void* x, int64_t T, const void* Wg_t, int64_t E,
                                  int64_t K, const GemmArgs& args, int slices, cudaStream_t stream);

enum EpiKind {
    kEpiSwiGLU = 0,
    kEpiGate = 1,
    kEpiRouter = 2,
    kEpiSwiGLUGather = 3,
    kEpiPartial = 4,
    kEpiCombine = 5
};

// Launch the tcgen05 grouped GEMM: A [rowsA, K] bf16 (K-major), B
// [rowsB, K] bf16 (K-major), tile N = bn.  Returns a cudaError_t.
cudaError_t launch_grouped_gemm(int epi, int bn, const void* A, int64_t rowsA, const void* B,
                                int64_t rowsB, int64_t K, const GemmArgs& args, int max_tiles,
                                cudaStream_t stream);

cudaError_t launch_offsets(const int32_t* topk_idx, const float* topk_w, int64_t A, int E, int P,
                           int64_t R_max, int32_t* counts, int32_t* padded_offsets,
                           int32_t* block_metadata, int32_t* num_blocks, int32_t* perm_row,
                           int32_t* row_src, float* row_gate, uint32_t* status,
                           int32_t* chunk_scratch, cudaStream_t stream);
int64_t offsets_num_chunks(int64_t A);

cudaError_t launch_permute(const void* x, const int32_t* perm_row, void* x_perm, int T, int d,
                           int k, cudaStream_t stream);
// out[t] = sum_j y[perm_row[t*k + j]] (+ extra[t]) (+ extra2[t]), fp32, in
// that order.
cudaError_t launch_combine(const void* y, const int32_t* perm_row, const void* shared_out,
                           void* out, int T, int d, int k, cudaStream_t stream,
                           const void* extra2 = nullptr);

// out[c, r] = in[r, c] with the output row of column c remapped by `mode`:
// 0: row c; 1: gate rows of W13; 2: up rows of W13.  Batched over `batch`.
cudaError_t launch_pack_transpose(const void* in, void* out, int rows, int cols, int64_t in_bstride,
                                  int64_t out_bstride, int out_ld, int mode, int batch,
                                  cudaStream_t stream);

int num_sms();

// out[i] = the value of e4m3 code q[i] as bf16 (exact), n % 16 == 0.
cudaError_t launch_widen_e4m3(const void* q, void* out, int64_t n, cudaStream_t stream);

// Device-side description of one launch of the small-M (swapped-operand)
// grouped GEMM.  A tile multiplies 256 rows of one expert's K-major weight
// matrix (panel p of that expert) by the token rows of one block of the
// table (at most 128); tiles of the dense shared expert (chunks of 128 token
// rows) follow the routed tiles when s_rows > 0.
struct SkinnyArgs {
    const int32_t* block_metadata;  // [nb_cap, 3] [expert, m_start, valid_m]
    const int32_t* num_blocks;      // [1], or null for a launch of shared-expert tiles only
    int32_t nb_cap;                 // capacity of the block table
    int32_t n_experts;              // valid expert ids are [0, n_experts)
    int32_t n_panels;               // routed panels of 256 weight rows per block
    int32_t n_chunks;               // token-row chunks per block (e4m3 tiles hold <= 64 rows)
    int32_t rows_per_expert;        // weight rows per expert (2 d_e or d)
    int32_t k_blocks;               // routed K / 64
    void* out;                      // routed output [out_rows, ldo] (bf16, or f16 h)
    int64_t ldo;
    int64_t out_rows;
    const float* row_gate;          // routed gate per padded row (gate epilogue), may be null
    const float* scale;             // e4m3 weights: fp32 scale per weight row
    const float* xscale;            // e4m3: scale of each token row pair (per padded row)
    void* gu_out;                   // SwiGLU: gate/up values saved [out_rows, ld_gu], or null
    int64_t ld_gu;
    // shared expert (dense tiles after the routed ones)
    int32_t s_rows;                 // token rows (0 = no shared tiles)
    int32_t s_panels;
    int32_t s_rows_per_expert;      // weight rows of the shared matrix
    int32_t s_k_blocks;
    void* s_out;                    // [s_rows, s_ldo]
    int64_t s_ldo;
    const float* s_scale;
    const float* s_xscale;
    void* s_gu_out;                 // SwiGLU: the shared expert's gate/up values, or null
    int64_t s_ld_gu;
    uint32_t* status;               // device error word, may be null
};

// Token rows per tile of the small-M kernel (a block with more valid rows is
// split into n_chunks chunks of this many rows).
int skinny_tile_rows(bool fp8);
// K per pipeline stage of the small-M kernel (128 bytes of each row).
int skinny_k_step(bool fp8);

// Small-M grouped GEMM (epi = kEpiSwiGLU or kEpiGate).  W / Ws: weights
// [rows, K] K-major, bf16 or (fp8) e4m3 codes; X / Xs: token rows [rows, K]
// bf16, or (fp8) their e4m3 pairs [2 rows, K].  max_tiles bounds the tile
// count (grid size).
cudaError_t launch_grouped_gemm_skinny(int epi, bool fp8, const void* W, int64_t rowsW,
                                       const void* X, int64_t rowsX, int64_t K, const void* Ws,
                                       int64_t rowsWs, const void* Xs, int64_t rowsXs, int64_t Ks,
                                       const SkinnyArgs& args, int max_tiles, cudaStream_t stream);

// 2D tensor map of a row-major [rows, cols] matrix of elem_bytes-wide
// elements (dtype: a CUtensorMapDataType value) with a {box_cols, box_rows}
// box and the 128-byte, 64-byte or no (0) swizzle.  False if the driver
// refuses it.
bool make_tensor_map_2d(void* tmap, const void* ptr, int64_t rows, int64_t cols, int elem_bytes,
                        int dtype, int box_cols, int box_rows, int swizzle_bytes);

// e4m3 packing: per-output-channel scales of W [batch][rows][cols] (column c
// = output channel c), written to scale[b * scale_bstride + packed_row(c,
// mode)]; then the codes of the transposed matrix at out[packed_row(c,
// mode) * out_ld + r].
cudaError_t launch_pack_fp8(const void* in, uint8_t* out, float* scale, int rows, int cols,
                            int64_t in_bstride, int64_t out_bstride, int64_t scale_bstride,
                            int out_ld, int mode, int batch, cudaStream_t stream);

// Permute of the e4m3-weight path: token rows as e4m3 pairs (x8 [2 R, d]:
// rows 2r, 2r + 1) with per-row scales; xs8 [2 T, d] / xs_scale [T], if not
// null, receive the dense pairs for the shared expert.
cudaError_t launch_permute_fp8(const void* x, const int32_t* perm_row, uint8_t* x8, float* x_scale,
                               uint8_t* xs8, float* xs_scale, int T, int d, int k,
                               cudaStream_t stream);

// e4m3 pairs of bf16 rows between the expert GEMMs: the valid rows of the
// block table's blocks of h [R, K] (h8 [2 R, K], h_scale [R]) and, if hs is
// not null, the Ts dense rows of hs [Ts, Ks] (hs8, hs_scale).
cudaError_t launch_split_rows_e4m3(const void* h, const int32_t* block_metadata,
                                   const int32_t* num_blocks, int nb_cap, int K, uint8_t* h8,
                                   float* h_scale, const void* hs, int Ts, int Ks, uint8_t* hs8,
                                   float* hs_scale, cudaStream_t stream);

// Sums S fp32 partial-logit slices in slice order, adds the bias and does the
// (group-limited) top-k and softmax of each token.
cudaError_t launch_router_reduce(const float* partial, int S, int T, int E, int k, int n_groups,
                                 int topk_groups, const float* bias, int32_t* topk_idx,
                                 float* topk_w, cudaStream_t stream);

cudaError_t launch_blocks_from_counts(const int32_t* counts, int n_src, int E, int P,
                                      int32_t* padded_offsets, int32_t* block_metadata,
                                      int32_t* num_blocks, int nb_cap, int32_t* piece_row,
                                      uint32_t* status, cudaStream_t stream);
cudaError_t launch_copy_pieces(const void* src, void* dst, int d, const int32_t* src_row,
                               const int32_t* dst_row, const int32_t* rows, int n, int max_rows,
                               const float* sgate, float* dgate, cudaStream_t stream);
cudaError_t launch_wait_selftest(uint64_t limit_ns, uint32_t* status, cudaStream_t stream);

constexpr int kMaxDevices = 64;

// Records a printf-style message as this thread's last error (read by
// moe_last_error) and returns `status` unchanged.
int record_error(int status, const char* fmt, ...);

}  // namespace moe
