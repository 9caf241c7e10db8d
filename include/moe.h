/*
 * moe.h -- C ABI of the GB300 (sm_103a) dropless MoE layer forward pass.
 *
 * One layer = router (GEMM + softmax + top-k, optionally group-limited)
 *           -> per-expert counts / padded offsets / block table
 *           -> permute (token rows into expert order)
 *           -> grouped SwiGLU expert GEMMs (+ dense shared expert)
 *           -> combine (sum back into token order).
 * The decomposition is the four-stage one of "MoE & MLA operators" (TileLang
 * tutorial), sec. 2.1, with the shared expert of "Dropless and grouped GEMM",
 * sec. 1 added to the routed result.
 *
 * Conventions for every entry point
 *  - Pointers named as device buffers are device pointers owned by the caller;
 *    the library never allocates, frees or keeps them.  bf16 tensors are
 *    passed as `void *` (IEEE bfloat16, 2 bytes per element), row-major.
 *  - `stream` is a cudaStream_t passed as `void *` (NULL = legacy default
 *    stream).  Every call only enqueues work on it and returns; nothing
 *    synchronises with the host, and no launch size depends on routed data:
 *    kernels read the number of blocks from device memory and size their
 *    grids from static upper bounds.
 *  - Argument errors return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED before
 *    anything is enqueued.  A failed launch returns MOE_ERR_CUDA.  Data errors
 *    that only the device can see (an expert id outside [0, E), a wait that
 *    timed out) set a word in the workspace, readable with
 *    moe_get_device_status().
 *  - A call with T == 0 enqueues nothing and returns MOE_OK; its token-row
 *    buffers (x, out, dout, dx, the given routing) may be NULL.
 *  - Requirements on shapes: d % 128 == 0, d_e % 128 == 0,
 *    d_shared % 128 == 0 (or 0), 1 <= E <= 256, 1 <= k <= 8, pad_multiple 64
 *    or 128, group-limited routing needs E % n_groups == 0,
 *    n_groups <= 32 and topk_groups * (E / n_groups) >= k.  Routing also needs
 *    k <= E; pre-routed input (moe_build_offsets) may repeat an expert.
 *
 * Derived sizes (all host-computable from the config, never from the data):
 *    A      = T * k                       routed assignments
 *    R_max  = A + E * (pad_multiple - 1)  padded-row capacity
 *    NB_max = A / pad_multiple + E        block capacity
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad size, inconsistent config */
    MOE_ERR_UNSUPPORTED = 2,  /* valid MoE, but a shape this build does not run */
    MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime/driver call or launch failed */
    MOE_ERR_DEVICE_CHECK = 5  /* the device flagged bad data or a timed-out wait */
} moe_status_t;

/* Device error bits reported by moe_get_device_status(). */
#define MOE_DEVERR_EXPERT_RANGE 0x1u /* an expert id outside [0, E) was skipped */
#define MOE_DEVERR_TIMEOUT 0x2u      /* a bounded wait inside a kernel gave up */
#define MOE_DEVERR_SEGMENT 0x4u      /* backward: a segment offset outside the padded rows
                                      * was skipped */

typedef struct {
    int32_t T;            /* tokens */
    int32_t d;            /* model width */
    int32_t d_e;          /* routed expert width */
    int32_t E;            /* routed experts */
    int32_t k;            /* experts per token */
    int32_t n_groups;     /* expert groups for group-limited routing, 0 = none */
    int32_t topk_groups;  /* groups kept per token when n_groups > 0 */
    int32_t pad_multiple; /* segment padding multiple P: 64 or 128 */
    int32_t d_shared;     /* shared expert width, 0 = no shared expert */
} moe_config_t;

/* Packed weights as produced by the moe_pack_* calls (device pointers). */
typedef struct {
    const void *Wg_t;   /* router weight, K-major: bf16 [E, d] */
    const float *bias;  /* per-expert logit bias fp32 [E], or NULL */
    const void *W13;    /* routed gate/up weights: bf16 [E, 2*d_e, d] */
    const void *W2;     /* routed down weights, K-major: bf16 [E, d, d_e] */
    const void *Ws13;   /* shared gate/up: bf16 [2*d_shared, d], or NULL */
    const void *Ws2;    /* shared down, K-major: bf16 [d, d_shared], or NULL */
} moe_weights_t;

/* e4m3 expert weights as produced by moe_pack_experts_fp8 (device pointers):
 * the K-major layouts of moe_weights_t with one byte per weight, and one fp32
 * scale per weight row (output channel).  The router stays bf16. */
typedef struct {
    const void *Wg_t;    /* router weight, K-major: bf16 [E, d] */
    const float *bias;   /* per-expert logit bias fp32 [E], or NULL */
    const void *W13q;    /* routed gate/up codes: e4m3 [E, 2*d_e, d] */
    const float *s13;    /* their scales: fp32 [E, 2*d_e] */
    const void *W2q;     /* routed down codes, K-major: e4m3 [E, d, d_e] */
    const float *s2;     /* fp32 [E, d] */
    const void *Ws13q;   /* shared gate/up codes: e4m3 [2*d_shared, d], or NULL */
    const float *ss13;   /* fp32 [2*d_shared] */
    const void *Ws2q;    /* shared down codes: e4m3 [d, d_shared], or NULL */
    const float *ss2;    /* fp32 [d] */
} moe_weights_fp8_t;

/* Extra weight layouts the backward pass multiplies by (device pointers).
 * The data gradients run on the same K-major grouped GEMMs as the forward,
 * so they need the weights with the other dimension as K.  W2 and Ws2 are
 * the caller's own arrays; W13t/Ws13t come from moe_pack_experts_bwd (the
 * gate and up weights interleaved per 128 columns, the order of the packed
 * W13); WgP from moe_pack_router_bwd. */
typedef struct {
    const void *W13t;   /* bf16 [E, d, 2*d_e]: row i = (W1[e][i], W3[e][i]) interleaved */
    const void *W2;     /* bf16 [E, d_e, d]: the unpacked W2 */
    const void *WgP;    /* bf16 [d, Ep], Ep = E rounded up to 128, columns >= E zero;
                         * NULL for a pre-routed forward (no router to
                         * differentiate through) */
    const void *Ws13t;  /* bf16 [d, 2*d_shared] (d_shared > 0), else NULL */
    const void *Ws2;    /* bf16 [d_shared, d]: the unpacked Ws2 (d_shared > 0), else NULL */
} moe_weights_bwd_t;

/* Gradients written by moe_layer_bwd (device pointers, caller-owned, fully
 * overwritten when T > 0; nothing is accumulated into them). */
typedef struct {
    void *dx;        /* bf16 [T, d] */
    float *dgates;   /* fp32 [T, k]: gradient of the routing weights (the
                      * topk_w of the forward), or NULL to keep it internal */
    float *dWg;      /* fp32 [d, E] router weight gradient, or NULL (a frozen
                      * router: dx still gets the router's term) */
    float *dbias;    /* fp32 [E] logit-bias gradient, or NULL */
    void *dW1, *dW3; /* bf16 [E, d, d_e] */
    void *dW2;       /* bf16 [E, d_e, d] */
    void *dWs1, *dWs3; /* bf16 [d, d_shared] (d_shared > 0), else NULL */
    void *dWs2;      /* bf16 [d_shared, d] (d_shared > 0), else NULL */
} moe_grads_t;

/* Offsets (bytes) of every intermediate inside the moe_layer_fwd workspace,
 * so a caller can read them back.  All offsets are multiples of 1024. */
typedef struct {
    size_t total;
    size_t status;         /* uint32 device error word + build scratch */
    size_t topk_idx;       /* int32 [T, k] */
    size_t topk_w;         /* fp32 [T, k] */
    size_t counts;         /* int32 [E] */
    size_t padded_offsets; /* int32 [E + 1] */
    size_t block_metadata; /* int32 [NB_max, 3] */
    size_t num_blocks;     /* int32 [1] */
    size_t perm_row;       /* int32 [A] */
    size_t row_src;        /* int32 [R_max] */
    size_t row_gate;       /* fp32 [R_max] */
    size_t x_perm;         /* bf16 [R_max, d] */
    size_t h;              /* bf16 [R_max, d_e] */
    size_t y;              /* bf16 [R_max, d] */
    size_t hs;             /* bf16 [T, d_shared] */
    size_t ys;             /* bf16 [T, d] */
    size_t router_partial; /* fp32 [S, T, E] split-K router logits (S > 1 only) */
    /* e4m3-weight layer only (moe_workspace_layout_fp8; empty otherwise): */
    size_t xs8;            /* e4m3 pairs of the token rows [2T, d] (d_shared > 0) */
    size_t h8;             /* e4m3 pairs of h [2R_max, d_e], then of hs [2T, d_shared] */
    size_t row_scale;      /* fp32 row scales: x [R_max], h [R_max], xs [T], hs [T] */
    size_t w16;            /* e4m3 layer with T*k > 32*E: the expert codes widened to bf16
                            * (routed W13, W2, shared Ws13, Ws2), empty otherwise */
    size_t visit_ready;    /* int32 [NB_max] scratch for moe_grouped_gemm_swiglu_permute (per-visit
                            * counts of permuted rows in place); not used by the layer */
} moe_workspace_layout_t;

/* ---------------------------------------------------------------- sizes -- */

/* Validates cfg (same rules as every call).  Returns MOE_OK or an error. */
moe_status_t moe_check_config(const moe_config_t *cfg);

/* Bytes of the moe_layer_fwd workspace; 0 if cfg is invalid. */
size_t moe_workspace_size(const moe_config_t *cfg);

/* Fills *layout with the moe_layer_fwd workspace layout. */
moe_status_t moe_workspace_layout(const moe_config_t *cfg, moe_workspace_layout_t *layout);

/* The same for moe_layer_fwd_fp8, whose workspace adds the xs8, h8 and
 * row_scale regions (x_perm then holds the e4m3 pairs of the permuted rows,
 * [2R_max, d] bytes). */
size_t moe_workspace_size_fp8(const moe_config_t *cfg);
moe_status_t moe_workspace_layout_fp8(const moe_config_t *cfg, moe_workspace_layout_t *layout);

/* Bytes of the scratch that moe_build_offsets needs (status word + per-chunk
 * expert counts); 0 if cfg is invalid. */
size_t moe_offsets_workspace_size(const moe_config_t *cfg);

/* ------------------------------------------------------------- packing -- */

/* Router weight W_g [d, E] (the orientation of "MoE & MLA operators",
 * sec. 2.2: logits = x[T,d] @ W_g[d,E]) -> Wg_t [E, d] (K-major).  One-time
 * weight preparation, not part of the forward pass. */
moe_status_t moe_pack_router(int32_t d, int32_t E, const void *Wg, void *Wg_t, void *stream);

/* Expert weights W1 (gate), W3 (up) [E, d, de] and W2 (down) [E, de, d] ->
 * W13 [E, 2*de, d] and W2_t [E, d, de], both K-major.  Inside W13 the gate
 * and up rows are interleaved per 128 output columns: rows
 * [256 j, 256 j + 128) hold gate columns [128 j, 128 j + 128) and rows
 * [256 j + 128, 256 j + 256) the matching up columns, so that one 256-wide
 * GEMM tile produces both halves of 128 SwiGLU outputs.  Gate and up share one
 * read of the activations ("MoE & MLA operators", sec. 2.4(c); "Dropless and
 * grouped GEMM", sec. 4 step 7: gate and up concatenated).  E = 1 packs a
 * shared expert.  Requires de % 128 == 0, d % 128 == 0. */
moe_status_t moe_pack_experts(int32_t E, int32_t d, int32_t de, const void *W1, const void *W3,
                              const void *W2, void *W13, void *W2_t, void *stream);

/* The gate/up half of moe_pack_experts for one layer's config, in the form
 * the layer's scope names: W1 (gate) and W3 (up), bf16 [E, d, d_e] each,
 * row-major as the pages write x W -> W13_packed bf16 [E, 2*d_e, d], K-major,
 * gate and up rows interleaved per 128 output columns exactly as
 * moe_pack_experts writes them ("MoE & MLA operators", sec. 2.4(c): the dual
 * GEMM of gate and up over one read of the activations).  The config is
 * checked like every other entry point's (d % 128, d_e % 128, E <= 256);
 * only d, d_e and E are used.  The down projection needs its own K-major
 * copy, which moe_pack_experts writes (it also packs a shared expert with
 * E = 1), and the router weight is packed by moe_pack_router.
 *   W1, W3      bf16 [E, d, d_e]   device, read
 *   W13_packed  bf16 [E, 2*d_e, d] device, written */
moe_status_t moe_pack_weights(const moe_config_t *cfg, const void *W1, const void *W3,
                              void *W13_packed, void *stream);

/* The same packing into e4m3 codes with one fp32 scale per output channel
 * ("MoE & MLA operators", sec. 6.1: fp8 expert weights, one byte each;
 * "Dropless and grouped GEMM", sec. 12: a scale that covers the whole
 * contraction is applied after the matmul).  For output channel c of a
 * matrix: scale = amax_c / 448 (IEEE fp32 division; 1 for an all-zero
 * channel) and code = the e4m3 value nearest to fp32(w / scale), ties to even,
 * saturating at 448.  Codes go where moe_pack_experts puts the bf16 values
 * (W13q [E, 2*de, d], W2q [E, d, de]); scales follow the packed rows
 * (s13 [E, 2*de], s2 [E, d]).  E = 1 packs a shared expert. */
moe_status_t moe_pack_experts_fp8(int32_t E, int32_t d, int32_t de, const void *W1,
                                  const void *W3, const void *W2, void *W13q, float *s13,
                                  void *W2q, float *s2, void *stream);

/* ----------------------------------------------------------- the stages -- */

/* a1. Router ("MoE & MLA operators", sec. 2.2): logits = x Wg + bias,
 * optionally restricted to the topk_groups best expert groups (group score =
 * the group's largest logit), top-k by logit (ties to the lower index), gates
 * = softmax over the k chosen logits.
 *   x        bf16 [T, d]          device, read
 *   Wg_t     bf16 [E, d]          device, read (moe_pack_router)
 *   bias     fp32 [E] or NULL     device, read
 *   topk_idx int32 [T, k]         device, written, descending logit order
 *   topk_w   fp32 [T, k]          device, written
 * Tensor cores compute the GEMM (fp32 accumulate); top-k runs in the
 * epilogue, one token row per thread. */
moe_status_t moe_route(const moe_config_t *cfg, const void *x, const void *Wg_t,
                       const float *bias, int32_t *topk_idx, float *topk_w, void *stream);

/* a1 for small batches: the router GEMM with K split into S slices (S from
 * the config: enough slices that the 128-token tiles x slices cover the GPU,
 * at most 16), the partial logits summed in slice order, then the bias, the
 * same group-limited top-k and softmax as moe_route.  Returns the same
 * outputs as moe_route.  Two forms, chosen from the config:
 *  - up to 4 slices and E <= 64 (within the kernel's shared memory): the S
 *    CTAs of a 128-token tile form a thread-block cluster and the slices
 *    meet in the first CTA's shared memory, one launch, no scratch
 *    (moe_route_splitk_scratch_size is 0 and `partial` is ignored);
 *  - otherwise fp32 partial logits go to `partial` and a second kernel sums
 *    them.
 * When the batch already fills the GPU (S = 1) it runs moe_route's single
 * kernel; the scratch size is 0 then too.
 *   partial  fp32 [S, T, E] device scratch, partial_bytes >= the size above */
size_t moe_route_splitk_scratch_size(const moe_config_t *cfg);
moe_status_t moe_route_splitk(const moe_config_t *cfg, const void *x, const void *Wg_t,
                              const float *bias, int32_t *topk_idx, float *topk_w, float *partial,
                              size_t partial_bytes, void *stream);

/* a2. Counts, padded offsets and the block table ("MoE & MLA operators",
 * sec. 2.3: padded offsets with padding_M = 128 and
 * block_metadata[total_m_blocks, 3] = [expert, m_start, valid_m]; "Dropless
 * and grouped GEMM", sec. 3: each segment rounded up to a multiple of 128,
 * sec. 5: segments in ascending expert order, the tile count computed on the
 * device).  Padded size of a segment = ceil(count / P) * P.
 *   topk_idx       int32 [A]        device, read (A = T*k, a = t*k + j)
 *   topk_w         fp32 [A] or NULL device, read (NULL = weight 1)
 *   counts         int32 [E]        device, written
 *   padded_offsets int32 [E + 1]    device, written (exclusive prefix sum)
 *   block_metadata int32 [NB_max,3] device, written: rows [0, num_blocks)
 *                                   = [expert, first padded row, valid rows]
 *   num_blocks     int32 [1]        device, written
 *   perm_row       int32 [A]        device, written: padded row of assignment a
 *                                   (-1 if its expert id was out of range)
 *   row_src        int32 [R_max]    device, written: assignment of a padded
 *                                   row, -1 for pad rows
 *   row_gate       fp32 [R_max]     device, written: routing weight of a
 *                                   padded row, 0 for pad rows
 *   ws, ws_bytes   scratch >= moe_offsets_workspace_size(cfg), device
 * Rows of a segment keep ascending assignment order, so the result is
 * deterministic.  An expert id outside [0, E) is skipped and flagged with
 * MOE_DEVERR_EXPERT_RANGE in the status word at the start of ws. */
moe_status_t moe_build_offsets(const moe_config_t *cfg, const int32_t *topk_idx,
                               const float *topk_w, int32_t *counts, int32_t *padded_offsets,
                               int32_t *block_metadata, int32_t *num_blocks, int32_t *perm_row,
                               int32_t *row_src, float *row_gate, void *ws, size_t ws_bytes,
                               void *stream);

/* Allocation-free variant of moe_build_offsets (the pages have no
 * counterpart; this exists for callers of this library).  Some callers cannot
 * allocate device memory where they run this stage; some serving runtimes,
 * for one, only hand out memory from a pool reserved at start-up.
 * This call takes the same inputs and outputs as moe_build_offsets but no
 * scratch: its per-chunk counts live in a 64 KiB array in the library's own
 * device memory, which every GPU that loads the library holds until the
 * process exits.  It never calls cudaMalloc, cudaFree or any allocating
 * routine.
 *   status  uint32 [1] device word that collects MOE_DEVERR_EXPERT_RANGE, or
 *           NULL to leave bad expert ids unreported
 * Limits: ceil(T*k / 2048) * E * 4 <= 65536 bytes (T*k <= 131072 at E = 256);
 * larger configs return MOE_ERR_WORKSPACE before anything is enqueued.
 * The first call on a device looks up the array's device address with a
 * host-side query (with that device current); later calls reuse it.
 * The address is kept per device and per CUDA context: after the device's
 * context is torn down and made again (cudaDeviceReset), the next call looks
 * it up again and counts as a first call.
 * All calls share the one array and it keeps the last call's contents (none
 * of it needs to start at zero); calls whose work overlaps on the GPU (on
 * different streams, or from different threads) race on it and must be
 * ordered by the caller. */
moe_status_t moe_build_offsets_noalloc(const moe_config_t *cfg, const int32_t *topk_idx,
                                       const float *topk_w, int32_t *counts,
                                       int32_t *padded_offsets, int32_t *block_metadata,
                                       int32_t *num_blocks, int32_t *perm_row, int32_t *row_src,
                                       float *row_gate, uint32_t *status, void *stream);

/* a3. Permute ("MoE & MLA operators", sec. 2.3: a data-dependent gather of
 * token rows into expert order): x_perm[perm_row[t*k + j]] = x[t].  Each
 * token row is read once and written k times with 16-byte accesses; pad rows
 * of x_perm are not written.
 *   x        bf16 [T, d]      device, read
 *   perm_row int32 [A]        device, read (negative entries are skipped)
 *   x_perm   bf16 [R_max, d]  device, written */
moe_status_t moe_permute(const moe_config_t *cfg, const void *x, const int32_t *perm_row,
                         void *x_perm, void *stream);

/* a3 for the e4m3-weight path.  The 8-bit MMAs take 8-bit operands on both
 * sides, so every 16-bit activation row v enters as an e4m3 pair with a
 * power-of-two row scale: 2^sig is the largest power of two with
 * max|v| * 2^sig <= 448, hi = e4m3(v * 2^sig) and lo = e4m3(v * 2^sig - hi)
 * (nearest, ties to even).  hi + lo equals v * 2^sig for every element within
 * a factor 2^10 of the row's largest magnitude and differs by at most 2^-10
 * below that, so the products keep the 16-bit activations' accuracy.
 *   x         bf16 [T, d]           device, read
 *   perm_row  int32 [A]             device, read
 *   x8        e4m3 [2 R_max, d]     device, written: rows 2r (hi) and 2r+1 (lo)
 *                                   of padded row r = perm_row[t*k + j]
 *   x_scale   fp32 [R_max]          device, written: 2^-sig of padded row r
 *   xs8, xs_scale  e4m3 [2T, d], fp32 [T]: the same pairs per token for the
 *                  shared expert, or both NULL */
moe_status_t moe_permute_fp8(const moe_config_t *cfg, const void *x, const int32_t *perm_row,
                             void *x8, float *x_scale, void *xs8, float *xs_scale, void *stream);

/* a4 + a5. Grouped SwiGLU expert GEMMs over the block table ("MoE & MLA
 * operators", sec. 2.4; "Dropless and grouped GEMM", sec. 5: one tile reads
 * exactly one expert's weights, the tile list lives on the device):
 *   h[r] = bf16( silu(x_perm[r] W1[e]) * (x_perm[r] W3[e]) )
 *   y[r] = bf16( row_gate[r] * (h[r] W2[e]) )
 * for every valid row r of every block [e, m_start, valid_m].  tcgen05 MMAs
 * with fp32 accumulators in tensor memory, issued on CTA pairs
 * (cta_group::2: a 256-row tile whose B operand is split between the two
 * SMs), operands staged by TMA; SwiGLU is
 * fused into the first GEMM's epilogue and the routing weight into the
 * second's ("MoE & MLA operators", sec. 2.5: output * expert weight in the
 * GEMM epilogue).  Pad rows of h and y are not written.
 *   x_perm         bf16 [R_max, d]     device, read
 *   W13, W2_t      packed weights      device, read (moe_pack_experts)
 *   block_metadata int32 [NB_max, 3]   device, read
 *   num_blocks     int32 [1]           device, read (never copied to the host)
 *   padded_offsets int32 [E + 1]       device, read: segment starts, so that a
 *                                      CTA pair takes an expert's blocks two
 *                                      (P = 128) or four (P = 64) at a time
 *   row_gate       fp32 [R_max] or NULL (NULL = 1)
 *   h              bf16 [R_max, d_e]   device, written
 *   y              bf16 [R_max, d]     device, written
 *   status         uint32 [1] device error word, or NULL */
moe_status_t moe_grouped_gemm_swiglu(const moe_config_t *cfg, const void *x_perm, const void *W13,
                                     const void *W2_t, const int32_t *block_metadata,
                                     const int32_t *num_blocks, const int32_t *padded_offsets,
                                     const float *row_gate, void *h, void *y, uint32_t *status,
                                     void *stream);

/* a4 + a5 for blocks with few rows (decode): the same h and y as
 * moe_grouped_gemm_swiglu from a second kernel that swaps the operands.  A
 * tile multiplies 256 weight rows of one expert (two M = 128 tcgen05 MMAs)
 * by the block's valid token rows (the MMA's N, valid_m rounded up to 16), so
 * an expert with two rows costs its weight bytes, not a 128-row tile
 * ("Dropless and grouped GEMM", sec. 10: the decode layout, valid rows per
 * expert with the block table as work list).  Tiles are (panel, block) pairs;
 * padded_offsets is not needed.  Arguments as moe_grouped_gemm_swiglu. */
moe_status_t moe_grouped_gemm_swiglu_skinny(const moe_config_t *cfg, const void *x_perm,
                                            const void *W13, const void *W2_t,
                                            const int32_t *block_metadata,
                                            const int32_t *num_blocks, const float *row_gate,
                                            void *h, void *y, uint32_t *status, void *stream);

/* a4 + a5 with e4m3 expert weights (moe_pack_experts_fp8) on the kernel of
 * moe_grouped_gemm_swiglu_skinny with 8-bit MMAs (tcgen05 kind::f8f6f4,
 * K = 32): the weight codes and the token-row pairs of moe_permute_fp8 are
 * multiplied as they are; the epilogue adds the hi and lo columns of a token
 * and applies its row scale and the weights' per-output-channel scales:
 *   h[r] = bf16( silu(s13_g * x_scale[r] * (x8 W1q)) * (s13_u * x_scale[r] * (x8 W3q)) )
 * A split kernel then writes the e4m3 pairs of h (h8, h_scale), and GEMM2
 *   y[r] = bf16( row_gate[r] * s2 * h_scale[r] * (h8 W2q) ).
 *   x8, x_scale    moe_permute_fp8 outputs      device, read
 *   h              bf16 [R_max, d_e]            device, written
 *   h8, h_scale    e4m3 [2 R_max, d_e], fp32 [R_max]  device, written
 *   y              bf16 [R_max, d]              device, written
 * Other arguments as moe_grouped_gemm_swiglu_skinny. */
moe_status_t moe_grouped_gemm_swiglu_fp8(const moe_config_t *cfg, const void *x8,
                                         const float *x_scale, const void *W13q, const float *s13,
                                         const void *W2q, const float *s2,
                                         const int32_t *block_metadata, const int32_t *num_blocks,
                                         const float *row_gate, void *h, void *h8, float *h_scale,
                                         void *y, uint32_t *status, void *stream);

/* a3 + a4 + a5 in one pair of launches: the grouped GEMMs of
 * moe_grouped_gemm_swiglu, with the permute of moe_permute done inside GEMM1
 * ("MoE & MLA operators", sec. 2.3) by two extra warps of every CTA.  They
 * copy the token rows into x_perm in padded-row order (the order the visits
 * are loaded in), a whole row per warp, and count the rows of every 256-row
 * visit in visit_ready; the CTA pair's TMA producer loads a visit's
 * rows once its count is complete (acquire, then a generic-to-async proxy
 * fence).  The copy warps wait on nothing, so the loads always come.  x_perm
 * ends as moe_permute leaves it (pad rows untouched).  This call clears
 * visit_ready itself (cudaMemsetAsync on the stream).  Measured no faster
 * than moe_permute followed by moe_grouped_gemm_swiglu (the copies' bytes
 * cost the GEMM what the permute kernel costs alone); the layer does not use
 * it.
 *   x            bf16 [T, d]       device, read
 *   row_src      int32 [R_max]     device, read (moe_build_offsets)
 *   x_perm       bf16 [R_max, d]   device, written
 *   visit_ready  int32 [NB_max]    device scratch
 * Other arguments as moe_grouped_gemm_swiglu (the CTA-pair kernel). */
moe_status_t moe_grouped_gemm_swiglu_permute(const moe_config_t *cfg, const void *x,
                                             const int32_t *row_src, void *x_perm,
                                             int32_t *visit_ready, const void *W13,
                                             const void *W2_t, const int32_t *block_metadata,
                                             const int32_t *num_blocks,
                                             const int32_t *padded_offsets, const float *row_gate,
                                             void *h, void *y, uint32_t *status, void *stream);

/* a3 + a4 + a5 fused: the grouped GEMMs of moe_grouped_gemm_swiglu with the
 * permute folded into GEMM1's A load ("Dropless and grouped GEMM", sec. 4:
 * gather the token rows by index instead of materialising the k copies).
 * Padded row r of expert e's segment reads x[row_src[r] / k]; pad rows read
 * zeros.  No x_perm buffer is read or written.
 *   x       bf16 [T, d]     device, read
 *   row_src int32 [R_max]   device, read (moe_build_offsets)
 * Other arguments and outputs as moe_grouped_gemm_swiglu. */
moe_status_t moe_grouped_gemm_swiglu_gather(const moe_config_t *cfg, const void *x,
                                            const int32_t *row_src, const void *W13,
                                            const void *W2_t, const int32_t *block_metadata,
                                            const int32_t *num_blocks,
                                            const int32_t *padded_offsets, const float *row_gate,
                                            void *h, void *y, uint32_t *status, void *stream);

/* a6. Dense shared expert ("Dropless and grouped GEMM", sec. 1: it reads the
 * original token rows, with no permute and no group sizes):
 *   hs = bf16( silu(x Ws1) * (x Ws3) ),  ys = bf16( hs Ws2 )
 * on the same tcgen05 kernels with a dense tile list.
 *   x bf16 [T, d], Ws13/Ws2_t packed (moe_pack_experts with E = 1),
 *   hs bf16 [T, d_shared], ys bf16 [T, d]; status as above. */
moe_status_t moe_shared_expert(const moe_config_t *cfg, const void *x, const void *Ws13,
                               const void *Ws2_t, void *hs, void *ys, uint32_t *status,
                               void *stream);

/* a6 in two halves, with the layer's fusions.  moe_shared_expert_up is
 * the gate/up GEMM, hs = bf16( silu(x Ws1) * (x Ws3) ); with perm_row and
 * x_perm (both or neither) it also performs a3, the permute of
 * moe_permute, in its epilogue: that GEMM's tiles are long (K = d), so
 * after handing each accumulator back the epilogue warps copy the tile's
 * column slice of their token rows to the k permuted positions
 * ("MoE & MLA operators", sec. 2.3) while the next tile's MMAs run.
 * x_perm then holds exactly what moe_permute writes (pad rows untouched).
 *   x bf16 [T, d], Ws13 packed (moe_pack_experts with E = 1), hs bf16
 *   [T, d_shared] written, perm_row int32 [A], x_perm bf16 [R_max, d]
 *   written; all device.
 * moe_shared_expert_down is the down projection, ys = bf16( hs Ws2 ).
 *   hs bf16 [T, d_shared], Ws2_t packed, ys bf16 [T, d] written. */
moe_status_t moe_shared_expert_up(const moe_config_t *cfg, const void *x, const void *Ws13,
                                  void *hs, const int32_t *perm_row, void *x_perm,
                                  uint32_t *status, void *stream);
moe_status_t moe_shared_expert_down(const moe_config_t *cfg, const void *hs, const void *Ws2_t,
                                    void *ys, uint32_t *status, void *stream);

/* a6's down projection + a7 fused: the combine in the shared expert's GEMM2
 * epilogue.  That tile covers token rows in token order, so the thread that
 * owns output row t adds the token's k routed rows there ("MoE & MLA
 * operators", sec. 2.5: the down-projection epilogue sums back into token
 * order; sec. 6.4: a fixed order, no atomics):
 *   out[t] = bf16( sum_{j=0..k-1} y[perm_row[t*k + j]] + bf16(hs Ws2)[t] )
 * in fp32 in exactly that order, one rounding at the end: bit for bit
 * moe_shared_expert_down followed by moe_combine, without writing or
 * reading ys.  Slower than the two calls at the default workload (the
 * gathers of the k rows hold up the epilogue of GEMM2's short tiles); the
 * layer does not use it.
 *   hs bf16 [T, d_shared], Ws2_t packed, y bf16 [R_max, d], perm_row int32
 *   [A], out bf16 [T, d] written; all device. */
moe_status_t moe_shared_expert_down_combine(const moe_config_t *cfg, const void *hs,
                                            const void *Ws2_t, const void *y,
                                            const int32_t *perm_row, void *out, uint32_t *status,
                                            void *stream);

/* a6 with e4m3 weights (moe_pack_experts_fp8 with E = 1) on the kernel of
 * moe_grouped_gemm_swiglu_fp8 with a dense tile list (chunks of 64 token rows
 * times panels of 256 weight rows).
 *   xs8, xs_scale  e4m3 [2T, d], fp32 [T] (moe_permute_fp8)
 *   hs             bf16 [T, d_shared]; hs8, hs_scale  e4m3 [2T, d_shared], fp32 [T]
 *   ys             bf16 [T, d]; status as above.
 * The layer (moe_layer_fwd_fp8) puts these tiles into its routed launches
 * instead, where they fill SMs that this call alone would leave idle. */
moe_status_t moe_shared_expert_fp8(const moe_config_t *cfg, const void *xs8, const float *xs_scale,
                                   const void *Ws13q, const float *ss13, const void *Ws2q,
                                   const float *ss2, void *hs, void *hs8, float *hs_scale,
                                   void *ys, uint32_t *status, void *stream);

/* a7. Combine ("MoE & MLA operators", sec. 2.5 and 6.4: k-way sum back into
 * token order in a fixed order, with wide accumulation):
 *   out[t] = bf16( sum_{j=0..k-1} y[perm_row[t*k + j]] + shared_out[t] )
 * summed in fp32 in exactly that order, one rounding at the end.  Pad rows
 * are never read; a negative perm_row entry contributes nothing.
 *   y bf16 [R_max, d], perm_row int32 [A], shared_out bf16 [T, d] or NULL,
 *   out bf16 [T, d]; all device. */
moe_status_t moe_combine(const moe_config_t *cfg, const void *y, const int32_t *perm_row,
                         const void *shared_out, void *out, void *stream);

/* --------------------------------------------------------- whole layer -- */

/* The whole forward pass of one layer: a1 .. a7 enqueued on one stream,
 * no host synchronisation.  ws must hold moe_workspace_size(cfg) bytes
 * (layout in moe_workspace_layout); its intermediates stay readable after
 * the call.  Requires w->Wg_t; w->Ws13/Ws2 when cfg->d_shared > 0.
 *   x bf16 [T, d], out bf16 [T, d]; all device.
 * When the batch has too few 128-token tiles to fill the GPU (decode sizes),
 * the router GEMM splits K into up to 16 slices whose fp32 partial logits
 * (workspace region router_partial) a second kernel sums in slice order
 * before the top-k; otherwise it is the single kernel of moe_route.
 * When the mean rows per expert, T*k/E, is at most 32 the expert GEMMs run
 * on the kernel of moe_grouped_gemm_swiglu_skinny, with the shared expert's
 * tiles appended to the same two launches, after moe_permute; otherwise on
 * the CTA-pair kernel of moe_grouped_gemm_swiglu, with the shared expert
 * split around it: moe_shared_expert_up (with the permute in its epilogue)
 * before the routed GEMMs, moe_shared_expert_down after them (with no
 * shared expert: moe_permute before the routed GEMMs).  moe_combine ends
 * the layer. */
moe_status_t moe_layer_fwd(const moe_config_t *cfg, const moe_weights_t *w, const void *x,
                           void *out, void *ws, size_t ws_bytes, void *stream);

/* The same layer for pre-routed input: the router is skipped and the given
 * routing (topk_idx int32 [T, k], topk_w fp32 [T, k], device) is used as is;
 * an expert may repeat within a token.  ("Dropless and grouped GEMM", sec. 4:
 * the rows that reach a card arrive already routed.) */
moe_status_t moe_layer_fwd_prerouted(const moe_config_t *cfg, const moe_weights_t *w,
                                     const void *x, const int32_t *topk_idx, const float *topk_w,
                                     void *out, void *ws, size_t ws_bytes, void *stream);

/* dst[i] = src[idx[i]] for i < n: bf16 rows of d elements (d % 8 == 0);
 * with src_gate/dst_gate (both or neither), fp32 dst_gate[i] =
 * src_gate[idx[i]] too; idx[i] < 0 leaves row i (and its gate) as it is.
 * The local part of the expert-parallel exchange ("Dropless and grouped
 * GEMM", sec. 14): the row pieces a rank keeps move between its senders'
 * layout and its expert-major layout here, the others arrive from its
 * peers.  src, idx, dst device; ranges must not overlap. */
moe_status_t moe_gather_rows(const void *src, const int32_t *idx, void *dst, int64_t n,
                             int32_t d, const float *src_gate, float *dst_gate, void *stream);

/* The unpadded schedule ("Dropless and grouped GEMM", sec. 11: instead of
 * padding each segment to a block multiple, a row tile that an expert
 * boundary cuts is executed once for each expert whose rows it holds; the
 * waste becomes repeated tiles instead of zero rows, at most E - 1 of them).
 *
 * a2 without padding: counts, and group_offsets [E + 1] = the exclusive
 * prefix sum of the counts; the assignments of expert e take rows
 * [group_offsets[e], group_offsets[e + 1]) in ascending assignment order.
 * perm_row [A], row_src [A] (the unpadded layout has A rows; -1 for rows
 * left over by out-of-range expert ids), row_gate [A] as moe_build_offsets
 * writes them; no block table.  ws as for moe_build_offsets. */
moe_status_t moe_build_offsets_unpadded(const moe_config_t *cfg, const int32_t *topk_idx,
                                        const float *topk_w, int32_t *counts,
                                        int32_t *group_offsets, int32_t *perm_row,
                                        int32_t *row_src, float *row_gate, void *ws,
                                        size_t ws_bytes, void *stream);

/* a4 + a5 on the unpadded layout: x_perm, h, y have A = T*k rows (bf16
 * [A, d], [A, d_e], [A, d]); the CTA pairs visit, for every expert, the
 * 256-row windows of the rows that its rows touch, and store only the rows of
 * that expert, so a window cut by an expert boundary is computed twice, once
 * with each expert's weights.  Weights, gates and epilogues as
 * moe_grouped_gemm_swiglu.  moe_permute and moe_combine run on this layout
 * unchanged (with the perm_row of moe_build_offsets_unpadded). */
moe_status_t moe_grouped_gemm_swiglu_unpadded(const moe_config_t *cfg, const void *x_perm,
                                              const void *W13, const void *W2_t,
                                              const int32_t *group_offsets, const float *row_gate,
                                              void *h, void *y, uint32_t *status, void *stream);

/* The receiving side of the expert-parallel dispatch ("Dropless and grouped
 * GEMM", sec. 4 step 5: the dispatch lands rows already grouped by expert and
 * padded to the alignment, and hands the receiver its per-expert counts;
 * sec. 14: expert parallelism with all-to-all).  counts[s * E + e] rows of
 * sender s for local expert e (e.g. the result of the counts all-to-all).
 * Expert e's segment holds the senders' rows back to back in sender order,
 * padded like any segment to ceil(c_e / P) * P rows, c_e = sum over s of
 * counts[s, e]; its valid rows are therefore a prefix of the segment, as in
 * the single-GPU layout, and the grouped GEMM entry points run on it as they
 * are.  This is a2's arithmetic for a batch that arrives as counts instead
 * of expert ids.
 *   counts          int32 [n_src, E] device, read (negative entries count
 *                   as 0 and set MOE_DEVERR_SEGMENT)
 *   padded_offsets  int32 [E + 1]    device, written
 *   block_metadata  int32 [nb_cap,3] device, written: [expert, first row,
 *                   valid rows] of blocks [0, num_blocks)
 *   num_blocks      int32 [1]        device, written (at most nb_cap; blocks
 *                   past nb_cap set MOE_DEVERR_SEGMENT)
 *   piece_row       int32 [n_src, E] device, written: the first row of sender
 *                   s's rows for expert e, or NULL
 *   status          uint32 [1] device error word, or NULL
 * 1 <= E <= 256, P in {64, 128}.  One launch; nothing goes to the host. */
moe_status_t moe_build_blocks_from_counts(const int32_t *counts, int32_t n_src, int32_t E,
                                          int32_t P, int32_t *padded_offsets,
                                          int32_t *block_metadata, int32_t *num_blocks,
                                          int32_t nb_cap, int32_t *piece_row, uint32_t *status,
                                          void *stream);

/* Row pieces between two row-major bf16 [*, d] buffers (d % 8 == 0): for
 * piece i < n, rows [src_row[i], src_row[i] + rows[i]) of src go to rows
 * [dst_row[i], dst_row[i] + rows[i]) of dst, and with src_gate/dst_gate
 * (both or neither) their fp32 gates too.  The piece descriptors are device
 * arrays, so the pieces an expert-parallel rank keeps ("Dropless and grouped
 * GEMM", sec. 14) move between its own layout and its expert-major layout
 * with nothing built on the host.  max_rows >= every rows[i] (sizes the
 * grid; larger pieces are not copied beyond it); n <= 65535; pieces must not
 * overlap in dst, and src and dst ranges must not overlap. */
moe_status_t moe_copy_pieces(const void *src, void *dst, int32_t d, const int32_t *src_row,
                             const int32_t *dst_row, const int32_t *rows, int32_t n,
                             int32_t max_rows, const float *src_gate, float *dst_gate,
                             void *stream);

/* out[i] = the e4m3 code q[i] widened to bf16 (exact: every e4m3 value is a
 * bf16 value); n % 16 == 0.  The e4m3 layer's first step above the small-M
 * regime. */
moe_status_t moe_widen_e4m3(const void *q, void *out, int64_t n, void *stream);

/* moe_grouped_gemm_swiglu on e4m3 codes widened to bf16 (moe_widen_e4m3 of
 * W13q, W2q): every accumulator is multiplied by its weight row's scale
 * (s13 [E, 2*d_e], s2 [E, d] as moe_pack_experts_fp8 wrote them) before the
 * SwiGLU or gate epilogue. */
moe_status_t moe_grouped_gemm_swiglu_scaled(const moe_config_t *cfg, const void *x_perm,
                                            const void *W13, const float *s13, const void *W2_t,
                                            const float *s2, const int32_t *block_metadata,
                                            const int32_t *num_blocks,
                                            const int32_t *padded_offsets, const float *row_gate,
                                            void *h, void *y, uint32_t *status, void *stream);

/* moe_shared_expert on widened e4m3 codes with per-row scales ss13 [2*d_s],
 * ss2 [d]. */
moe_status_t moe_shared_expert_scaled(const moe_config_t *cfg, const void *x, const void *Ws13,
                                      const float *ss13, const void *Ws2_t, const float *ss2,
                                      void *hs, void *ys, uint32_t *status, void *stream);

/* The layer with e4m3 expert weights (routed and shared).  When T*k <=
 * 32*E (few rows per expert: the weight bytes set the pace): router and
 * offsets as moe_layer_fwd, then moe_permute_fp8, the e4m3 grouped GEMMs on
 * 8-bit MMAs with the shared expert's tiles in the same launches (GEMM1, the
 * split of h and hs into e4m3 pairs, GEMM2), and the combine.  Above that
 * (the tensor pipe sets the pace): the codes are widened to bf16 (exact)
 * into the workspace's w16 region, and the layer runs as moe_layer_fwd with
 * the accumulators of every GEMM scaled per output channel.  ws must hold
 * moe_workspace_size_fp8(cfg) bytes (layout: moe_workspace_layout_fp8).
 * Requires w->W13q/s13/W2q/s2, w->Wg_t, and the shared codes and scales when
 * d_shared > 0. */
moe_status_t moe_layer_fwd_fp8(const moe_config_t *cfg, const moe_weights_fp8_t *w,
                               const void *x, void *out, void *ws, size_t ws_bytes, void *stream);

/* moe_layer_fwd_fp8 for pre-routed input (as moe_layer_fwd_prerouted). */
moe_status_t moe_layer_fwd_fp8_prerouted(const moe_config_t *cfg, const moe_weights_fp8_t *w,
                                         const void *x, const int32_t *topk_idx,
                                         const float *topk_w, void *out, void *ws,
                                         size_t ws_bytes, void *stream);

/* ------------------------------------------------------------- backward -- */

/* Backward weight layout of the routed experts: W13t [E, d, 2*d_e] from the
 * caller's W1, W3 bf16 [E, d, d_e] (row i of expert e holds W1[e][i] and
 * W3[e][i] interleaved per 128 columns).  d, d_e multiples of 128.  Also
 * packs the shared expert (E = 1, W1 = Ws1, W3 = Ws3, d_e = d_shared). */
moe_status_t moe_pack_experts_bwd(int32_t E, int32_t d, int32_t de, const void *W1,
                                  const void *W3, void *W13t, void *stream);

/* WgP bf16 [d, Ep] from the caller's router weight Wg bf16 [d, E]; Ep = E
 * rounded up to 128, the extra columns zero. */
moe_status_t moe_pack_router_bwd(int32_t d, int32_t E, const void *Wg, void *WgP, void *stream);

/* Bytes of a gate/up save (moe_layer_fwd_save); 0 if cfg is invalid.  The
 * routed rows' values come first, bf16 [R_max, 2*d_e] in the padded order and
 * the packed gate/up column order (pad rows unwritten), then the shared
 * expert's, bf16 [T, 2*d_shared], at the next 1024-byte boundary. */
size_t moe_gate_up_save_size(const moe_config_t *cfg);

/* moe_layer_fwd (topk_idx NULL) or moe_layer_fwd_prerouted (topk_idx and
 * topk_w given) that also stores the gate/up GEMM's values x W13 (bf16, as
 * the backward's recomputation would produce them) into gu_save, which must
 * hold moe_gate_up_save_size(cfg) bytes.  Handing gu_save to moe_layer_bwd
 * spares it the recomputation: memory for time, against the pages' choice
 * of keeping only the routing ("Dropless and grouped GEMM", sec. 4). */
moe_status_t moe_layer_fwd_save(const moe_config_t *cfg, const moe_weights_t *w, const void *x,
                                const int32_t *topk_idx, const float *topk_w, void *out, void *ws,
                                size_t ws_bytes, void *gu_save, size_t gu_save_bytes,
                                void *stream);

/* Bytes of the moe_layer_bwd workspace; 0 if cfg is invalid. */
size_t moe_backward_workspace_size(const moe_config_t *cfg);

/* Backward of the bf16 layer.  The only state it keeps from the forward is
 * the routing: the sort indices and what derives from them ("Dropless and
 * grouped GEMM", sec. 4: the sort's residual is its indices, not the
 * T*k x d copy).  It reads the first moe_workspace_layout(cfg).x_perm bytes
 * of the forward workspace fwd_ws -- status word, topk_idx, topk_w, counts,
 * padded offsets, block table, perm_row, row_src, row_gate -- as the
 * moe_layer_fwd (or _prerouted) call that produced the output left them;
 * fwd_ws_bytes may be just that prefix, so a caller training several layers
 * can keep the prefix per layer and share the rest of the workspace.  The
 * permuted token rows are gathered again from x, the gate/up products
 * recomputed (or, when gu_saved is not NULL, read from the save that
 * moe_layer_fwd_save wrote, gu_saved_bytes >= moe_gate_up_save_size(cfg)),
 * and h recomputed from them.  dout bf16 [T, d] is the gradient of out.
 * Nothing in fwd_ws is written but the device error word.
 *
 * Gradients (the routing choice is a constant; the bf16 rounding of h passes
 * its gradient through):
 *   dW2[e]  = sum over e's rows a of h_a^T (p_a dout[t])
 *   dW1/dW3 from the SwiGLU backward of the recomputed g, u
 *   dgates  = <dout[t], h_a W2[e]> for each of the k choices
 *   dWg, dbias through the softmax over the k chosen logits (when
 *           wb->WgP is given: a routed forward)
 *   dx      = the k rows' dx_perm + the router's term (routed forward) + the
 *           shared expert's term (d_shared > 0)
 * Accumulation is fp32 inside each GEMM; GEMM outputs, dW1/dW3/dW2 and the
 * shared weight gradients are rounded to bf16 once, dWg and dbias stay fp32.
 *
 * T = 0 returns MOE_OK after the shape checks, without reading any pointer
 * or enqueuing anything (the gradient arrays are not touched).
 *
 * Returns MOE_ERR_INVALID_ARG on NULL buffers a gradient needs,
 * MOE_ERR_WORKSPACE when bws_bytes < moe_backward_workspace_size(cfg),
 * fwd_ws_bytes is shorter than the routing state or a gate/up save is too
 * short, the shape errors of
 * moe_check_config, MOE_ERR_CUDA on a launch error.  Asynchronous on
 * `stream`; bounded waits inside the kernels set MOE_DEVERR_TIMEOUT in the
 * forward workspace's device error word. */
moe_status_t moe_layer_bwd(const moe_config_t *cfg, const moe_weights_t *w,
                           const moe_weights_bwd_t *wb, const void *x, const void *dout,
                           const void *fwd_ws, size_t fwd_ws_bytes, const void *gu_saved,
                           size_t gu_saved_bytes, const moe_grads_t *grads, void *bws,
                           size_t bws_bytes, void *stream);

/* ---------------------------------------------------------- diagnostics -- */

/* Synchronises `stream`, reads the uint32 device error word at the start of
 * ws (a moe_layer_fwd workspace or a moe_build_offsets scratch) into
 * *bits (may be NULL) and clears it.  Returns MOE_OK if it was 0, else
 * MOE_ERR_DEVICE_CHECK.  This is the only call that synchronises; it is meant
 * for checking, not for the hot path. */
moe_status_t moe_get_device_status(void *ws, uint32_t *bits, void *stream);

/* Self-test of the failure path: one kernel waits on an mbarrier that nothing
 * signals, using the bounded wait of every kernel in this library, gives up
 * after limit_ns (0 < limit_ns <= 10 s) and sets MOE_DEVERR_TIMEOUT in the
 * device word *status.  The GPU context stays usable afterwards.  No fault,
 * trap or hang is involved. */
moe_status_t moe_selftest_wait_timeout(uint64_t limit_ns, uint32_t *status, void *stream);

/* Static description of a status code. */
const char *moe_status_string(moe_status_t s);

/* Thread-local text of the last error seen by this thread (argument or CUDA
 * error detail), "" if none. */
const char *moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
