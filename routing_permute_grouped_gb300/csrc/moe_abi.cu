// moe_abi.cu -- the extern "C" entry points declared in include/moe.h:
// argument validation, the workspace layout, and the launch sequence of the
// layer on the caller's stream.  No entry point allocates memory or waits for
// the device, except moe_get_device_status().
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/moe.h"
#include "internal.h"
#include "backward.h"
#include "ep.h"

namespace moe {

static thread_local std::string g_last_error;

static moe_status_t fail(moe_status_t s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

int record_error(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

static moe_status_t cuda_fail(cudaError_t e, const char* where) {
    return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

int num_sms() {
    static int cached[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && cached[dev]) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    if (dev < 64) cached[dev] = n;
    return n;
}

static inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Sizes {
    int64_t A, R, NB, chunks;
};

static Sizes sizes_of(const moe_config_t& c) {
    Sizes s;
    s.A = static_cast<int64_t>(c.T) * c.k;
    s.R = s.A + static_cast<int64_t>(c.E) * (c.pad_multiple - 1);
    s.NB = s.A / c.pad_multiple + c.E;
    s.chunks = offsets_num_chunks(s.A);
    return s;
}

// Shape rules shared by every entry point.  `routed` adds the rule k <= E
// and the group-limit rules, which only the router needs.
static moe_status_t check_cfg(const moe_config_t* c, bool routed) {
    if (!c) return fail(MOE_ERR_INVALID_ARG, "config is NULL");
    if (c->T < 0 || c->d <= 0 || c->d_e <= 0 || c->E <= 0 || c->k <= 0)
        return fail(MOE_ERR_INVALID_ARG, "T must be >= 0 and d, d_e, E, k > 0");
    if (c->d % 128) return fail(MOE_ERR_UNSUPPORTED, "d = %d is not a multiple of 128", c->d);
    if (c->d_e % 128) return fail(MOE_ERR_UNSUPPORTED, "d_e = %d is not a multiple of 128", c->d_e);
    if (c->d_shared < 0 || c->d_shared % 128)
        return fail(MOE_ERR_UNSUPPORTED, "d_shared = %d must be 0 or a multiple of 128", c->d_shared);
    if (c->E > 256) return fail(MOE_ERR_UNSUPPORTED, "E = %d > 256", c->E);
    if (c->k > 8) return fail(MOE_ERR_UNSUPPORTED, "k = %d > 8", c->k);
    if (c->pad_multiple != 64 && c->pad_multiple != 128)
        return fail(MOE_ERR_UNSUPPORTED, "pad_multiple = %d must be 64 or 128", c->pad_multiple);
    const int64_t A = static_cast<int64_t>(c->T) * c->k;
    if (A + static_cast<int64_t>(c->E) * c->pad_multiple > (1ll << 30))
        return fail(MOE_ERR_UNSUPPORTED, "T*k too large for 32-bit row indices");
    if (routed) {
        if (c->k > c->E) return fail(MOE_ERR_INVALID_ARG, "k = %d > E = %d", c->k, c->E);
        if (c->n_groups < 0) return fail(MOE_ERR_INVALID_ARG, "n_groups < 0");
        if (c->n_groups > 0) {
            if (c->n_groups > 32 || c->E % c->n_groups)
                return fail(MOE_ERR_INVALID_ARG, "n_groups = %d must divide E and be <= 32",
                            c->n_groups);
            if (c->topk_groups <= 0 || c->topk_groups > c->n_groups)
                return fail(MOE_ERR_INVALID_ARG, "topk_groups = %d outside [1, n_groups]",
                            c->topk_groups);
            if (c->topk_groups * (c->E / c->n_groups) < c->k)
                return fail(MOE_ERR_INVALID_ARG, "topk_groups * (E / n_groups) < k");
        }
    }
    return MOE_OK;
}

// K slices of the layer's router GEMM: enough 128-token tiles x slices to
// cover the GPU (about 128 CTAs) when the batch is small, at most 16, and
// never an empty slice.  1 = the fused single-kernel router.
static int router_splits(const moe_config_t& c) {
    const int m_tiles = (c.T + 127) / 128;
    const int k_blocks = c.d / 64;
    int S = m_tiles > 0 ? 128 / m_tiles : 1;
    S = S < 1 ? 1 : (S > 16 ? 16 : S);
    if (S > k_blocks) S = k_blocks;
    const int per = (k_blocks + S - 1) / S;
    return (k_blocks + per - 1) / per;
}

static int router_bn(int E);

// The split-K router runs as one clustered kernel (slices reduced through
// distributed shared memory, no scratch) when its slices and tile width fit
// that kernel; otherwise as partial logits in a scratch + a reduce kernel.
static bool router_uses_cluster(const moe_config_t& c) {
    const int S = router_splits(c);
    return S > 1 && router_cluster_fits(router_bn(c.E), S);
}

// The small-M kernel serves the layer when the mean rows per expert is small
// enough that 256-row visits would mostly multiply padding.
static bool use_skinny(const moe_config_t& c) {
    return static_cast<int64_t>(c.T) * c.k <= 32ll * c.E;
}

// Elements of the routed and of the shared expert weights (gate/up + down).
static size_t routed_weight_elems(const moe_config_t& c) {
    return static_cast<size_t>(c.E) * 3 * c.d * c.d_e;
}
static size_t shared_weight_elems(const moe_config_t& c) {
    return static_cast<size_t>(3) * c.d * (c.d_shared ? c.d_shared : 0);
}

static moe_workspace_layout_t layout_of(const moe_config_t& c, bool fp8 = false) {
    const Sizes s = sizes_of(c);
    moe_workspace_layout_t L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 1024);
        return o;
    };
    L.status = take(256 + static_cast<size_t>(s.chunks) * c.E * 4);
    L.topk_idx = take(s.A * 4);
    L.topk_w = take(s.A * 4);
    L.counts = take(static_cast<size_t>(c.E) * 4);
    L.padded_offsets = take(static_cast<size_t>(c.E + 1) * 4);
    L.block_metadata = take(static_cast<size_t>(s.NB) * 12);
    L.num_blocks = take(4);
    L.perm_row = take(s.A * 4);
    L.row_src = take(s.R * 4);
    L.row_gate = take(s.R * 4);
    L.x_perm = take(static_cast<size_t>(s.R) * c.d * 2);
    L.h = take(static_cast<size_t>(s.R) * c.d_e * 2);
    L.y = take(static_cast<size_t>(s.R) * c.d * 2);
    L.hs = take(static_cast<size_t>(c.T) * (c.d_shared ? c.d_shared : 0) * 2);
    L.ys = take(static_cast<size_t>(c.T) * (c.d_shared ? c.d : 0) * 2);
    const int S = router_splits(c);
    L.router_partial =
        take(S > 1 && !router_uses_cluster(c) ? static_cast<size_t>(S) * c.T * c.E * 4 : 0);
    // e4m3-weight layer only: token-row pairs for the shared expert, the pairs
    // of h (routed then shared) and the row scales (x, h, shared x, shared h)
    const size_t ds = c.d_shared ? static_cast<size_t>(c.d_shared) : 0;
    L.xs8 = take(fp8 && ds ? static_cast<size_t>(c.T) * c.d * 2 : 0);
    L.h8 = take(fp8 ? (static_cast<size_t>(s.R) * c.d_e + static_cast<size_t>(c.T) * ds) * 2 : 0);
    L.row_scale = take(fp8 ? (2 * static_cast<size_t>(s.R) + 2 * static_cast<size_t>(c.T)) * 4 : 0);
    // e4m3 layer above the small-M regime: the codes widened to bf16 for the
    // CTA-pair GEMMs (routed W13, W2, then shared Ws13, Ws2)
    const bool wide = fp8 && !use_skinny(c);
    L.w16 = take(wide ? (routed_weight_elems(c) + shared_weight_elems(c)) * 2 : 0);
    L.visit_ready = take(static_cast<size_t>(s.NB) * 4);
    L.total = off;
    return L;
}

static size_t offsets_ws_bytes(const moe_config_t& c) {
    return 256 + static_cast<size_t>(sizes_of(c).chunks) * c.E * 4;
}

static int router_bn(int E) {
    if (E <= 16) return 16;
    if (E <= 32) return 32;
    if (E <= 64) return 64;
    if (E <= 128) return 128;
    return 256;
}

// ------------------------------------------------------------- stages --

static moe_status_t do_route(const moe_config_t& c, const void* x, const void* Wg_t,
                             const float* bias, int32_t* topk_idx, float* topk_w,
                             cudaStream_t st) {
    GemmArgs a{};
    a.dense_rows = c.T;
    a.n_tiles = 1;
    a.k_blocks = c.d / 64;
    a.b_rows_per_expert = 0;
    a.bias = bias;
    a.E = c.E;
    a.k = c.k;
    a.n_groups = c.n_groups;
    a.topk_groups = c.topk_groups;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    const int tiles = (c.T + 127) / 128;
    cudaError_t e = launch_grouped_gemm(kEpiRouter, router_bn(c.E), x, c.T, Wg_t, c.E, c.d, a,
                                        tiles, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "router GEMM");
}

// The layer's router: fused (top-k in the GEMM epilogue) when the batch
// fills the GPU, otherwise split-K partial logits + a reduce/top-k kernel.
static moe_status_t do_route_layer(const moe_config_t& c, const void* x, const void* Wg_t,
                                   const float* bias, int32_t* topk_idx, float* topk_w,
                                   float* partial, cudaStream_t st, uint32_t* status = nullptr) {
    const int S = router_splits(c);
    if (S <= 1) return do_route(c, x, Wg_t, bias, topk_idx, topk_w, st);
    GemmArgs a{};
    a.dense_rows = c.T;
    a.n_tiles = S;
    a.k_blocks = c.d / 64;
    a.k_per_split = (a.k_blocks + S - 1) / S;
    a.E = c.E;
    if (router_uses_cluster(c)) {
        a.bias = bias;
        a.k = c.k;
        a.n_groups = c.n_groups;
        a.topk_groups = c.topk_groups;
        a.topk_idx = topk_idx;
        a.topk_w = topk_w;
        a.status = status;
        cudaError_t e = launch_router_cluster(router_bn(c.E), x, c.T, Wg_t, c.E, c.d, a, S, st);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e, "router GEMM (split K over a cluster)");
    }
    a.partial = partial;
    const int tiles = ((c.T + 127) / 128) * S;
    cudaError_t e = launch_grouped_gemm(kEpiPartial, router_bn(c.E), x, c.T, Wg_t, c.E, c.d, a,
                                        tiles, st);
    if (e != cudaSuccess) return cuda_fail(e, "router GEMM (split K)");
    e = launch_router_reduce(partial, S, c.T, c.E, c.k, c.n_groups, c.topk_groups, bias, topk_idx,
                             topk_w, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "router reduce");
}

static moe_status_t do_offsets(const moe_config_t& c, const int32_t* topk_idx, const float* topk_w,
                               int32_t* counts, int32_t* po, int32_t* meta, int32_t* nb,
                               int32_t* perm_row, int32_t* row_src, float* row_gate, void* ws,
                               cudaStream_t st) {
    const Sizes s = sizes_of(c);
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    cudaError_t e = launch_offsets(topk_idx, topk_w, s.A, c.E, c.pad_multiple, s.R, counts, po,
                                   meta, nb, perm_row, row_src, row_gate,
                                   reinterpret_cast<uint32_t*>(w8),
                                   reinterpret_cast<int32_t*>(w8 + 256), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "offsets kernels");
}

// GEMM1 reads its A rows either from the permuted buffer x_perm (TMA) or,
// when x_perm is null, straight from the token rows x through row_src (the
// permute fused into the A load).
static moe_status_t do_experts(const moe_config_t& c, const void* x_perm, const void* W13,
                               const void* W2_t, const int32_t* meta, const int32_t* nb,
                               const int32_t* po, const float* row_gate, void* h, void* y,
                               uint32_t* status, cudaStream_t st, const void* x = nullptr,
                               const int32_t* row_src = nullptr, void* gu = nullptr,
                               const float* s13 = nullptr, const float* s2 = nullptr,
                               int32_t* visit_ready = nullptr) {
    const Sizes s = sizes_of(c);
    GemmArgs a{};
    a.block_metadata = meta;
    a.num_blocks = nb;
    a.nb_cap = static_cast<int32_t>(s.NB);
    a.padded_offsets = po;
    a.block_rows = c.pad_multiple;
    a.n_experts = c.E;
    a.status = status;
    // GEMM1: N = 2*d_e (gate/up interleaved), K = d
    a.n_tiles = (2 * c.d_e) / 256;
    a.k_blocks = c.d / 64;
    a.b_rows_per_expert = 2 * c.d_e;
    a.out = h;
    a.ldo = c.d_e;
    a.out_rows = s.R;
    a.gu_out = gu;  // the gate/up values saved for the backward, or null
    a.ld_gu = 2 * c.d_e;
    a.col_scale = s13;  // widened e4m3 weights: their per-channel scales
    const bool gather = x_perm == nullptr;
    a.gather_x = x;
    a.row_src = row_src;
    a.gather_k = c.k;
    if (visit_ready && !gather) {
        // the permute by GEMM1's copy warps: x_perm is written in the launch
        // that reads it (visit_ready cleared by the caller)
        a.cp_x = x;
        a.cp_row_src = row_src;
        a.cp_out = const_cast<void*>(x_perm);
        a.cp_ready = visit_ready;
        a.cp_k = c.k;
        a.cp_nvec = c.d / 8;
    }
    cudaError_t e = launch_grouped_gemm(gather ? kEpiSwiGLUGather : kEpiSwiGLU, 256,
                                        gather ? x : x_perm, gather ? c.T : s.R, W13,
                                        static_cast<int64_t>(c.E) * 2 * c.d_e, c.d, a,
                                        static_cast<int>(s.NB * a.n_tiles), st);
    if (e != cudaSuccess) return cuda_fail(e, "grouped GEMM1 (gate/up + SwiGLU)");
    a.cp_out = nullptr;
    // GEMM2: N = d, K = d_e
    const int bn2 = (c.d % 256 == 0) ? 256 : 128;
    a.gu_out = nullptr;
    a.col_scale = s2;
    a.n_tiles = c.d / bn2;
    a.k_blocks = c.d_e / 64;
    a.b_rows_per_expert = c.d;
    a.out = y;
    a.ldo = c.d;
    a.row_gate = row_gate;
    e = launch_grouped_gemm(kEpiGate, bn2, h, s.R, W2_t, static_cast<int64_t>(c.E) * c.d, c.d_e, a,
                            static_cast<int>(s.NB * a.n_tiles), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "grouped GEMM2 (down + gate)");
}

// The grouped GEMMs on the unpadded layout: rows [group_offsets[e],
// group_offsets[e + 1]) belong to expert e, with no padding between experts.
static moe_status_t do_experts_unpadded(const moe_config_t& c, const void* x_perm, const void* W13,
                                        const void* W2_t, const int32_t* group_offsets,
                                        const float* row_gate, void* h, void* y, uint32_t* status,
                                        cudaStream_t st) {
    const int64_t A = static_cast<int64_t>(c.T) * c.k;
    const int64_t windows = (A + 255) / 256 + c.E;  // at most: one more per expert boundary
    GemmArgs a{};
    a.unpadded = 1;
    a.padded_offsets = group_offsets;
    a.block_rows = c.pad_multiple;
    a.n_experts = c.E;
    a.status = status;
    a.n_tiles = (2 * c.d_e) / 256;
    a.k_blocks = c.d / 64;
    a.b_rows_per_expert = 2 * c.d_e;
    a.out = h;
    a.ldo = c.d_e;
    a.out_rows = A;
    cudaError_t e = launch_grouped_gemm(kEpiSwiGLU, 256, x_perm, A, W13,
                                        static_cast<int64_t>(c.E) * 2 * c.d_e, c.d, a,
                                        static_cast<int>(windows * a.n_tiles), st);
    if (e != cudaSuccess) return cuda_fail(e, "grouped GEMM1, unpadded");
    const int bn2 = (c.d % 256 == 0) ? 256 : 128;
    a.n_tiles = c.d / bn2;
    a.k_blocks = c.d_e / 64;
    a.b_rows_per_expert = c.d;
    a.out = y;
    a.ldo = c.d;
    a.row_gate = row_gate;
    e = launch_grouped_gemm(kEpiGate, bn2, h, A, W2_t, static_cast<int64_t>(c.E) * c.d, c.d_e, a,
                            static_cast<int>(windows * a.n_tiles), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "grouped GEMM2, unpadded");
}

// Operands of one expert (or of the shared expert) on the small-M kernel.
struct SkinnyIO {
    const void* x;         // token rows: bf16 [rows, d], or (e4m3) their pairs [2 rows, d]
    const float* x_scale;  // e4m3: scale of each token-row pair
    const void* W13;       // packed gate/up: bf16 or e4m3 codes
    const float* s13;      // e4m3: per-row scales
    const void* W2;        // packed down
    const float* s2;
    void* h;               // bf16 [rows, width]
    uint8_t* h8;           // e4m3: pairs of h [2 rows, width]
    float* h_scale;        // e4m3: their scales
    void* y;               // bf16 [rows, d]
    void* gu;              // bf16 [rows, 2 width]: GEMM1's gate/up values saved, or null
};

// The expert GEMMs on the swapped-operand kernel for blocks with few rows.
// With sh, the shared expert's dense tiles (T token rows) are appended to the
// same launches.  e4m3 weights: GEMM1 writes h in bf16, a split kernel turns
// the rows of h (and hs) into e4m3 pairs, GEMM2 multiplies those.
static moe_status_t do_experts_skinny(const moe_config_t& c, bool fp8, const SkinnyIO& r,
                                      const int32_t* meta, const int32_t* nb,
                                      const float* row_gate, uint32_t* status, cudaStream_t st,
                                      const SkinnyIO* sh = nullptr) {
    const Sizes s = sizes_of(c);
    const bool shared = c.d_shared > 0 && sh != nullptr;
    const int rows = skinny_tile_rows(fp8);
    const int ks = skinny_k_step(fp8);
    const int64_t chunks = (static_cast<int64_t>(c.T) + rows - 1) / rows;  // shared-expert tiles
    // a block holds at most min(P, T*k) valid rows (T*k: an expert may repeat
    // within a token of pre-routed input)
    const int64_t max_rows = std::min<int64_t>(c.pad_multiple, static_cast<int64_t>(c.T) * c.k);
    SkinnyArgs a{};
    a.n_chunks = static_cast<int32_t>((max_rows + rows - 1) / rows);
    a.block_metadata = meta;
    a.num_blocks = nb;
    a.nb_cap = static_cast<int32_t>(s.NB);
    a.n_experts = c.E;
    a.status = status;
    a.out_rows = s.R;
    // GEMM1: panels of 128 gate + 128 up rows, K = d
    a.n_panels = c.d_e / 128;
    a.rows_per_expert = 2 * c.d_e;
    a.k_blocks = c.d / ks;
    a.out = r.h;
    a.ldo = c.d_e;
    a.scale = r.s13;
    a.xscale = r.x_scale;
    a.gu_out = r.gu;
    a.ld_gu = 2 * c.d_e;
    if (shared) {
        a.s_rows = c.T;
        a.s_panels = c.d_shared / 128;
        a.s_rows_per_expert = 2 * c.d_shared;
        a.s_k_blocks = c.d / ks;
        a.s_out = sh->h;
        a.s_ldo = c.d_shared;
        a.s_scale = sh->s13;
        a.s_xscale = sh->x_scale;
        a.s_gu_out = sh->gu;
        a.s_ld_gu = 2 * c.d_shared;
    }
    int64_t tiles = s.NB * a.n_panels * a.n_chunks + (shared ? chunks * a.s_panels : 0);
    cudaError_t e = launch_grouped_gemm_skinny(
        kEpiSwiGLU, fp8, r.W13, static_cast<int64_t>(c.E) * 2 * c.d_e, r.x, s.R, c.d,
        shared ? sh->W13 : nullptr, 2 * static_cast<int64_t>(c.d_shared), shared ? sh->x : nullptr,
        c.T, c.d, a, static_cast<int>(tiles < (1 << 30) ? tiles : (1 << 30)), st);
    if (e != cudaSuccess) return cuda_fail(e, "grouped GEMM1, small-M kernel");
    if (fp8) {
        e = launch_split_rows_e4m3(r.h, meta, nb, meta ? static_cast<int>(s.NB) : 0, c.d_e, r.h8,
                                   r.h_scale, shared ? sh->h : nullptr, c.T, c.d_shared,
                                   shared ? sh->h8 : nullptr, shared ? sh->h_scale : nullptr, st);
        if (e != cudaSuccess) return cuda_fail(e, "e4m3 pairs of h");
    }
    // GEMM2: panels of 256 output rows, K = d_e (d_shared for the shared tiles)
    a.gu_out = nullptr;
    a.s_gu_out = nullptr;
    a.n_panels = (c.d + 255) / 256;
    a.rows_per_expert = c.d;
    a.k_blocks = c.d_e / ks;
    a.out = r.y;
    a.ldo = c.d;
    a.row_gate = row_gate;
    a.scale = r.s2;
    a.xscale = r.h_scale;
    if (shared) {
        a.s_panels = (c.d + 255) / 256;
        a.s_rows_per_expert = c.d;
        a.s_k_blocks = c.d_shared / ks;
        a.s_out = sh->y;
        a.s_ldo = c.d;
        a.s_scale = sh->s2;
        a.s_xscale = sh->h_scale;
    }
    tiles = s.NB * a.n_panels * a.n_chunks + (shared ? chunks * a.s_panels : 0);
    const void* h_in = fp8 ? static_cast<const void*>(r.h8) : r.h;
    const void* hs_in = shared ? (fp8 ? static_cast<const void*>(sh->h8) : sh->h) : nullptr;
    e = launch_grouped_gemm_skinny(kEpiGate, fp8, r.W2, static_cast<int64_t>(c.E) * c.d, h_in, s.R,
                                   c.d_e, shared ? sh->W2 : nullptr, c.d, hs_in, c.T, c.d_shared, a,
                                   static_cast<int>(tiles < (1 << 30) ? tiles : (1 << 30)), st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "grouped GEMM2, small-M kernel");
}

// The permute in the shared expert's GEMM1 epilogue (null x_perm: none).
struct FusedPermute {
    const int32_t* perm_row;
    void* x_perm;
};

// The routed rows that the shared expert's GEMM2 adds into its output rows
// when the combine is fused there (null y: no fusion).
struct FusedCombine {
    const void* y;
    const int32_t* perm_row;
    void* out;
};

// The shared expert's gate/up GEMM: hs = bf16(silu(x Ws1) * (x Ws3)), 256-row
// visits of the token rows; with perm, the permute in its epilogue.
static moe_status_t do_shared_up(const moe_config_t& c, const void* x, const void* Ws13, void* hs,
                                 uint32_t* status, cudaStream_t st, void* gus = nullptr,
                                 const float* ss13 = nullptr, const FusedPermute* perm = nullptr) {
    GemmArgs a{};
    a.dense_rows = c.T;
    a.status = status;
    a.block_rows = 256;
    a.n_tiles = (2 * c.d_shared) / 256;
    a.k_blocks = c.d / 64;
    a.b_rows_per_expert = 0;
    a.out = hs;
    a.ldo = c.d_shared;
    a.out_rows = c.T;
    a.gu_out = gus;
    a.ld_gu = 2 * c.d_shared;
    a.col_scale = ss13;
    if (perm && perm->x_perm) {
        a.perm_x = x;
        a.perm_rows = perm->perm_row;
        a.perm_out = perm->x_perm;
        a.perm_k = c.k;
        a.perm_nvec = c.d / 8;
    }
    const int mblocks = (c.T + 255) / 256;  // 256-row visits of the CTA-pair kernel
    cudaError_t e = launch_grouped_gemm(kEpiSwiGLU, 256, x, c.T, Ws13, 2 * c.d_shared, c.d, a,
                                        mblocks * a.n_tiles, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "shared GEMM1");
}

// The shared expert's down projection: ys = bf16(hs Ws2); with comb, the
// combine in its epilogue writes the layer output instead.
static moe_status_t do_shared_down(const moe_config_t& c, const void* hs, const void* Ws2_t,
                                   void* ys, uint32_t* status, cudaStream_t st,
                                   const float* ss2 = nullptr, const FusedCombine* comb = nullptr) {
    GemmArgs a{};
    a.dense_rows = c.T;
    a.status = status;
    a.block_rows = 256;
    const int bn2 = (c.d % 256 == 0) ? 256 : 128;
    a.col_scale = ss2;
    a.n_tiles = c.d / bn2;
    a.k_blocks = c.d_shared / 64;
    a.b_rows_per_expert = 0;
    a.out = ys;
    a.ldo = c.d;
    a.out_rows = c.T;
    int epi = kEpiGate;
    if (comb && comb->y) {
        // the combine in GEMM2's epilogue: the output rows are the layer's
        a.out = comb->out;
        a.comb_y = comb->y;
        a.comb_perm = comb->perm_row;
        a.comb_k = c.k;
        a.comb_ldy = c.d;
        epi = kEpiCombine;
    }
    const int mblocks = (c.T + 255) / 256;
    cudaError_t e = launch_grouped_gemm(epi, bn2, hs, c.T, Ws2_t, c.d, c.d_shared, a,
                                        mblocks * a.n_tiles, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "shared GEMM2");
}

static moe_status_t do_shared(const moe_config_t& c, const void* x, const void* Ws13,
                              const void* Ws2_t, void* hs, void* ys, uint32_t* status,
                              cudaStream_t st, void* gus = nullptr, const float* ss13 = nullptr,
                              const float* ss2 = nullptr) {
    moe_status_t r = do_shared_up(c, x, Ws13, hs, status, st, gus, ss13);
    return r != MOE_OK ? r : do_shared_down(c, hs, Ws2_t, ys, status, st, ss2);
}

// Pointers into a layer workspace.
struct LayerBufs {
    const moe_workspace_layout_t L;
    uint8_t* b;
    void* at(size_t o) const { return static_cast<void*>(b + o); }
    uint32_t* status() const { return static_cast<uint32_t*>(at(L.status)); }
    int32_t* meta() const { return static_cast<int32_t*>(at(L.block_metadata)); }
    int32_t* nb() const { return static_cast<int32_t*>(at(L.num_blocks)); }
    int32_t* perm_row() const { return static_cast<int32_t*>(at(L.perm_row)); }
    float* row_gate() const { return static_cast<float*>(at(L.row_gate)); }
    const int32_t* po() const { return static_cast<const int32_t*>(at(L.padded_offsets)); }
};

// The front of the layer shared by both weight formats: the router (or the
// given routing) and the offsets stage.
static moe_status_t layer_front(const moe_config_t& c, const void* Wg_t, const float* bias,
                                const void* x, const int32_t* pre_idx, const float* pre_w,
                                const LayerBufs& B, cudaStream_t st) {
    int32_t* topk_idx = static_cast<int32_t*>(B.at(B.L.topk_idx));
    float* topk_w = static_cast<float*>(B.at(B.L.topk_w));
    if (!pre_idx) {
        moe_status_t r = do_route_layer(c, x, Wg_t, bias, topk_idx, topk_w,
                                        static_cast<float*>(B.at(B.L.router_partial)), st,
                                        B.status());
        if (r != MOE_OK) return r;
    } else {
        topk_idx = const_cast<int32_t*>(pre_idx);
        topk_w = const_cast<float*>(pre_w);
    }
    return do_offsets(c, topk_idx, topk_w, static_cast<int32_t*>(B.at(B.L.counts)),
                      static_cast<int32_t*>(B.at(B.L.padded_offsets)), B.meta(), B.nb(),
                      B.perm_row(), static_cast<int32_t*>(B.at(B.L.row_src)), B.row_gate(),
                      B.at(B.L.status), st);
}

static moe_status_t check_layer_args(const moe_config_t* cfg, bool routed, const void* Wg_t,
                                     const void* x, const float* pre_w, void* out, void* ws,
                                     size_t ws_bytes, bool fp8 = false) {
    moe_status_t r = check_cfg(cfg, routed);
    if (r != MOE_OK) return r;
    // an empty batch has no token rows: x, out and the gates may be null
    if (cfg->T > 0 && (!x || !out)) return fail(MOE_ERR_INVALID_ARG, "null x or out");
    if (routed && !Wg_t) return fail(MOE_ERR_INVALID_ARG, "null router weight");
    if (!routed && !pre_w && cfg->T > 0) return fail(MOE_ERR_INVALID_ARG, "null pre-routed gates");
    const size_t need = layout_of(*cfg, fp8).total;
    if (!ws || ws_bytes < need)
        return fail(MOE_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, need);
    return MOE_OK;
}

// Bytes of the routed part of a gate/up save (the shared expert's follows).
static size_t gate_up_routed_bytes(const moe_config_t& c) {
    return align_up(static_cast<size_t>(sizes_of(c).R) * 2 * c.d_e * 2, 1024);
}

static size_t gate_up_save_bytes(const moe_config_t& c) {
    return gate_up_routed_bytes(c) + static_cast<size_t>(c.T) * 2 * c.d_shared * 2;
}

static moe_status_t layer(const moe_config_t* cfg, const moe_weights_t* w, const void* x,
                          const int32_t* pre_idx, const float* pre_w, void* out, void* ws,
                          size_t ws_bytes, cudaStream_t st, void* gu_save = nullptr) {
    if (!w) return fail(MOE_ERR_INVALID_ARG, "null weights");
    moe_status_t r = check_layer_args(cfg, pre_idx == nullptr, w->Wg_t, x, pre_w, out, ws, ws_bytes);
    if (r != MOE_OK) return r;
    const moe_config_t& c = *cfg;
    if (!w->W13 || !w->W2) return fail(MOE_ERR_INVALID_ARG, "null routed expert weights");
    if (c.d_shared && (!w->Ws13 || !w->Ws2))
        return fail(MOE_ERR_INVALID_ARG, "d_shared > 0 but null shared expert weights");
    if (c.T == 0) return MOE_OK;
    const LayerBufs B{layout_of(c), static_cast<uint8_t*>(ws)};
    const moe_workspace_layout_t& L = B.L;
    r = layer_front(c, w->Wg_t, w->bias, x, pre_idx, pre_w, B, st);
    if (r != MOE_OK) return r;
    const void* shared = c.d_shared ? B.at(L.ys) : nullptr;
    // gate/up values saved for the backward: routed rows, then the shared expert's
    void* gu = gu_save;
    void* gus = gu_save && c.d_shared ? static_cast<uint8_t*>(gu_save) + gate_up_routed_bytes(c)
                                      : nullptr;
    cudaError_t e = cudaSuccess;
    if (use_skinny(c)) {
        e = launch_permute(x, B.perm_row(), B.at(L.x_perm), c.T, c.d, c.k, st);
        if (e != cudaSuccess) return cuda_fail(e, "permute");
        const SkinnyIO ro{B.at(L.x_perm), nullptr, w->W13, nullptr, w->W2, nullptr,
                          B.at(L.h), nullptr, nullptr, B.at(L.y), gu};
        const SkinnyIO so{x, nullptr, w->Ws13, nullptr, w->Ws2, nullptr,
                          B.at(L.hs), nullptr, nullptr, B.at(L.ys), gus};
        r = do_experts_skinny(c, false, ro, B.meta(), B.nb(), B.row_gate(), B.status(), st,
                              c.d_shared ? &so : nullptr);
        if (r != MOE_OK) return r;
    } else {
        if (c.d_shared) {
            // the shared expert's GEMM1 first, with the permute in the slack
            // of its epilogue; its GEMM2 after the routed GEMMs
            const FusedPermute fp{B.perm_row(), B.at(L.x_perm)};
            r = do_shared_up(c, x, w->Ws13, B.at(L.hs), B.status(), st, gus, nullptr, &fp);
        } else {
            // the permute as its own kernel (in GEMM1's copy warps it was no
            // faster: moe_grouped_gemm_swiglu_permute)
            e = launch_permute(x, B.perm_row(), B.at(L.x_perm), c.T, c.d, c.k, st);
            r = e == cudaSuccess ? MOE_OK : cuda_fail(e, "permute");
        }
        if (r != MOE_OK) return r;
        r = do_experts(c, B.at(L.x_perm), w->W13, w->W2, B.meta(), B.nb(), B.po(), B.row_gate(),
                       B.at(L.h), B.at(L.y), B.status(), st, nullptr, nullptr, gu);
        if (r != MOE_OK) return r;
        if (c.d_shared) {
            r = do_shared_down(c, B.at(L.hs), w->Ws2, B.at(L.ys), B.status(), st);
            if (r != MOE_OK) return r;
        }
    }
    e = launch_combine(B.at(L.y), B.perm_row(), shared, out, c.T, c.d, c.k, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine");
}

static moe_status_t layer_fp8(const moe_config_t* cfg, const moe_weights_fp8_t* w, const void* x,
                              const int32_t* pre_idx, const float* pre_w, void* out, void* ws,
                              size_t ws_bytes, cudaStream_t st) {
    if (!w) return fail(MOE_ERR_INVALID_ARG, "null weights");
    moe_status_t r =
        check_layer_args(cfg, pre_idx == nullptr, w->Wg_t, x, pre_w, out, ws, ws_bytes, true);
    if (r != MOE_OK) return r;
    const moe_config_t& c = *cfg;
    if (!w->W13q || !w->s13 || !w->W2q || !w->s2)
        return fail(MOE_ERR_INVALID_ARG, "null routed expert codes or scales");
    if (c.d_shared && (!w->Ws13q || !w->ss13 || !w->Ws2q || !w->ss2))
        return fail(MOE_ERR_INVALID_ARG, "d_shared > 0 but null shared expert codes or scales");
    if (c.T == 0) return MOE_OK;
    const LayerBufs B{layout_of(c, true), static_cast<uint8_t*>(ws)};
    const moe_workspace_layout_t& L = B.L;
    if (!use_skinny(c)) {
        // Enough rows per expert that the tensor pipe, not the weight bytes,
        // sets the pace: widen the codes to bf16 (exact) and run the CTA-pair
        // GEMMs, which scale their accumulators per output channel ("Dropless
        // and grouped GEMM", sec. 12: a scale covering the whole contraction
        // multiplies the product).
        uint8_t* w16 = static_cast<uint8_t*>(B.at(L.w16));
        const size_t n13 = static_cast<size_t>(c.E) * 2 * c.d_e * c.d;
        const size_t n2 = static_cast<size_t>(c.E) * c.d * c.d_e;
        const size_t ns13 = static_cast<size_t>(2) * c.d_shared * c.d;
        void* W13w = w16;
        void* W2w = w16 + n13 * 2;
        void* Ws13w = w16 + (n13 + n2) * 2;
        void* Ws2w = w16 + (n13 + n2 + ns13) * 2;
        cudaError_t e = launch_widen_e4m3(w->W13q, W13w, static_cast<int64_t>(n13), st);
        if (e == cudaSuccess) e = launch_widen_e4m3(w->W2q, W2w, static_cast<int64_t>(n2), st);
        if (e == cudaSuccess && c.d_shared) {
            e = launch_widen_e4m3(w->Ws13q, Ws13w, static_cast<int64_t>(ns13), st);
            if (e == cudaSuccess) e = launch_widen_e4m3(w->Ws2q, Ws2w, static_cast<int64_t>(ns13 / 2), st);
        }
        if (e != cudaSuccess) return cuda_fail(e, "widen e4m3 weights");
        r = layer_front(c, w->Wg_t, w->bias, x, pre_idx, pre_w, B, st);
        if (r != MOE_OK) return r;
        if (c.d_shared) {  // as the bf16 layer: the permute in the shared GEMM1's epilogue
            const FusedPermute fp{B.perm_row(), B.at(L.x_perm)};
            r = do_shared_up(c, x, Ws13w, B.at(L.hs), B.status(), st, nullptr, w->ss13, &fp);
            if (r != MOE_OK) return r;
        } else {
            e = launch_permute(x, B.perm_row(), B.at(L.x_perm), c.T, c.d, c.k, st);
            if (e != cudaSuccess) return cuda_fail(e, "permute");
        }
        r = do_experts(c, B.at(L.x_perm), W13w, W2w, B.meta(), B.nb(), B.po(), B.row_gate(),
                       B.at(L.h), B.at(L.y), B.status(), st, nullptr, nullptr, nullptr, w->s13, w->s2);
        if (r != MOE_OK) return r;
        if (c.d_shared) {
            r = do_shared_down(c, B.at(L.hs), Ws2w, B.at(L.ys), B.status(), st, w->ss2);
            if (r != MOE_OK) return r;
        }
        e = launch_combine(B.at(L.y), B.perm_row(), c.d_shared ? B.at(L.ys) : nullptr, out, c.T, c.d,
                           c.k, st);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine");
    }
    r = layer_front(c, w->Wg_t, w->bias, x, pre_idx, pre_w, B, st);
    if (r != MOE_OK) return r;
    const Sizes s = sizes_of(c);
    float* scales = static_cast<float*>(B.at(L.row_scale));  // x [R], h [R], xs [T], hs [T]
    uint8_t* h8 = static_cast<uint8_t*>(B.at(L.h8));
    uint8_t* x8 = static_cast<uint8_t*>(B.at(L.x_perm));
    uint8_t* xs8 = c.d_shared ? static_cast<uint8_t*>(B.at(L.xs8)) : nullptr;
    cudaError_t e = launch_permute_fp8(x, B.perm_row(), x8, scales, xs8,
                                       c.d_shared ? scales + 2 * s.R : nullptr, c.T, c.d, c.k, st);
    if (e != cudaSuccess) return cuda_fail(e, "permute (e4m3 pairs)");
    const SkinnyIO ro{x8, scales, w->W13q, w->s13, w->W2q, w->s2,
                      B.at(L.h), h8, scales + s.R, B.at(L.y)};
    const SkinnyIO so{xs8, scales + 2 * s.R, w->Ws13q, w->ss13, w->Ws2q, w->ss2,
                      B.at(L.hs), h8 + static_cast<size_t>(s.R) * c.d_e * 2,
                      scales + 2 * s.R + c.T, B.at(L.ys)};
    r = do_experts_skinny(c, true, ro, B.meta(), B.nb(), B.row_gate(), B.status(), st,
                          c.d_shared ? &so : nullptr);
    if (r != MOE_OK) return r;
    e = launch_combine(B.at(L.y), B.perm_row(), c.d_shared ? B.at(L.ys) : nullptr, out, c.T, c.d,
                       c.k, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine");
}

// ------------------------------------------------------------ backward --

struct BwdLayout {
    size_t total;
    size_t dgates, dz, xp, gu, hp, dh, dgu, dxp;                     // routed experts
    size_t dl32, dl16, dxr;                                            // router
    size_t gus, hs, dhs, dgus, dxs;                                  // shared expert
    int64_t Ep;
};

static inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

static BwdLayout bwd_layout_of(const moe_config_t& c) {
    const Sizes s = sizes_of(c);
    BwdLayout B{};
    B.Ep = round_up(c.E, 128);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 1024);
        return o;
    };
    const size_t R = static_cast<size_t>(s.R), T = static_cast<size_t>(c.T);
    const size_t d = c.d, de = c.d_e, ds = c.d_shared, E = c.E;
    B.dgates = take(T * c.k * 4);
    B.dz = take(R * d * 2);
    B.xp = take(R * d * 2);
    B.gu = take(R * 2 * de * 2);
    B.hp = take(R * de * 2);
    B.dh = take(R * de * 2);
    B.dgu = take(R * 2 * de * 2);
    B.dxp = take(R * d * 2);
    B.dl32 = take(T * E * 4);
    B.dl16 = take(T * B.Ep * 2);
    B.dxr = take(T * d * 2);
    B.gus = take(T * 2 * ds * 2);
    B.hs = take(T * ds * 2);
    B.dhs = take(T * ds * 2);
    B.dgus = take(T * 2 * ds * 2);
    B.dxs = take(T * d * 2);
    B.total = off;
    return B;
}

// A plain bf16 GEMM on the CTA-pair kernel: out[r] = A[r] B[e]^T for the
// blocks of the table (meta != null) or for `rows` dense rows.
static cudaError_t pair_gemm(const moe_config_t& c, const void* A, int64_t rowsA, const void* B,
                             int64_t rowsB_per_expert, int64_t K, int64_t N, void* out,
                             int64_t out_rows, const int32_t* meta, const int32_t* nb,
                             const int32_t* po, uint32_t* status, cudaStream_t st) {
    const Sizes s = sizes_of(c);
    const int bn = N % 256 == 0 ? 256 : 128;
    GemmArgs a{};
    a.status = status;
    a.n_tiles = static_cast<int32_t>(N / bn);
    a.k_blocks = static_cast<int32_t>((K + 63) / 64);
    a.out = out;
    a.ldo = N;
    a.out_rows = out_rows;
    int64_t tiles;
    int64_t rowsB;
    if (meta) {
        a.block_metadata = meta;
        a.num_blocks = nb;
        a.nb_cap = static_cast<int32_t>(s.NB);
        a.padded_offsets = po;
        a.block_rows = c.pad_multiple;
        a.n_experts = c.E;
        a.b_rows_per_expert = static_cast<int32_t>(rowsB_per_expert);
        tiles = s.NB * a.n_tiles;
        rowsB = rowsB_per_expert * c.E;
    } else {
        a.dense_rows = static_cast<int32_t>(rowsA);
        a.block_rows = 256;
        tiles = ((rowsA + 255) / 256) * a.n_tiles;
        rowsB = rowsB_per_expert;
    }
    return launch_grouped_gemm(kEpiGate, bn, A, rowsA, B, rowsB, K, a,
                               static_cast<int>(tiles < (1 << 30) ? tiles : (1 << 30)), st);
}

static moe_status_t layer_bwd(const moe_config_t* cfg, const moe_weights_t* w,
                              const moe_weights_bwd_t* wb, const void* x, const void* dout,
                              const void* fwd_ws, size_t fwd_ws_bytes, const void* gu_saved,
                              size_t gu_saved_bytes, const moe_grads_t* g, void* bws,
                              size_t bws_bytes, cudaStream_t st) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    const moe_config_t& c = *cfg;
    if (c.T == 0) return MOE_OK;  // nothing to differentiate; no pointer is read
    if (!w || !wb || !g || !x || !dout || !fwd_ws)
        return fail(MOE_ERR_INVALID_ARG, "null weights, gradients, x, dout or forward workspace");
    if (!w->W13 || !wb->W13t || !wb->W2 || !g->dx || !g->dW1 || !g->dW3 || !g->dW2)
        return fail(MOE_ERR_INVALID_ARG, "null routed expert weights or gradients");
    const bool router = wb->WgP != nullptr;
    if ((g->dWg || g->dbias) && !router)
        return fail(MOE_ERR_INVALID_ARG, "router gradients asked for without WgP");
    const bool shared = c.d_shared > 0;
    if (shared && (!w->Ws13 || !wb->Ws13t || !wb->Ws2 || !g->dWs1 || !g->dWs3 || !g->dWs2))
        return fail(MOE_ERR_INVALID_ARG, "d_shared > 0 but null shared weights or gradients");
    // the backward reads only the routing state at the front of the forward
    // workspace (everything before x_perm)
    const moe_workspace_layout_t L = layout_of(c);
    if (fwd_ws_bytes < L.x_perm)
        return fail(MOE_ERR_WORKSPACE, "forward routing state of %zu bytes, %zu expected",
                    fwd_ws_bytes, L.x_perm);
    if (gu_saved && gu_saved_bytes < gate_up_save_bytes(c))
        return fail(MOE_ERR_WORKSPACE, "gate/up save of %zu bytes, %zu expected", gu_saved_bytes,
                    gate_up_save_bytes(c));
    const BwdLayout B = bwd_layout_of(c);
    if (!bws || bws_bytes < B.total)
        return fail(MOE_ERR_WORKSPACE, "backward workspace of %zu bytes, %zu needed", bws_bytes,
                    B.total);
    const Sizes s = sizes_of(c);
    const uint8_t* fw = static_cast<const uint8_t*>(fwd_ws);
    uint8_t* bw = static_cast<uint8_t*>(bws);
    auto F = [&](size_t o) { return const_cast<void*>(static_cast<const void*>(fw + o)); };
    auto W = [&](size_t o) { return static_cast<void*>(bw + o); };
    uint32_t* status = static_cast<uint32_t*>(F(L.status));
    const int32_t* meta = static_cast<const int32_t*>(F(L.block_metadata));
    const int32_t* nb = static_cast<const int32_t*>(F(L.num_blocks));
    const int32_t* po = static_cast<const int32_t*>(F(L.padded_offsets));
    const int32_t* perm_row = static_cast<const int32_t*>(F(L.perm_row));
    const int32_t* row_src = static_cast<const int32_t*>(F(L.row_src));
    const float* row_gate = static_cast<const float*>(F(L.row_gate));
    float* dgates = g->dgates ? g->dgates : static_cast<float*>(W(B.dgates));
    const int d = c.d, de = c.d_e, E = c.E;
    cudaError_t e;
#define MOE_BWD_CHECK(what)                  \
    if (e != cudaSuccess) return cuda_fail(e, what)
    // combine backward: the rows of dout in the padded order (dz_a = dout[t]);
    // the permuted token rows again, from x and the sort indices
    e = launch_permute(dout, perm_row, W(B.dz), c.T, d, c.k, st);
    if (e == cudaSuccess) e = launch_permute(x, perm_row, W(B.xp), c.T, d, c.k, st);
    MOE_BWD_CHECK("permutes of dout and x");
    // routed experts, data gradients: dh = dz W2^T (before the routing
    // weight), [g|u] and h recomputed, dgu and dgates, dx_perm
    e = pair_gemm(c, W(B.dz), s.R, wb->W2, de, d, de, W(B.dh), s.R, meta, nb, po, status, st);
    MOE_BWD_CHECK("dh = dz W2^T");
    // the gate/up values: saved by the forward, or recomputed
    const void* gu = gu_saved;
    if (!gu) {
        e = pair_gemm(c, W(B.xp), s.R, w->W13, 2 * de, d, 2 * de, W(B.gu), s.R, meta, nb, po, status,
                      st);
        MOE_BWD_CHECK("gate/up recomputation");
        gu = W(B.gu);
    }
    e = launch_swiglu_bwd(gu, W(B.dh), row_src, row_gate, po + E, W(B.hp), W(B.dgu), dgates,
                          W(B.dz), W(B.xp), d, s.R, de, st);
    MOE_BWD_CHECK("SwiGLU backward");
    e = pair_gemm(c, W(B.dgu), s.R, wb->W13t, d, 2 * de, d, W(B.dxp), s.R, meta, nb, po, status, st);
    MOE_BWD_CHECK("dx_perm = dgu W13");
    // routed experts, weight gradients over each expert's rows (pad rows
    // zeroed above): dW2 = (p h)^T dz, [dW1 | dW3] = x_perm^T dgu
    const int32_t* counts = static_cast<const int32_t*>(F(L.counts));
    e = launch_wgrad(W(B.hp), de, W(B.dz), d, s.R, po, E, 0, g->dW2, nullptr, status, st, 0, counts);
    MOE_BWD_CHECK("dW2");
    e = launch_wgrad(W(B.xp), d, W(B.dgu), 2 * de, s.R, po, E, 0, g->dW1, g->dW3, status, st, 0,
                     counts);
    MOE_BWD_CHECK("dW1, dW3");
    const void* dxr = nullptr;
    if (router) {
        const int32_t* idx = static_cast<const int32_t*>(F(L.topk_idx));
        const float* gates = static_cast<const float*>(F(L.topk_w));
        e = launch_router_bwd(dgates, idx, gates, static_cast<float*>(W(B.dl32)), W(B.dl16), c.T, E,
                              c.k, static_cast<int>(B.Ep), g->dbias, st);
        MOE_BWD_CHECK("router backward");
    }
    if (router && g->dWg) {
        // dWg [d, E] = x^T dlogits (fp32), on the weight-gradient kernel
        e = launch_wgrad(x, d, W(B.dl16), B.Ep, c.T, nullptr, 1, c.T, g->dWg, nullptr, status, st, E);
        MOE_BWD_CHECK("dWg");
    }
    if (router) {
        e = pair_gemm(c, W(B.dl16), c.T, wb->WgP, d, B.Ep, d, W(B.dxr), c.T, nullptr, nullptr,
                      nullptr, status, st);
        MOE_BWD_CHECK("dx from the router");
        dxr = W(B.dxr);
    }
    const void* dxs = nullptr;
    if (shared) {
        const int ds = c.d_shared;
        const void* gus = gu_saved ? static_cast<const uint8_t*>(gu_saved) + gate_up_routed_bytes(c)
                                   : nullptr;
        if (!gus) {
            e = pair_gemm(c, x, c.T, w->Ws13, 2 * ds, d, 2 * ds, W(B.gus), c.T, nullptr, nullptr,
                          nullptr, status, st);
            gus = W(B.gus);
        }
        if (e == cudaSuccess)
            e = pair_gemm(c, dout, c.T, wb->Ws2, ds, d, ds, W(B.dhs), c.T, nullptr, nullptr, nullptr,
                          status, st);
        if (e == cudaSuccess)
            e = launch_swiglu_bwd(gus, W(B.dhs), nullptr, nullptr, nullptr, W(B.hs), W(B.dgus),
                                  nullptr, nullptr, nullptr, 0, c.T, ds, st);
        if (e == cudaSuccess)
            e = pair_gemm(c, W(B.dgus), c.T, wb->Ws13t, d, 2 * ds, d, W(B.dxs), c.T, nullptr, nullptr,
                          nullptr, status, st);
        MOE_BWD_CHECK("shared expert data gradients");
        if (e == cudaSuccess)
            e = launch_wgrad(W(B.hs), ds, dout, d, c.T, nullptr, 1, c.T, g->dWs2, nullptr, status, st);
        if (e == cudaSuccess)
            e = launch_wgrad(x, d, W(B.dgus), 2 * ds, c.T, nullptr, 1, c.T, g->dWs1, g->dWs3, status,
                             st);
        MOE_BWD_CHECK("shared expert weight gradients");
        dxs = W(B.dxs);
    }
    // dx: the k rows of each token (permute backward), then the router and
    // shared-expert terms, in that order
    if (!dxr) {
        dxr = dxs;
        dxs = nullptr;
    }
    e = launch_combine(W(B.dxp), perm_row, dxr, g->dx, c.T, d, c.k, st, dxs);
    MOE_BWD_CHECK("dx");
#undef MOE_BWD_CHECK
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_check_config(const moe_config_t* cfg) { return check_cfg(cfg, false); }

size_t moe_workspace_size(const moe_config_t* cfg) {
    if (check_cfg(cfg, false) != MOE_OK) return 0;
    return layout_of(*cfg).total;
}

size_t moe_workspace_size_fp8(const moe_config_t* cfg) {
    if (check_cfg(cfg, false) != MOE_OK) return 0;
    return layout_of(*cfg, true).total;
}

moe_status_t moe_workspace_layout_fp8(const moe_config_t* cfg, moe_workspace_layout_t* layout) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!layout) return fail(MOE_ERR_INVALID_ARG, "layout is NULL");
    *layout = layout_of(*cfg, true);
    return MOE_OK;
}

moe_status_t moe_workspace_layout(const moe_config_t* cfg, moe_workspace_layout_t* layout) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!layout) return fail(MOE_ERR_INVALID_ARG, "layout is NULL");
    *layout = layout_of(*cfg);
    return MOE_OK;
}

size_t moe_offsets_workspace_size(const moe_config_t* cfg) {
    if (check_cfg(cfg, false) != MOE_OK) return 0;
    return offsets_ws_bytes(*cfg);
}

moe_status_t moe_pack_router(int32_t d, int32_t E, const void* Wg, void* Wg_t, void* stream) {
    if (d <= 0 || E <= 0 || !Wg || !Wg_t) return fail(MOE_ERR_INVALID_ARG, "bad router pack args");
    cudaError_t e = launch_pack_transpose(Wg, Wg_t, d, E, 0, 0, d, 0, 1,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "pack router");
}

moe_status_t moe_pack_experts(int32_t E, int32_t d, int32_t de, const void* W1, const void* W3,
                              const void* W2, void* W13, void* W2_t, void* stream) {
    if (E <= 0 || d <= 0 || de <= 0 || !W1 || !W3 || !W2 || !W13 || !W2_t)
        return fail(MOE_ERR_INVALID_ARG, "bad expert pack args");
    if (d % 128 || de % 128) return fail(MOE_ERR_UNSUPPORTED, "d and de must be multiples of 128");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t dd = d, dde = de;
    cudaError_t e = launch_pack_transpose(W1, W13, d, de, dd * dde, 2 * dde * dd, d, 1, E, st);
    if (e == cudaSuccess) e = launch_pack_transpose(W3, W13, d, de, dd * dde, 2 * dde * dd, d, 2, E, st);
    if (e == cudaSuccess) e = launch_pack_transpose(W2, W2_t, de, d, dde * dd, dd * dde, de, 0, E, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "pack experts");
}

moe_status_t moe_pack_weights(const moe_config_t* cfg, const void* W1, const void* W3,
                              void* W13_packed, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!W1 || !W3 || !W13_packed) return fail(MOE_ERR_INVALID_ARG, "null gate/up weights");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t dd = cfg->d, dde = cfg->d_e;
    cudaError_t e = launch_pack_transpose(W1, W13_packed, cfg->d, cfg->d_e, dd * dde, 2 * dde * dd,
                                          cfg->d, 1, cfg->E, st);
    if (e == cudaSuccess)
        e = launch_pack_transpose(W3, W13_packed, cfg->d, cfg->d_e, dd * dde, 2 * dde * dd, cfg->d,
                                  2, cfg->E, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "pack gate/up weights");
}

moe_status_t moe_pack_experts_fp8(int32_t E, int32_t d, int32_t de, const void* W1, const void* W3,
                                  const void* W2, void* W13q, float* s13, void* W2q, float* s2,
                                  void* stream) {
    if (E <= 0 || d <= 0 || de <= 0 || !W1 || !W3 || !W2 || !W13q || !s13 || !W2q || !s2)
        return fail(MOE_ERR_INVALID_ARG, "bad e4m3 expert pack args");
    if (d % 128 || de % 128) return fail(MOE_ERR_UNSUPPORTED, "d and de must be multiples of 128");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t dd = d, dde = de;
    uint8_t* q13 = static_cast<uint8_t*>(W13q);
    uint8_t* q2 = static_cast<uint8_t*>(W2q);
    cudaError_t e = launch_pack_fp8(W1, q13, s13, d, de, dd * dde, 2 * dde * dd, 2 * dde, d, 1, E, st);
    if (e == cudaSuccess)
        e = launch_pack_fp8(W3, q13, s13, d, de, dd * dde, 2 * dde * dd, 2 * dde, d, 2, E, st);
    if (e == cudaSuccess) e = launch_pack_fp8(W2, q2, s2, de, d, dde * dd, dd * dde, dd, de, 0, E, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "pack experts (e4m3)");
}

moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* Wg_t, const float* bias,
                       int32_t* topk_idx, float* topk_w, void* stream) {
    moe_status_t r = check_cfg(cfg, true);
    if (r != MOE_OK) return r;
    if (!x || !Wg_t || !topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    return do_route(*cfg, x, Wg_t, bias, topk_idx, topk_w, static_cast<cudaStream_t>(stream));
}

size_t moe_route_splitk_scratch_size(const moe_config_t* cfg) {
    if (check_cfg(cfg, true) != MOE_OK) return 0;
    const int S = router_splits(*cfg);
    return S > 1 && !router_uses_cluster(*cfg) ? static_cast<size_t>(S) * cfg->T * cfg->E * 4 : 0;
}

moe_status_t moe_route_splitk(const moe_config_t* cfg, const void* x, const void* Wg_t,
                              const float* bias, int32_t* topk_idx, float* topk_w, float* partial,
                              size_t partial_bytes, void* stream) {
    moe_status_t r = check_cfg(cfg, true);
    if (r != MOE_OK) return r;
    if (!x || !Wg_t || !topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    const size_t need = moe_route_splitk_scratch_size(cfg);
    if (need && (!partial || partial_bytes < need))
        return fail(MOE_ERR_WORKSPACE, "split-K router scratch of %zu bytes, %zu needed",
                    partial_bytes, need);
    if (cfg->T == 0) return MOE_OK;
    return do_route_layer(*cfg, x, Wg_t, bias, topk_idx, topk_w, partial,
                          static_cast<cudaStream_t>(stream));
}

moe_status_t moe_build_offsets(const moe_config_t* cfg, const int32_t* topk_idx,
                               const float* topk_w, int32_t* counts, int32_t* padded_offsets,
                               int32_t* block_metadata, int32_t* num_blocks, int32_t* perm_row,
                               int32_t* row_src, float* row_gate, void* ws, size_t ws_bytes,
                               void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!topk_idx || !counts || !padded_offsets || !block_metadata || !num_blocks || !perm_row ||
        !row_src || !row_gate)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    const size_t need = offsets_ws_bytes(*cfg);
    if (!ws || ws_bytes < need)
        return fail(MOE_ERR_WORKSPACE, "offsets scratch of %zu bytes, %zu needed", ws_bytes, need);
    if (cfg->T == 0) return MOE_OK;
    return do_offsets(*cfg, topk_idx, topk_w, counts, padded_offsets, block_metadata, num_blocks,
                      perm_row, row_src, row_gate, ws, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_permute(const moe_config_t* cfg, const void* x, const int32_t* perm_row,
                         void* x_perm, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!x || !perm_row || !x_perm) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    cudaError_t e = launch_permute(x, perm_row, x_perm, cfg->T, cfg->d, cfg->k,
                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "permute");
}

moe_status_t moe_grouped_gemm_swiglu(const moe_config_t* cfg, const void* x_perm, const void* W13,
                                     const void* W2_t, const int32_t* block_metadata,
                                     const int32_t* num_blocks, const int32_t* padded_offsets,
                                     const float* row_gate, void* h, void* y, uint32_t* status,
                                     void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!x_perm || !W13 || !W2_t || !block_metadata || !num_blocks || !padded_offsets || !h || !y)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    return do_experts(*cfg, x_perm, W13, W2_t, block_metadata, num_blocks, padded_offsets, row_gate,
                      h, y, status, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_gemm_swiglu_permute(const moe_config_t* cfg, const void* x,
                                             const int32_t* row_src, void* x_perm,
                                             int32_t* visit_ready, const void* W13,
                                             const void* W2_t, const int32_t* block_metadata,
                                             const int32_t* num_blocks,
                                             const int32_t* padded_offsets, const float* row_gate,
                                             void* h, void* y, uint32_t* status, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (cfg->T == 0) return MOE_OK;
    if (!x || !row_src || !x_perm || !visit_ready || !W13 || !W2_t || !block_metadata ||
        !num_blocks || !padded_offsets || !h || !y)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(visit_ready, 0, static_cast<size_t>(sizes_of(*cfg).NB) * 4, st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing visit_ready");
    return do_experts(*cfg, x_perm, W13, W2_t, block_metadata, num_blocks, padded_offsets, row_gate,
                      h, y, status, st, x, row_src, nullptr, nullptr, nullptr, visit_ready);
}

moe_status_t moe_gather_rows(const void* src, const int32_t* idx, void* dst, int64_t n, int32_t d,
                             const float* src_gate, float* dst_gate, void* stream) {
    if (n < 0 || d <= 0) return fail(MOE_ERR_INVALID_ARG, "bad gather sizes");
    if (d % 8) return fail(MOE_ERR_UNSUPPORTED, "d = %d is not a multiple of 8", d);
    if ((src_gate == nullptr) != (dst_gate == nullptr))
        return fail(MOE_ERR_INVALID_ARG, "src_gate and dst_gate must both be given or both be NULL");
    if (n == 0) return MOE_OK;
    if (!src || !idx || !dst) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    cudaError_t e = launch_gather_rows(src, idx, dst, n, d, src_gate, dst_gate,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "gather rows");
}

moe_status_t moe_build_offsets_unpadded(const moe_config_t* cfg, const int32_t* topk_idx,
                                        const float* topk_w, int32_t* counts,
                                        int32_t* group_offsets, int32_t* perm_row,
                                        int32_t* row_src, float* row_gate, void* ws,
                                        size_t ws_bytes, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!topk_idx || !counts || !group_offsets || !perm_row || !row_src || !row_gate || !ws)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (ws_bytes < offsets_ws_bytes(*cfg))
        return fail(MOE_ERR_WORKSPACE, "offsets scratch of %zu bytes, %zu needed", ws_bytes,
                    offsets_ws_bytes(*cfg));
    if (cfg->T == 0) return MOE_OK;
    const int64_t A = static_cast<int64_t>(cfg->T) * cfg->k;
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    cudaError_t e = launch_offsets(topk_idx, topk_w, A, cfg->E, 1, A, counts, group_offsets, nullptr,
                                   nullptr, perm_row, row_src, row_gate,
                                   reinterpret_cast<uint32_t*>(w8),
                                   reinterpret_cast<int32_t*>(w8 + 256),
                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "offsets kernels (unpadded)");
}

moe_status_t moe_grouped_gemm_swiglu_unpadded(const moe_config_t* cfg, const void* x_perm,
                                              const void* W13, const void* W2_t,
                                              const int32_t* group_offsets, const float* row_gate,
                                              void* h, void* y, uint32_t* status, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!x_perm || !W13 || !W2_t || !group_offsets || !h || !y)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    return do_experts_unpadded(*cfg, x_perm, W13, W2_t, group_offsets, row_gate, h, y, status,
                               static_cast<cudaStream_t>(stream));
}

moe_status_t moe_build_blocks_from_counts(const int32_t* counts, int32_t n_src, int32_t E,
                                          int32_t P, int32_t* padded_offsets,
                                          int32_t* block_metadata, int32_t* num_blocks,
                                          int32_t nb_cap, int32_t* piece_row, uint32_t* status,
                                          void* stream) {
    if (n_src <= 0 || E <= 0 || nb_cap < 0) return fail(MOE_ERR_INVALID_ARG, "bad sizes");
    if (E > 256) return fail(MOE_ERR_UNSUPPORTED, "E = %d > 256", E);
    if (P != 64 && P != 128) return fail(MOE_ERR_UNSUPPORTED, "P = %d must be 64 or 128", P);
    if (!counts || !padded_offsets || !num_blocks || (nb_cap > 0 && !block_metadata))
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    cudaError_t e = launch_blocks_from_counts(counts, n_src, E, P, padded_offsets, block_metadata,
                                              num_blocks, nb_cap, piece_row, status,
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "blocks from counts");
}

moe_status_t moe_copy_pieces(const void* src, void* dst, int32_t d, const int32_t* src_row,
                             const int32_t* dst_row, const int32_t* rows, int32_t n,
                             int32_t max_rows, const float* src_gate, float* dst_gate,
                             void* stream) {
    if (n < 0 || d <= 0 || max_rows < 0) return fail(MOE_ERR_INVALID_ARG, "bad piece sizes");
    if (d % 8) return fail(MOE_ERR_UNSUPPORTED, "d = %d is not a multiple of 8", d);
    if (n > 65535) return fail(MOE_ERR_UNSUPPORTED, "n = %d pieces > 65535", n);
    if ((src_gate == nullptr) != (dst_gate == nullptr))
        return fail(MOE_ERR_INVALID_ARG, "src_gate and dst_gate must both be given or both be NULL");
    if (n == 0 || max_rows == 0) return MOE_OK;
    if (!src || !dst || !src_row || !dst_row || !rows) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    cudaError_t e = launch_copy_pieces(src, dst, d, src_row, dst_row, rows, n, max_rows, src_gate,
                                       dst_gate, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "copy pieces");
}

moe_status_t moe_widen_e4m3(const void* q, void* out, int64_t n, void* stream) {
    if (n < 0 || (n > 0 && (!q || !out))) return fail(MOE_ERR_INVALID_ARG, "bad widen args");
    if (n % 16) return fail(MOE_ERR_UNSUPPORTED, "n = %lld is not a multiple of 16",
                            static_cast<long long>(n));
    if (n == 0) return MOE_OK;
    cudaError_t e = launch_widen_e4m3(q, out, n, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "widen e4m3");
}

moe_status_t moe_grouped_gemm_swiglu_scaled(const moe_config_t* cfg, const void* x_perm,
                                            const void* W13, const float* s13, const void* W2_t,
                                            const float* s2, const int32_t* block_metadata,
                                            const int32_t* num_blocks, const int32_t* padded_offsets,
                                            const float* row_gate, void* h, void* y,
                                            uint32_t* status, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!x_perm || !W13 || !s13 || !W2_t || !s2 || !block_metadata || !num_blocks ||
        !padded_offsets || !h || !y)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    return do_experts(*cfg, x_perm, W13, W2_t, block_metadata, num_blocks, padded_offsets, row_gate,
                      h, y, status, static_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr, s13,
                      s2);
}

moe_status_t moe_shared_expert_scaled(const moe_config_t* cfg, const void* x, const void* Ws13,
                                      const float* ss13, const void* Ws2_t, const float* ss2,
                                      void* hs, void* ys, uint32_t* status, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (cfg->d_shared <= 0) return fail(MOE_ERR_INVALID_ARG, "d_shared must be > 0");
    if (!x || !Ws13 || !ss13 || !Ws2_t || !ss2 || !hs || !ys)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    return do_shared(*cfg, x, Ws13, Ws2_t, hs, ys, status, static_cast<cudaStream_t>(stream), nullptr,
                     ss13, ss2);
}

moe_status_t moe_permute_fp8(const moe_config_t* cfg, const void* x, const int32_t* perm_row,
                             void* x8, float* x_scale, void* xs8, float* xs_scale, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!x || !perm_row || !x8 || !x_scale) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if ((xs8 == nullptr) != (xs_scale == nullptr))
        return fail(MOE_ERR_INVALID_ARG, "xs8 and xs_scale must both be given or both be NULL");
    if (cfg->T == 0) return MOE_OK;
    cudaError_t e = launch_permute_fp8(x, perm_row, static_cast<uint8_t*>(x8), x_scale,
                                       static_cast<uint8_t*>(xs8), xs_scale, cfg->T, cfg->d, cfg->k,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "permute (e4m3 pairs)");
}

moe_status_t moe_grouped_gemm_swiglu_skinny(const moe_config_t* cfg, const void* x_perm,
                                            const void* W13, const void* W2_t,
                                            const int32_t* block_metadata,
                                            const int32_t* num_blocks, const float* row_gate,
                                            void* h, void* y, uint32_t* status, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!x_perm || !W13 || !W2_t || !block_metadata || !num_blocks || !h || !y)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    const SkinnyIO ro{x_perm, nullptr, W13, nullptr, W2_t, nullptr, h, nullptr, nullptr, y};
    return do_experts_skinny(*cfg, false, ro, block_metadata, num_blocks, row_gate, status,
                             static_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_gemm_swiglu_fp8(const moe_config_t* cfg, const void* x8,
                                         const float* x_scale, const void* W13q, const float* s13,
                                         const void* W2q, const float* s2,
                                         const int32_t* block_metadata, const int32_t* num_blocks,
                                         const float* row_gate, void* h, void* h8, float* h_scale,
                                         void* y, uint32_t* status, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!x8 || !x_scale || !W13q || !s13 || !W2q || !s2 || !block_metadata || !num_blocks || !h ||
        !h8 || !h_scale || !y)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    const SkinnyIO ro{x8, x_scale, W13q, s13, W2q, s2, h, static_cast<uint8_t*>(h8), h_scale, y};
    return do_experts_skinny(*cfg, true, ro, block_metadata, num_blocks, row_gate, status,
                             static_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_gemm_swiglu_gather(const moe_config_t* cfg, const void* x,
                                            const int32_t* row_src, const void* W13,
                                            const void* W2_t, const int32_t* block_metadata,
                                            const int32_t* num_blocks,
                                            const int32_t* padded_offsets, const float* row_gate,
                                            void* h, void* y, uint32_t* status, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!x || !row_src || !W13 || !W2_t || !block_metadata || !num_blocks || !padded_offsets ||
        !h || !y)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    return do_experts(*cfg, nullptr, W13, W2_t, block_metadata, num_blocks, padded_offsets,
                      row_gate, h, y, status, static_cast<cudaStream_t>(stream), x, row_src);
}

moe_status_t moe_shared_expert(const moe_config_t* cfg, const void* x, const void* Ws13,
                               const void* Ws2_t, void* hs, void* ys, uint32_t* status,
                               void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (cfg->d_shared <= 0) return fail(MOE_ERR_INVALID_ARG, "d_shared must be > 0");
    if (!x || !Ws13 || !Ws2_t || !hs || !ys) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    return do_shared(*cfg, x, Ws13, Ws2_t, hs, ys, status, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_shared_expert_up(const moe_config_t* cfg, const void* x, const void* Ws13,
                                  void* hs, const int32_t* perm_row, void* x_perm,
                                  uint32_t* status, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (cfg->d_shared <= 0) return fail(MOE_ERR_INVALID_ARG, "d_shared must be > 0");
    if (!x_perm != !perm_row) return fail(MOE_ERR_INVALID_ARG, "perm_row and x_perm: both or neither");
    if (cfg->T == 0) return MOE_OK;
    if (!x || !Ws13 || !hs) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    const FusedPermute fp{perm_row, x_perm};
    return do_shared_up(*cfg, x, Ws13, hs, status, static_cast<cudaStream_t>(stream), nullptr,
                        nullptr, &fp);
}

moe_status_t moe_shared_expert_down(const moe_config_t* cfg, const void* hs, const void* Ws2_t,
                                    void* ys, uint32_t* status, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (cfg->d_shared <= 0) return fail(MOE_ERR_INVALID_ARG, "d_shared must be > 0");
    if (cfg->T == 0) return MOE_OK;
    if (!hs || !Ws2_t || !ys) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    return do_shared_down(*cfg, hs, Ws2_t, ys, status, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_shared_expert_down_combine(const moe_config_t* cfg, const void* hs,
                                            const void* Ws2_t, const void* y,
                                            const int32_t* perm_row, void* out, uint32_t* status,
                                            void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (cfg->d_shared <= 0) return fail(MOE_ERR_INVALID_ARG, "d_shared must be > 0");
    if (cfg->T == 0) return MOE_OK;
    if (!hs || !Ws2_t || !y || !perm_row || !out) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    const FusedCombine fc{y, perm_row, out};
    return do_shared_down(*cfg, hs, Ws2_t, nullptr, status, static_cast<cudaStream_t>(stream),
                          nullptr, &fc);
}

moe_status_t moe_shared_expert_fp8(const moe_config_t* cfg, const void* xs8, const float* xs_scale,
                                   const void* Ws13q, const float* ss13, const void* Ws2q,
                                   const float* ss2, void* hs, void* hs8, float* hs_scale, void* ys,
                                   uint32_t* status, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (cfg->d_shared <= 0) return fail(MOE_ERR_INVALID_ARG, "d_shared must be > 0");
    if (!xs8 || !xs_scale || !Ws13q || !ss13 || !Ws2q || !ss2 || !hs || !hs8 || !hs_scale || !ys)
        return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    // no block table: a launch of the shared expert's dense tiles only
    const SkinnyIO none{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                        nullptr, nullptr};
    const SkinnyIO so{xs8, xs_scale, Ws13q, ss13, Ws2q, ss2, hs, static_cast<uint8_t*>(hs8), hs_scale,
                      ys};
    return do_experts_skinny(*cfg, true, none, nullptr, nullptr, nullptr, status,
                             static_cast<cudaStream_t>(stream), &so);
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* y, const int32_t* perm_row,
                         const void* shared_out, void* out, void* stream) {
    moe_status_t r = check_cfg(cfg, false);
    if (r != MOE_OK) return r;
    if (!y || !perm_row || !out) return fail(MOE_ERR_INVALID_ARG, "null pointer");
    if (cfg->T == 0) return MOE_OK;
    cudaError_t e = launch_combine(y, perm_row, shared_out, out, cfg->T, cfg->d, cfg->k,
                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine");
}

moe_status_t moe_layer_fwd(const moe_config_t* cfg, const moe_weights_t* w, const void* x,
                           void* out, void* ws, size_t ws_bytes, void* stream) {
    return layer(cfg, w, x, nullptr, nullptr, out, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_layer_fwd_prerouted(const moe_config_t* cfg, const moe_weights_t* w,
                                     const void* x, const int32_t* topk_idx, const float* topk_w,
                                     void* out, void* ws, size_t ws_bytes, void* stream) {
    if (!topk_idx) return fail(MOE_ERR_INVALID_ARG, "null pre-routed indices");
    return layer(cfg, w, x, topk_idx, topk_w, out, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

size_t moe_gate_up_save_size(const moe_config_t* cfg) {
    if (check_cfg(cfg, false) != MOE_OK) return 0;
    return gate_up_save_bytes(*cfg);
}

moe_status_t moe_layer_fwd_save(const moe_config_t* cfg, const moe_weights_t* w, const void* x,
                                const int32_t* topk_idx, const float* topk_w, void* out, void* ws,
                                size_t ws_bytes, void* gu_save, size_t gu_save_bytes, void* stream) {
    moe_status_t r = check_cfg(cfg, topk_idx == nullptr);
    if (r != MOE_OK) return r;
    if (cfg->T > 0 && (!gu_save || gu_save_bytes < gate_up_save_bytes(*cfg)))
        return fail(MOE_ERR_WORKSPACE, "gate/up save of %zu bytes, %zu needed", gu_save_bytes,
                    gate_up_save_bytes(*cfg));
    return layer(cfg, w, x, topk_idx, topk_w, out, ws, ws_bytes, static_cast<cudaStream_t>(stream),
                 gu_save);
}

moe_status_t moe_layer_fwd_fp8(const moe_config_t* cfg, const moe_weights_fp8_t* w, const void* x,
                               void* out, void* ws, size_t ws_bytes, void* stream) {
    return layer_fp8(cfg, w, x, nullptr, nullptr, out, ws, ws_bytes,
                     static_cast<cudaStream_t>(stream));
}

moe_status_t moe_layer_fwd_fp8_prerouted(const moe_config_t* cfg, const moe_weights_fp8_t* w,
                                         const void* x, const int32_t* topk_idx,
                                         const float* topk_w, void* out, void* ws,
                                         size_t ws_bytes, void* stream) {
    if (!topk_idx) return fail(MOE_ERR_INVALID_ARG, "null pre-routed indices");
    return layer_fp8(cfg, w, x, topk_idx, topk_w, out, ws, ws_bytes,
                     static_cast<cudaStream_t>(stream));
}

moe_status_t moe_pack_experts_bwd(int32_t E, int32_t d, int32_t de, const void* W1, const void* W3,
                                  void* W13t, void* stream) {
    if (E <= 0 || d <= 0 || de <= 0 || !W1 || !W3 || !W13t)
        return fail(MOE_ERR_INVALID_ARG, "bad backward expert pack args");
    if (d % 128 || de % 128) return fail(MOE_ERR_UNSUPPORTED, "d and de must be multiples of 128");
    cudaError_t e = launch_interleave(const_cast<void*>(W1), const_cast<void*>(W3), W13t,
                                      static_cast<int64_t>(E) * d, de, 0,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "pack experts (backward)");
}

moe_status_t moe_pack_router_bwd(int32_t d, int32_t E, const void* Wg, void* WgP, void* stream) {
    if (d <= 0 || E <= 0 || !Wg || !WgP) return fail(MOE_ERR_INVALID_ARG, "bad router pack args");
    const size_t ep = static_cast<size_t>((E + 127) / 128 * 128);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemset2DAsync(WgP, ep * 2, 0, ep * 2, d, st);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(WgP, ep * 2, Wg, static_cast<size_t>(E) * 2, static_cast<size_t>(E) * 2, d,
                              cudaMemcpyDeviceToDevice, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "pack router (backward)");
}

size_t moe_backward_workspace_size(const moe_config_t* cfg) {
    if (check_cfg(cfg, false) != MOE_OK) return 0;
    return bwd_layout_of(*cfg).total;
}

moe_status_t moe_layer_bwd(const moe_config_t* cfg, const moe_weights_t* w,
                           const moe_weights_bwd_t* wb, const void* x, const void* dout,
                           const void* fwd_ws, size_t fwd_ws_bytes, const void* gu_saved,
                           size_t gu_saved_bytes, const moe_grads_t* grads, void* bws,
                           size_t bws_bytes, void* stream) {
    return layer_bwd(cfg, w, wb, x, dout, fwd_ws, fwd_ws_bytes, gu_saved, gu_saved_bytes, grads, bws,
                     bws_bytes, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_get_device_status(void* ws, uint32_t* bits, void* stream) {
    if (!ws) return fail(MOE_ERR_INVALID_ARG, "ws is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && v) e = cudaMemsetAsync(ws, 0, sizeof v, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    if (bits) *bits = v;
    return v ? fail(MOE_ERR_DEVICE_CHECK, "device status bits 0x%x", v) : MOE_OK;
}

moe_status_t moe_selftest_wait_timeout(uint64_t limit_ns, uint32_t* status, void* stream) {
    if (!status || limit_ns == 0 || limit_ns > 10000000000ull)
        return fail(MOE_ERR_INVALID_ARG, "status must be non-null and 0 < limit_ns <= 10 s");
    cudaError_t e = launch_wait_selftest(limit_ns, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "wait self-test");
}

const char* moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_CHECK: return "device-side check failed";
        default: return "unknown status";
    }
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
