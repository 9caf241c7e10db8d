// offsets_noalloc.cu -- an allocation-free variant of moe_build_offsets.
//
// moe_build_offsets needs a small device scratch (per-chunk expert counts)
// that its caller allocates.  Some callers cannot allocate device memory at
// the point where they run this stage, for one runtimes that hand out memory
// only from a pool reserved at start-up and forbid any allocation on the
// serving path.  This variant keeps its
// scratch in a fixed-size array in the library's own device memory instead,
// so the caller passes inputs and outputs only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {

// The per-chunk counts of the offsets kernels (int32 [chunks, E]).  Every
// GPU that loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = 64 * 1024;
static __device__ __align__(256) unsigned char g_offsets_scratch[kNoAllocScratchBytes];

// Device address of g_offsets_scratch in the current context.  In host code
// the symbol name is only a host-side stand-in, so the address is looked up
// with the device current and cached per device together with the context it
// was found in: after cudaDeviceReset (or any teardown of the primary
// context) the module is loaded again, possibly at another address, so a
// call in a new context looks the address up afresh.
typedef CUresult (*PFN_ctxGetCurrent)(CUcontext*);

static PFN_ctxGetCurrent ctx_get_current() {
    static PFN_ctxGetCurrent fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_ctxGetCurrent>(p);
    });
    return fn;
}

static void* noalloc_scratch(int dev, cudaError_t* err) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    static CUcontext ctx_of[kMaxDevices] = {};
    std::lock_guard<std::mutex> lock(mu);
    *err = cudaSuccess;
    PFN_ctxGetCurrent get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    if (addr[dev] && ctx && ctx == ctx_of[dev]) return addr[dev];
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_offsets_scratch);  // sets the context up if needed
    if (*err != cudaSuccess) return nullptr;
    ctx = nullptr;
    if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    addr[dev] = p;
    ctx_of[dev] = ctx;
    return p;
}

#define set_last_error(status, ...) static_cast<moe_status_t>(record_error(status, __VA_ARGS__))

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_build_offsets_noalloc(const moe_config_t* cfg, const int32_t* topk_idx,
                                                  const float* topk_w, int32_t* counts,
                                                  int32_t* padded_offsets, int32_t* block_metadata,
                                                  int32_t* num_blocks, int32_t* perm_row,
                                                  int32_t* row_src, float* row_gate,
                                                  uint32_t* status, void* stream) {
    moe_status_t r = moe_check_config(cfg);
    if (r != MOE_OK) return r;
    if (!topk_idx || !counts || !padded_offsets || !block_metadata || !num_blocks || !perm_row ||
        !row_src || !row_gate)
        return set_last_error(MOE_ERR_INVALID_ARG, "null pointer");
    const int64_t A = static_cast<int64_t>(cfg->T) * cfg->k;
    const size_t need = static_cast<size_t>(offsets_num_chunks(A)) * cfg->E * 4;
    if (need > kNoAllocScratchBytes)
        return set_last_error(MOE_ERR_WORKSPACE,
                              "allocation-free offsets need %zu bytes of scratch; the static "
                              "scratch holds %zu (T*k <= %lld at this E)",
                              need, kNoAllocScratchBytes,
                              static_cast<long long>(kNoAllocScratchBytes / 4 / cfg->E) * 2048);
    if (cfg->T == 0) return MOE_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_last_error(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return set_last_error(MOE_ERR_UNSUPPORTED, "device index %d >= %d", dev, kMaxDevices);
    void* scratch = noalloc_scratch(dev, &e);
    if (!scratch)
        return set_last_error(MOE_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    // Nothing in the scratch has to start at zero: the histogram pass writes
    // every [chunk, expert] count before the scan and the scatter read them.
    const int64_t R = A + static_cast<int64_t>(cfg->E) * (cfg->pad_multiple - 1);
    e = launch_offsets(topk_idx, topk_w, A, cfg->E, cfg->pad_multiple, R, counts, padded_offsets,
                       block_metadata, num_blocks, perm_row, row_src, row_gate, status,
                       static_cast<int32_t*>(scratch), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return set_last_error(MOE_ERR_CUDA, "offsets kernels: %s", cudaGetErrorString(e));
    return MOE_OK;
}
