// dispatch_noalloc.cu -- the pooled dispatch for callers that cannot allocate
// device memory.
//
// moe_dispatch_pooled needs a few MB of scratch (per-assignment slots and
// ranks, per-source expert counts and their prefix sums), which the caller
// normally allocates.  Some callers cannot: a host application that reserved
// the device's memory up front and forbids allocations afterwards, code on a
// latency-critical path where cudaMalloc's implicit device synchronisation is
// not acceptable, or a plug-in that receives tensors but no allocator.  For
// them this file keeps the scratch in a fixed device array that exists for
// as long as the library is loaded, and forwards to moe_dispatch_pooled.
#include <mutex>

#include <cuda.h>

#include "internal.h"

// The fixed scratch.  Every GPU that loads the library holds these bytes
// until the process exits.  In host code this name is only a stand-in for
// the symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_dispatch_scratch[MOE_DISPATCH_NOALLOC_SCRATCH_BYTES];

namespace moe {
namespace {

constexpr size_t kScratchBytes = MOE_DISPATCH_NOALLOC_SCRATCH_BYTES;

std::mutex g_mu;
void* g_scratch_ptr[128];                 // device address of g_dispatch_scratch, per device
unsigned long long g_scratch_ctx[128];    // id of the context that address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <class F>
F driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(f);
}

// Id of this thread's current CUDA context (unique within the process and
// never reused, so a context made after cudaDeviceReset gets a new one);
// 0 when there is no current context or the id cannot be read.
unsigned long long current_context_id() {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id) return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of the scratch on the current device.  Looked up with that
// device current the first time a context of the device calls here, and
// cached with the context's id; a later context of the same device (after a
// device reset) looks it up again.  Without a readable context id nothing is
// cached.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return MOE_ECUDA;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_mu);
    if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) return MOE_ECUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_dispatch_pooled_noalloc(const moe_config_t* cfg, const uint16_t* z,
                                           const int32_t* idx, uint16_t* pool, int32_t* slot_of,
                                           uint8_t* drop, int32_t* expert_rows,
                                           int32_t* expert_count, moe_drop_stats_t* stats,
                                           void* stream) {
    moe_plan_t plan;
    int rc = moe_plan(cfg, &plan);
    if (rc) return rc;
    if (static_cast<size_t>(plan.ws_dispatch_bytes) > moe::kScratchBytes) return MOE_ENOSPC;
    void* ws = nullptr;
    if ((rc = moe::scratch_address(&ws))) return rc;
    // Nothing in the scratch has to start at zero: within one call every word
    // the kernels read was written earlier in the same call.
    return moe_dispatch_pooled(cfg, z, idx, ws, moe::kScratchBytes, pool, slot_of, drop,
                               expert_rows, expert_count, stats, nullptr, stream);
}
