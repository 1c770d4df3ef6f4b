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

#include "internal.h"

// The fixed scratch.  Every GPU that loads the library holds these bytes
// until the process exits.  In host code this name is only a stand-in for
// the symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_dispatch_scratch[MOE_DISPATCH_NOALLOC_SCRATCH_BYTES];

namespace moe {
namespace {

constexpr size_t kScratchBytes = MOE_DISPATCH_NOALLOC_SCRATCH_BYTES;

std::mutex g_mu;
void* g_scratch_ptr[128];   // device address of g_dispatch_scratch, per device

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return MOE_ECUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) return MOE_ECUDA;
        g_scratch_ptr[dev] = p;
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
                               expert_rows, expert_count, stats, stream);
}
