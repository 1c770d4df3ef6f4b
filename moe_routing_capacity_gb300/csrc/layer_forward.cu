// layer_forward.cu -- the whole layer forward in one call, and a pipeline
// that feeds it from host memory.
//
// moe_layer_forward enqueues the layer's calls in order on one stream:
// router top-k with the latent projection (one pass over x), the pooled
// dispatch with the pool fill inside the shared experts' gate/up launch
// (or the plain dispatch when there are no shared experts), the grouped
// experts, and the combine with the up-projection and the shared
// down-projection.  Host code only: every step runs in the library's kernels.
//
// moe_host_pipe_* keep `depth` device staging buffers (the caller's) in a
// ring and two copy streams of their own: batch i's x is copied host ->
// device while batch i-1 computes and batch i-2's output copies back, the
// three ordered by events, as a serving loop would run it.
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"

namespace {

struct NvtxScope {
    explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
    ~NvtxScope() { nvtxRangePop(); }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

struct moe_host_pipe {
    moe_config_t cfg;
    int depth;
    int device;
    int64_t submitted;
    size_t x_bytes, out_bytes;
    std::vector<uint16_t*> xd, od;
    std::vector<moe_drop_stats_t*> sd;
    cudaStream_t h2d, d2h;
    std::vector<cudaEvent_t> ev_in;     // x of the slot has landed
    std::vector<cudaEvent_t> ev_done;   // the forward of the slot read x and wrote out
    std::vector<cudaEvent_t> ev_out;    // out of the slot has been copied back
};

namespace {

void destroy_pipe(moe_host_pipe* p) {
    if (!p) return;
    if (p->h2d) cudaStreamDestroy(p->h2d);
    if (p->d2h) cudaStreamDestroy(p->d2h);
    for (auto* v : {&p->ev_in, &p->ev_done, &p->ev_out})
        for (cudaEvent_t e : *v)
            if (e) cudaEventDestroy(e);
    delete p;
}

}  // namespace

extern "C" {

int moe_layer_forward(const moe_config_t* cfg, const moe_layer_buffers_t* b, const uint16_t* x,
                      uint16_t* out, void* stream) {
    NvtxScope range(__func__);
    if (!cfg || !b) return MOE_EINVAL;
    int rc;
    if ((rc = moe_route_project(cfg, x, b->Wr, b->bias, b->W_ld, b->logits, b->idx, b->w, b->tie,
                                b->z, b->status, stream)))
        return rc;
    const bool shared = cfg->n_shared > 0;
    if (shared)
        rc = moe_dispatch_shared_overlap(cfg, b->z, b->idx, b->ws_dispatch, b->ws_dispatch_bytes,
                                         b->pool, b->slot_of, b->drop, b->expert_rows,
                                         b->expert_count, b->stats, b->bank, x, b->Wsg, b->Wsu,
                                         b->a, b->status, stream);
    else
        rc = moe_dispatch_pooled(cfg, b->z, b->idx, b->ws_dispatch, b->ws_dispatch_bytes, b->pool,
                                 b->slot_of, b->drop, b->expert_rows, b->expert_count, b->stats,
                                 b->bank, stream);
    if (rc) return rc;
    if ((rc = moe_expert_ffn_grouped(cfg, b->pool, b->bank, b->expert_rows, b->expert_count, b->Wg,
                                     b->Wu, b->Wd, b->ws_ffn, b->ws_ffn_bytes, b->ypool, b->status,
                                     stream)))
        return rc;
    // with shared experts their activations a were computed beside the dispatch
    return moe_combine(cfg, b->ypool, b->slot_of, b->w, b->W_lu, shared ? nullptr : x, nullptr,
                       nullptr, shared ? b->Wsd : nullptr, b->c, shared ? b->a : nullptr, out,
                       b->status, stream);
}

int moe_host_pipe_create(const moe_config_t* cfg, int depth, uint16_t* const* x_dev,
                         uint16_t* const* out_dev, moe_drop_stats_t* const* stats_dev,
                         moe_host_pipe_t** pipe) {
    if (!cfg || !pipe || depth < 1 || depth > 16 || !x_dev || !out_dev || !stats_dev)
        return MOE_EINVAL;
    *pipe = nullptr;
    moe_plan_t plan;
    int rc = moe_plan(cfg, &plan);
    if (rc) return rc;
    if (cfg->T > 0 && cfg->d_model <= 0) return MOE_EINVAL;
    for (int i = 0; i < depth; ++i)
        if (!x_dev[i] || !out_dev[i] || !stats_dev[i] || !aligned16(x_dev[i]) ||
            !aligned16(out_dev[i]) || (reinterpret_cast<uintptr_t>(stats_dev[i]) & 7))
            return MOE_EINVAL;
    moe_host_pipe* p = new (std::nothrow) moe_host_pipe();
    if (!p) return MOE_ENOSPC;
    p->cfg = *cfg;
    p->depth = depth;
    p->submitted = 0;
    p->x_bytes = static_cast<size_t>(cfg->T) * cfg->d_model * 2;
    p->out_bytes = p->x_bytes;
    p->h2d = p->d2h = nullptr;
    p->xd.assign(x_dev, x_dev + depth);
    p->od.assign(out_dev, out_dev + depth);
    p->sd.assign(stats_dev, stats_dev + depth);
    p->ev_in.assign(depth, nullptr);
    p->ev_done.assign(depth, nullptr);
    p->ev_out.assign(depth, nullptr);
    bool ok = cudaGetDevice(&p->device) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < depth; ++i)
        ok = cudaEventCreateWithFlags(&p->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->ev_done[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->ev_out[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        destroy_pipe(p);
        return MOE_ECUDA;
    }
    *pipe = p;
    return MOE_OK;
}

int moe_host_pipe_submit(moe_host_pipe_t* p, const moe_layer_buffers_t* b, const uint16_t* x_host,
                         uint16_t* out_host, moe_drop_stats_t* stats_host, void* stream) {
    NvtxScope range(__func__);
    if (!p || !b || (p->x_bytes && (!x_host || !out_host))) return MOE_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device) return MOE_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int s = static_cast<int>(p->submitted % p->depth);
    const bool reuse = p->submitted >= p->depth;
    // x of the slot: free once the forward that last read it has run
    if (reuse && cudaStreamWaitEvent(p->h2d, p->ev_done[s], 0) != cudaSuccess) return MOE_ECUDA;
    if (p->x_bytes &&
        cudaMemcpyAsync(p->xd[s], x_host, p->x_bytes, cudaMemcpyHostToDevice, p->h2d) != cudaSuccess)
        return MOE_ECUDA;
    if (cudaEventRecord(p->ev_in[s], p->h2d) != cudaSuccess ||
        cudaStreamWaitEvent(st, p->ev_in[s], 0) != cudaSuccess)
        return MOE_ECUDA;
    // out of the slot: free once its previous contents were copied back
    if (reuse && cudaStreamWaitEvent(st, p->ev_out[s], 0) != cudaSuccess) return MOE_ECUDA;
    int rc = moe_layer_forward(&p->cfg, b, p->xd[s], p->od[s], stream);
    if (rc) return rc;
    // the batch's drop statistics, kept per slot (the next forward rewrites b->stats)
    if (b->stats && cudaMemcpyAsync(p->sd[s], b->stats, sizeof(moe_drop_stats_t),
                                    cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return MOE_ECUDA;
    if (cudaEventRecord(p->ev_done[s], st) != cudaSuccess ||
        cudaStreamWaitEvent(p->d2h, p->ev_done[s], 0) != cudaSuccess)
        return MOE_ECUDA;
    if (p->out_bytes &&
        cudaMemcpyAsync(out_host, p->od[s], p->out_bytes, cudaMemcpyDeviceToHost, p->d2h) !=
            cudaSuccess)
        return MOE_ECUDA;
    if (stats_host && cudaMemcpyAsync(stats_host, p->sd[s], sizeof(moe_drop_stats_t),
                                      cudaMemcpyDeviceToHost, p->d2h) != cudaSuccess)
        return MOE_ECUDA;
    if (cudaEventRecord(p->ev_out[s], p->d2h) != cudaSuccess) return MOE_ECUDA;
    ++p->submitted;
    return MOE_OK;
}

int moe_host_pipe_sync(moe_host_pipe_t* p) {
    if (!p) return MOE_EINVAL;
    if (cudaStreamSynchronize(p->h2d) != cudaSuccess || cudaStreamSynchronize(p->d2h) != cudaSuccess)
        return MOE_ECUDA;
    return MOE_OK;
}

int moe_host_pipe_destroy(moe_host_pipe_t* p) {
    if (!p) return MOE_OK;
    const int rc = moe_host_pipe_sync(p);
    destroy_pipe(p);
    return rc;
}

}  // extern "C"
