// abi.cu -- the library's C entry points: argument checks, the plan
// (capacities, pool and scratch sizes), and the launch sequence of each step.
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"

namespace {
// One NVTX range per C-ABI compute call (a no-op unless a profiler attaches),
// so that profiler timelines group each call's kernels under its name.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace
#define MOE_NVTX_RANGE() NvtxRange moe_nvtx_range_(__func__)

namespace moe {

int current_device(int* device, int* num_sms) {
    static std::mutex mu;
    static int cached_sms[128];
    static int cached_ok[128];   // 0 unknown, 1 sm_103, -1 other
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return MOE_ECUDA;
    std::lock_guard<std::mutex> lk(mu);
    if (cached_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ECUDA;
        cached_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        cached_sms[dev] = sms;
    }
    if (cached_ok[dev] != 1) return MOE_ENODEV;
    *device = dev;
    *num_sms = cached_sms[dev];
    return MOE_OK;
}

int ensure_smem_attr(const void* func, int bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> done;   // (kernel, device) -> limit set
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ECUDA;
    std::lock_guard<std::mutex> lk(mu);
    int& have = done[std::make_pair(func, dev)];
    if (have >= bytes) return MOE_OK;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return MOE_ECUDA;
    have = bytes;
    return MOE_OK;
}

// ---------------------------------------------------------------- timing trace

namespace {
std::mutex trace_mu;
cudaEvent_t* trace_ev = nullptr;
const char** trace_names = nullptr;
int trace_cap = 0;
int trace_n = 0;
bool trace_on = false;

void trace_free() {
    for (int i = 0; i < trace_cap; ++i) cudaEventDestroy(trace_ev[i]);
    delete[] trace_ev;
    delete[] trace_names;
    trace_ev = nullptr;
    trace_names = nullptr;
    trace_cap = trace_n = 0;
}
}  // namespace

void trace_after(cudaStream_t st, const char* name) {
    std::lock_guard<std::mutex> lk(trace_mu);
    if (!trace_on || trace_n >= trace_cap) return;
    if (cudaEventRecord(trace_ev[trace_n], st) != cudaSuccess) return;
    trace_names[trace_n++] = name;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Capacity = smallest integer >= cf * num / den with cf read to six decimals,
// clamped to [0, most]; a factor >= 1e6 (or infinite) means no cap.
static int64_t capacity(double cf, int64_t num, int64_t den, int64_t most) {
    if (std::isinf(cf) || cf >= 1e6) return most;
    const long long scale = std::llround(cf * 1e6);
    if (den == 0) return 0;
    const __int128 n = static_cast<__int128>(scale) * num;
    const __int128 d = static_cast<__int128>(1000000) * den;
    __int128 c = (n + d - 1) / d;
    if (c > most) c = most;
    if (c < 0) c = 0;
    return static_cast<int64_t>(c);
}

struct Geom {
    DispatchGeom g;
    int d, H, Hs, ns;
    moe_plan_t plan;
};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static int make_geom(const moe_config_t* c, Geom* out) {
    if (!c || !out) return MOE_EINVAL;
    if (c->T < 0 || c->d_model <= 0 || c->d_latent <= 0 || c->n_experts <= 0 || c->n_ranks <= 0 ||
        c->top_k <= 0 || c->n_waves <= 0 || c->n_shared < 0 || c->n_shared > 3 ||
        c->h_expert <= 0 || (c->n_shared > 0 && c->h_shared <= 0) || c->reserved != 0)
        return MOE_EINVAL;
    if (c->d_model % 8 || c->d_latent % 8 || c->h_expert % 8 || (c->n_shared && c->h_shared % 8))
        return MOE_EINVAL;
    if (c->top_k > 32 || c->top_k > c->n_experts || c->n_experts > 1024) return MOE_EINVAL;
    if (c->T % c->n_ranks || c->n_experts % c->n_ranks ||
        (c->n_experts / c->n_ranks) % c->n_waves)
        return MOE_EINVAL;
    if (!(c->cf_send > 0) || !(c->cf_recv > 0)) return MOE_EINVAL;   // also rejects NaN
    if (c->T > (1ll << 31) / c->top_k) return MOE_EINVAL;

    DispatchGeom& g = out->g;
    g.ragged = 0;
    g.T = c->T;
    g.k = c->top_k;
    g.E = c->n_experts;
    g.S = g.D = c->n_ranks;
    g.W = c->n_waves;
    g.E_l = g.E / g.D;
    g.E_w = g.E_l / g.W;
    g.L = c->d_latent;
    g.T_s = g.T / g.S;
    const int64_t most_send = g.T_s * std::min<int64_t>(g.k, g.E_w);
    const int64_t cs = capacity(c->cf_send, g.T_s * g.k, static_cast<int64_t>(g.D) * g.W, most_send);
    const int64_t cr = capacity(c->cf_recv, g.T * g.k, g.E, g.T);
    const int64_t pool_rows = static_cast<int64_t>(g.D) * g.W * g.S * cs;
    if (pool_rows > INT32_MAX || cr > INT32_MAX) return MOE_EINVAL;
    g.c_send = static_cast<int>(cs);
    g.c_recv = static_cast<int>(cr);
    g.pool_rows = pool_rows;
    out->d = c->d_model;
    out->H = c->h_expert;
    out->Hs = c->h_shared;
    out->ns = c->n_shared;

    moe_plan_t& p = out->plan;
    std::memset(&p, 0, sizeof(p));
    p.tokens_per_rank = g.T_s;
    p.experts_per_rank = g.E_l;
    p.experts_per_wave = g.E_w;
    p.c_send = g.c_send;
    p.c_recv = g.c_recv;
    p.pool_rows = g.pool_rows;
    p.pool_row_bytes = 2 * pool_pitch(g.L);
    p.ws_dispatch_bytes = static_cast<int64_t>(dispatch_ws_layout(g).total);
    const size_t max_mt = static_cast<size_t>(g.E) * ((g.c_recv + 127) / 128);
    // the tile list of the gathered path or the chunk list of the bank path
    const size_t tiles_bytes =
        align_up(std::max(max_mt * 8 + 16, expert_pair_chunks_bytes(g.E, g.c_recv)), 1024);
    p.h_offset_bytes = static_cast<int64_t>(tiles_bytes);
    p.ws_ffn_bytes = static_cast<int64_t>(tiles_bytes + static_cast<size_t>(g.E) * g.c_recv * out->H * 2);
    return MOE_OK;
}

// The dropless ragged layout: no caps, a pool of exactly T*k rows, h stored
// flat with each expert's rows at its offset.
static int make_geom_ragged(const moe_config_t* c, Geom* out) {
    int rc = make_geom(c, out);
    if (rc) return rc;
    DispatchGeom& g = out->g;
    const int64_t n = g.T * g.k;
    if (n > INT32_MAX / 2) return MOE_EINVAL;
    g.ragged = 1;
    g.c_send = INT32_MAX;   // never binds
    g.c_recv = INT32_MAX;
    g.pool_rows = n;
    moe_plan_t& p = out->plan;
    p.c_send = 0;
    p.c_recv = 0;
    p.pool_rows = n;
    p.ws_dispatch_bytes = static_cast<int64_t>(dispatch_ws_layout(g).total);
    const size_t max_mt = static_cast<size_t>(n / 128 + g.E);
    // the tile list of the gathered path or the group lists of the bank path
    const size_t tiles_bytes =
        align_up(std::max(max_mt * 8 + 16, expert_pair_lists_bytes_ragged(g.E, n)), 1024);
    p.h_offset_bytes = static_cast<int64_t>(tiles_bytes);
    p.ws_ffn_bytes = static_cast<int64_t>(tiles_bytes + static_cast<size_t>(n) * out->H * 2);
    return MOE_OK;
}

// The row-group expert kernels take these widths (else the gathered GEMMs).
static bool pair_path_fits(const Geom& G) { return G.g.L % 256 == 0 && G.H % 128 == 0; }

}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return 6; }

int moe_check_status(void) {
    const int v[4] = {check_status_route(), check_status_gemm(), check_status_backward(),
                      check_status_expert_pair()};
    for (int x : v)
        if (x) return x;
    return 0;
}

#if MOE_CHECK
int moe_check_set_wave_wait_limit_ns(unsigned long long ns) {
    const int rc = moe::set_wave_wait_limit(ns);
    return rc;
}
#endif

int moe_trace_begin(int capacity) {
    std::lock_guard<std::mutex> lk(trace_mu);
    if (capacity < 0) return MOE_EINVAL;
    if (capacity != trace_cap) {
        trace_free();
        if (capacity > 0) {
            trace_ev = new cudaEvent_t[capacity];
            trace_names = new const char*[capacity];
            for (int i = 0; i < capacity; ++i)
                if (cudaEventCreate(&trace_ev[i]) != cudaSuccess) {
                    trace_cap = i;
                    trace_free();
                    return MOE_ECUDA;
                }
            trace_cap = capacity;
        }
    }
    trace_n = 0;
    trace_on = capacity > 0;
    return MOE_OK;
}

int moe_trace_mark(void* stream) {
    trace_after(static_cast<cudaStream_t>(stream), "mark");
    return MOE_OK;
}

int moe_trace_end(void) {
    std::lock_guard<std::mutex> lk(trace_mu);
    trace_on = false;
    return trace_n;
}

int moe_trace_event(int i, const char** name, float* ms_since_prev) {
    std::lock_guard<std::mutex> lk(trace_mu);
    if (i < 0 || i >= trace_n || !name || !ms_since_prev) return MOE_EINVAL;
    *name = trace_names[i];
    *ms_since_prev = 0.0f;
    if (cudaEventSynchronize(trace_ev[i]) != cudaSuccess) return MOE_ECUDA;
    if (i > 0 && cudaEventElapsedTime(ms_since_prev, trace_ev[i - 1], trace_ev[i]) != cudaSuccess)
        return MOE_ECUDA;
    return MOE_OK;
}

const char* moe_strerror(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_EINVAL: return "invalid argument (sizes, divisibility, alignment or null pointer)";
        case MOE_ENOSPC: return "scratch buffer smaller than moe_plan requires";
        case MOE_ECUDA: return "CUDA runtime or driver call failed";
        case MOE_ETIMEOUT: return "device-side wait timed out";
        case MOE_ENODEV: return "current device is not an sm_103 (GB300) GPU";
        default: return "unknown error";
    }
}

int moe_plan(const moe_config_t* cfg, moe_plan_t* plan) {
    if (!plan) return MOE_EINVAL;
    Geom G;
    const int rc = make_geom(cfg, &G);
    if (rc) return rc;
    *plan = G.plan;
    return MOE_OK;
}

int moe_router_topk(const moe_config_t* cfg, const uint16_t* x, const uint16_t* Wr,
                    const float* bias, float* logits, int32_t* idx, float* w, uint8_t* tie,
                    int32_t* status, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom(cfg, &G);
    if (rc) return rc;
    if (G.g.T == 0) return MOE_OK;
    if (!x || !Wr || !logits || !idx || !w || !tie || !status) return MOE_EINVAL;
    if (!aligned16(x) || !aligned16(Wr)) return MOE_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    GemmDesc d;
    std::memset(&d, 0, sizeof(d));
    d.a_mode = A_DENSE;
    d.M = G.g.T;
    d.N = G.g.E;
    d.nseg = 1;
    d.seg[0] = GemmSeg{x, G.d, Wr, G.d, G.d};
    d.b_rows = G.g.E;
    d.out = logits;
    d.ldo = G.g.E;
    d.bias = bias;
    d.status = status;
    d.epi = EPI_F32;
    // E <= 384: one 128 x 384 tile per 128 tokens (a single wave of CTAs at
    // the workloads' sizes); wider routers use 128 x 128 tiles
    d.bn = G.g.E <= 384 ? 384 : 128;
    d.name = "gemm_router";
    if ((rc = gemm_launch(d, st))) return rc;
    return launch_topk(logits, G.g.T, G.g.E, G.g.k, idx, w, tie, st);
}

int moe_route_project(const moe_config_t* cfg, const uint16_t* x, const uint16_t* Wr,
                      const float* bias, const uint16_t* W_ld, float* logits, int32_t* idx,
                      float* w, uint8_t* tie, uint16_t* z, int32_t* status, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom(cfg, &G);
    if (rc) return rc;
    if (G.g.T == 0) return MOE_OK;
    if (!x || !Wr || !W_ld || !logits || !idx || !w || !tie || !z || !status) return MOE_EINVAL;
    if (!aligned16(x) || !aligned16(Wr) || !aligned16(W_ld) || !aligned16(z)) return MOE_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (G.g.L % 256) {   // no whole latent tiles: the two separate passes
        if ((rc = moe_router_topk(cfg, x, Wr, bias, logits, idx, w, tie, status, stream))) return rc;
        return moe_latent_proj(x, W_ld, G.g.T, G.d, G.g.L, z, status, stream);
    }
    GemmDesc d;
    std::memset(&d, 0, sizeof(d));
    d.a_mode = A_DENSE;
    d.epi = EPI_SPLIT;
    d.bn = 256;
    d.M = G.g.T;
    d.N = G.g.L;
    d.nseg = 1;
    d.seg[0] = GemmSeg{x, G.d, W_ld, G.d, G.d};
    d.b_rows = G.g.L;
    d.B_up = Wr;
    d.b2_rows = G.g.E;
    d.nsplit = G.g.L / 256;
    d.N2 = G.g.E;
    d.out = z;
    d.ldo = G.g.L;
    d.out2 = logits;
    d.ldo2 = G.g.E;
    d.bias = bias;
    d.status = status;
    d.name = "gemm_latent_router";
    if ((rc = gemm_launch(d, st))) return rc;
    return launch_topk(logits, G.g.T, G.g.E, G.g.k, idx, w, tie, st);
}

int moe_latent_proj(const uint16_t* in, const uint16_t* W, int64_t M, int32_t K, int32_t N,
                    uint16_t* out, int32_t* status, void* stream) {
    MOE_NVTX_RANGE();
    if (M < 0 || K <= 0 || N <= 0 || K % 8 || N % 8) return MOE_EINVAL;
    if (M == 0) return MOE_OK;
    if (!in || !W || !out || !status) return MOE_EINVAL;
    if (!aligned16(in) || !aligned16(W) || !aligned16(out)) return MOE_EINVAL;
    GemmDesc d;
    std::memset(&d, 0, sizeof(d));
    d.a_mode = A_DENSE;
    d.epi = EPI_BF16;
    d.bn = 256;
    d.M = M;
    d.N = N;
    d.nseg = 1;
    d.seg[0] = GemmSeg{in, K, W, K, K};
    d.b_rows = N;
    d.out = out;
    d.ldo = N;
    d.status = status;
    d.name = "gemm_latent";
    return gemm_launch(d, static_cast<cudaStream_t>(stream));
}

int moe_matmul(const uint16_t* A, int a_mn, int64_t lda, const uint16_t* B, int b_mn,
               int64_t ldb, int64_t M, int32_t N, int32_t K, void* out, int out_f32, int64_t ldo,
               int32_t* status, void* stream) {
    MOE_NVTX_RANGE();
    if (M < 0 || N <= 0 || K <= 0 || lda <= 0 || ldb <= 0 || ldo < N) return MOE_EINVAL;
    if (lda % 8 || ldb % 8 || (out_f32 ? ldo % 4 : ldo % 8) || (!out_f32 && N % 8))
        return MOE_EINVAL;
    if ((!a_mn && lda < K) || (a_mn && lda < M) || (!b_mn && ldb < K) || (b_mn && ldb < N))
        return MOE_EINVAL;
    if (M == 0) return MOE_OK;
    if (!A || !B || !out || !status || !aligned16(A) || !aligned16(B) || !aligned16(out))
        return MOE_EINVAL;
    GemmDesc d;
    std::memset(&d, 0, sizeof(d));
    d.a_mode = A_DENSE;
    d.epi = out_f32 ? EPI_F32 : EPI_BF16;
    d.a_mn = a_mn ? 1 : 0;
    d.b_mn = b_mn ? 1 : 0;
    d.bn = 256;
    d.M = M;
    d.N = N;
    d.nseg = 1;
    d.seg[0] = GemmSeg{A, lda, B, ldb, K};
    d.b_rows = N;
    d.out = out;
    d.ldo = ldo;
    d.status = status;
    d.name = "gemm_matmul";
    return gemm_launch(d, static_cast<cudaStream_t>(stream));
}

int moe_dispatch_pooled(const moe_config_t* cfg, const uint16_t* z, const int32_t* idx, void* ws,
                        size_t ws_bytes, uint16_t* pool, int32_t* slot_of, uint8_t* drop,
                        int32_t* expert_rows, int32_t* expert_count, moe_drop_stats_t* stats,
                        uint16_t* bank, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom(cfg, &G);
    if (rc) return rc;
    if (!stats || !expert_count || (G.g.T > 0 && (!z || !idx || !slot_of || !drop)) ||
        (G.g.pool_rows > 0 && !pool) || (G.plan.c_recv > 0 && !expert_rows) ||
        (G.plan.ws_dispatch_bytes > 0 && !ws))
        return MOE_EINVAL;
    if ((z && !aligned16(z)) || (pool && !aligned16(pool)) || (ws && !aligned16(ws)) ||
        (bank && (!aligned16(bank) || G.g.L % 8)))
        return MOE_EINVAL;
    if (ws_bytes < static_cast<size_t>(G.plan.ws_dispatch_bytes)) return MOE_ENOSPC;
    int dev, sms;
    if ((rc = current_device(&dev, &sms))) return rc;
    return launch_dispatch(G.g, z, idx, ws, pool, slot_of, drop, expert_rows, expert_count, stats,
                           static_cast<cudaStream_t>(stream), -1, true, bank);
}

int moe_plan_ragged(const moe_config_t* cfg, moe_plan_t* plan) {
    if (!plan) return MOE_EINVAL;
    Geom G;
    const int rc = make_geom_ragged(cfg, &G);
    if (rc) return rc;
    *plan = G.plan;
    return MOE_OK;
}

int moe_dispatch_ragged(const moe_config_t* cfg, const uint16_t* z, const int32_t* idx, void* ws,
                        size_t ws_bytes, uint16_t* pool, int32_t* slot_of, uint8_t* drop,
                        int32_t* expert_offsets, int32_t* expert_rows, int32_t* expert_count,
                        moe_drop_stats_t* stats, uint16_t* bank, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom_ragged(cfg, &G);
    if (rc) return rc;
    if (!stats || !expert_count || !expert_offsets || !ws ||
        (G.g.T > 0 && (!z || !idx || !slot_of || !drop || !pool || !expert_rows)))
        return MOE_EINVAL;
    if ((z && !aligned16(z)) || (pool && !aligned16(pool)) || !aligned16(ws) ||
        (bank && (!aligned16(bank) || G.g.L % 8)))
        return MOE_EINVAL;
    if (ws_bytes < static_cast<size_t>(G.plan.ws_dispatch_bytes)) return MOE_ENOSPC;
    int dev, sms;
    if ((rc = current_device(&dev, &sms))) return rc;
    return launch_dispatch_ragged(G.g, z, idx, ws, pool, slot_of, drop, expert_offsets,
                                  expert_rows, expert_count, stats, bank,
                                  static_cast<cudaStream_t>(stream));
}

int moe_expert_ffn_ragged(const moe_config_t* cfg, const uint16_t* pool, const uint16_t* bank,
                          const int32_t* expert_offsets, const int32_t* expert_rows,
                          const int32_t* expert_count, const uint16_t* Wg, const uint16_t* Wu,
                          const uint16_t* Wd, void* ws, size_t ws_bytes, uint16_t* ypool,
                          int32_t* status, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom_ragged(cfg, &G);
    if (rc) return rc;
    const DispatchGeom& g = G.g;
    if (g.pool_rows == 0) return MOE_OK;
    if (!pool || !expert_offsets || !expert_rows || !expert_count || !Wg || !Wu || !Wd || !ws ||
        !ypool || !status)
        return MOE_EINVAL;
    if (!aligned16(pool) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) ||
        !aligned16(ypool) || !aligned16(ws))
        return MOE_EINVAL;
    if (ws_bytes < static_cast<size_t>(G.plan.ws_ffn_bytes)) return MOE_ENOSPC;
    if (bank && !aligned16(bank)) return MOE_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    uint16_t* h = reinterpret_cast<uint16_t*>(wsb + G.plan.h_offset_bytes);
    if (bank && pair_path_fits(G)) {
        rc = expert_ffn_pair_ragged(g.E, g.pool_rows, g.L, G.H, bank, expert_offsets, expert_rows,
                                    expert_count, Wg, Wu, Wd, ws, h, ypool, status, st);
        if (rc != MOE_EINVAL) return rc;   // else: the gathered products below
    }
    int32_t* tiles = reinterpret_cast<int32_t*>(wsb);
    const int max_mt = static_cast<int>(g.pool_rows / 128 + g.E);
    int32_t* tile_count = reinterpret_cast<int32_t*>(wsb + static_cast<size_t>(max_mt) * 8);
    if ((rc = launch_build_tiles(expert_count, g.E, 128, tiles, tile_count, st))) return rc;
    const int L = g.L, H = G.H;
    const int n = static_cast<int>(g.pool_rows);

    GemmDesc d1;
    std::memset(&d1, 0, sizeof(d1));
    d1.a_mode = A_GATHER;
    d1.epi = EPI_SWIGLU;
    d1.bn = 256;
    d1.N = H;
    d1.nseg = 1;
    d1.seg[0] = GemmSeg{nullptr, 0, Wg, L, L};
    d1.B_up = Wu;
    d1.groups = g.E;
    d1.b_rows = H;
    d1.b_gstride = static_cast<int64_t>(H) * L;
    d1.tile_list = tiles;
    d1.tile_count = tile_count;
    d1.max_tiles = max_mt;
    d1.rowmap = expert_rows;
    d1.counts = expert_count;
    d1.goff = expert_offsets;
    d1.gather_src = pool;
    d1.gather_pitch = pool_pitch(L);
    d1.gather_rows = n;
    d1.out = h;
    d1.ldo = H;
    d1.status = status;
    d1.name = "gemm_expert_gateup";
    if ((rc = gemm_launch(d1, st))) return rc;

    GemmDesc d2;
    std::memset(&d2, 0, sizeof(d2));
    d2.a_mode = A_GROUPED;
    d2.epi = EPI_SCATTER;
    d2.bn = 256;
    d2.N = L;
    d2.nseg = 1;
    d2.seg[0] = GemmSeg{h, H, Wd, H, H};
    d2.groups = g.E;
    d2.rows_per_group = n;   // with goff: rows of the flat h
    d2.b_rows = L;
    d2.b_gstride = static_cast<int64_t>(L) * H;
    d2.tile_list = tiles;
    d2.tile_count = tile_count;
    d2.max_tiles = max_mt;
    d2.rowmap = expert_rows;
    d2.counts = expert_count;
    d2.goff = expert_offsets;
    d2.out = ypool;
    d2.ldo = L;
    d2.status = status;
    d2.name = "gemm_expert_down";
    d2.gather_rows = g.pool_rows;   // the scatter's destination rows
    return gemm_launch(d2, st);
}

// The capped layout's expert FFN: gate/up with the rows gathered from the
// pool, then the down-projection scattered back to the rows.  wp (optional):
// the wave pipeline's copy of waves 1.. into the pool inside the gate/up launch.
struct WavePipe {
    int32_t* ready;
    PackArgs a;
};

// The per-expert bank path (CTA pairs, rows on the MMA's N axis) takes
// widths that are whole 256-column output blocks and 128-unit hidden blocks.
static int expert_ffn_capped(const Geom& G, uint16_t* pool, const int32_t* expert_rows,
                             const int32_t* expert_count, const uint16_t* Wg, const uint16_t* Wu,
                             const uint16_t* Wd, void* ws, uint16_t* ypool, int32_t* status,
                             cudaStream_t st, const WavePipe* wp, const uint16_t* bank = nullptr) {
    int rc;
    const DispatchGeom& g = G.g;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    if (bank && !wp && pair_path_fits(G))
        return expert_ffn_pair(g.E, g.c_recv, g.L, G.H, bank, expert_rows, expert_count, Wg, Wu,
                               Wd, ws, reinterpret_cast<uint16_t*>(wsb + G.plan.h_offset_bytes),
                               ypool, g.pool_rows, status, st);
    int32_t* tiles = reinterpret_cast<int32_t*>(wsb);
    const int max_mt = g.E * ((g.c_recv + 127) / 128);
    int32_t* tile_count = reinterpret_cast<int32_t*>(wsb + static_cast<size_t>(max_mt) * 8);
    uint16_t* h = reinterpret_cast<uint16_t*>(wsb + G.plan.h_offset_bytes);
    // the pipeline takes the tiles wave by wave, so that every CTA works on
    // wave 0 while the later waves' rows are being copied
    if ((rc = launch_build_tiles(expert_count, g.E, 128, tiles, tile_count, st, wp ? g.E_l : 0,
                                 wp ? g.E_w : 0)))
        return rc;

    const int L = g.L, H = G.H;
    GemmDesc d1;
    std::memset(&d1, 0, sizeof(d1));
    d1.a_mode = A_GATHER;
    d1.epi = EPI_SWIGLU;
    d1.bn = 256;
    d1.N = H;
    d1.nseg = 1;
    d1.seg[0] = GemmSeg{nullptr, 0, Wg, L, L};
    d1.B_up = Wu;
    d1.groups = g.E;
    d1.rows_per_group = g.c_recv;
    d1.b_rows = H;
    d1.b_gstride = static_cast<int64_t>(H) * L;
    d1.tile_list = tiles;
    d1.tile_count = tile_count;
    d1.max_tiles = max_mt;
    d1.rowmap = expert_rows;
    d1.counts = expert_count;
    d1.rowmap_ld = g.c_recv;
    d1.gather_src = pool;
    d1.gather_pitch = pool_pitch(L);
    d1.gather_rows = g.pool_rows;
    d1.out = h;
    d1.ldo = H;
    d1.out_gstride = static_cast<int64_t>(g.c_recv) * H;
    d1.status = status;
    d1.name = "gemm_expert_gateup";
    if (wp) {
        d1.wp_ready = wp->ready;
        d1.wp_g = g;
        d1.wp_a = wp->a;
    }
    if ((rc = gemm_launch(d1, st))) return rc;

    GemmDesc d2;
    std::memset(&d2, 0, sizeof(d2));
    d2.a_mode = A_GROUPED;
    d2.epi = EPI_SCATTER;
    d2.bn = 256;
    d2.N = L;
    d2.nseg = 1;
    d2.seg[0] = GemmSeg{h, H, Wd, H, H};
    d2.groups = g.E;
    d2.rows_per_group = g.c_recv;
    d2.a_gstride = static_cast<int64_t>(g.c_recv) * H;
    d2.b_rows = L;
    d2.b_gstride = static_cast<int64_t>(L) * H;
    d2.tile_list = tiles;
    d2.tile_count = tile_count;
    d2.max_tiles = max_mt;
    d2.rowmap = expert_rows;
    d2.counts = expert_count;
    d2.rowmap_ld = g.c_recv;
    d2.out = ypool;
    d2.ldo = L;
    d2.status = status;
    d2.name = "gemm_expert_down";
    d2.gather_rows = g.pool_rows;   // the scatter's destination rows
    return gemm_launch(d2, st);
}

static int check_ffn_args(const Geom& G, const uint16_t* pool, const int32_t* expert_rows,
                          const int32_t* expert_count, const uint16_t* Wg, const uint16_t* Wu,
                          const uint16_t* Wd, const void* ws, size_t ws_bytes,
                          const uint16_t* ypool, const int32_t* status) {
    if (!pool || !expert_rows || !expert_count || !Wg || !Wu || !Wd || !ws || !ypool || !status)
        return MOE_EINVAL;
    if (!aligned16(pool) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) ||
        !aligned16(ypool) || !aligned16(ws))
        return MOE_EINVAL;
    if (ws_bytes < static_cast<size_t>(G.plan.ws_ffn_bytes)) return MOE_ENOSPC;
    return MOE_OK;
}

int moe_expert_ffn_grouped(const moe_config_t* cfg, const uint16_t* pool, const uint16_t* bank,
                           const int32_t* expert_rows, const int32_t* expert_count,
                           const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, void* ws,
                           size_t ws_bytes, uint16_t* ypool, int32_t* status, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom(cfg, &G);
    if (rc) return rc;
    if (G.g.pool_rows == 0 || G.g.c_recv == 0) return MOE_OK;
    if ((rc = check_ffn_args(G, pool, expert_rows, expert_count, Wg, Wu, Wd, ws, ws_bytes, ypool,
                             status)))
        return rc;
    if (bank && !aligned16(bank)) return MOE_EINVAL;
    return expert_ffn_capped(G, const_cast<uint16_t*>(pool), expert_rows, expert_count, Wg, Wu,
                             Wd, ws, ypool, status, static_cast<cudaStream_t>(stream), nullptr,
                             bank);
}

int moe_dispatch_expert_waves(const moe_config_t* cfg, const uint16_t* z, const int32_t* idx,
                              void* ws, size_t ws_bytes, uint16_t* pool, int32_t* slot_of,
                              uint8_t* drop, int32_t* expert_rows, int32_t* expert_count,
                              moe_drop_stats_t* stats, const uint16_t* Wg, const uint16_t* Wu,
                              const uint16_t* Wd, void* ffn_ws, size_t ffn_ws_bytes,
                              uint16_t* ypool, int32_t* status, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom(cfg, &G);
    if (rc) return rc;
    const DispatchGeom& g = G.g;
    if (!stats || !expert_count || (g.T > 0 && (!z || !idx || !slot_of || !drop)) ||
        (g.pool_rows > 0 && !pool) || (G.plan.c_recv > 0 && !expert_rows) ||
        (G.plan.ws_dispatch_bytes > 0 && !ws))
        return MOE_EINVAL;
    if ((z && !aligned16(z)) || (pool && !aligned16(pool)) || (ws && !aligned16(ws)))
        return MOE_EINVAL;
    if (ws_bytes < static_cast<size_t>(G.plan.ws_dispatch_bytes)) return MOE_ENOSPC;
    const bool ffn = g.pool_rows > 0 && g.c_recv > 0;
    if (ffn && (rc = check_ffn_args(G, pool, expert_rows, expert_count, Wg, Wu, Wd, ffn_ws,
                                    ffn_ws_bytes, ypool, status)))
        return rc;
    int dev, sms;
    if ((rc = current_device(&dev, &sms))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // with one wave, no rows or no expert rows there is nothing to overlap:
    // the dispatch fills every wave and the expert FFN runs as usual
    const bool pipe = ffn && g.T > 0 && g.W > 1;
    if ((rc = launch_dispatch(g, z, idx, ws, pool, slot_of, drop, expert_rows, expert_count, stats,
                              st, pipe ? 0 : -1)))
        return rc;
    if (!ffn) return MOE_OK;
    const DispatchWs L = dispatch_ws_layout(g);
    uint8_t* w = static_cast<uint8_t*>(ws);
    WavePipe wp;
    std::memset(&wp, 0, sizeof(wp));
    wp.ready = reinterpret_cast<int32_t*>(w + L.wave_ready_off);
    wp.a.z = z;
    wp.a.idx = idx;
    wp.a.send_row = reinterpret_cast<const int64_t*>(w + L.send_row_off);
    wp.a.pool = pool;
    return expert_ffn_capped(G, pool, expert_rows, expert_count, Wg, Wu, Wd, ffn_ws, ypool,
                             status, st, pipe ? &wp : nullptr);
}

}  // extern "C"

// The shared experts' gate/up; with pack, its extra warps also carry the
// dispatch's pack (final decisions, row lists, copies, tags) of the layout
// g describes.
static int shared_gateup(const Geom& G, const PackArgs* pack, const uint16_t* x,
                         const uint16_t* Wsg, const uint16_t* Wsu, uint16_t* a, int32_t* status,
                         cudaStream_t st) {
    const DispatchGeom& g = G.g;
    const int d = G.d, hs_all = G.ns * G.Hs;
    GemmDesc s1;
    std::memset(&s1, 0, sizeof(s1));
    s1.a_mode = A_DENSE;
    s1.epi = EPI_SWIGLU;
    s1.bn = 256;
    s1.M = g.T;
    s1.N = hs_all;
    s1.nseg = 1;
    s1.seg[0] = GemmSeg{x, d, Wsg, d, d};
    s1.B_up = Wsu;
    s1.b_rows = hs_all;
    s1.out = a;
    s1.ldo = hs_all;
    s1.status = status;
    s1.name = "gemm_shared_gateup";
    if (pack) {
        s1.wp_g = g;
        s1.wp_a = *pack;
    }
    return gemm_launch(s1, st);
}

static PackArgs pack_args(const DispatchGeom& g, void* ws, const uint16_t* z, const int32_t* idx,
                          uint16_t* pool, int32_t* slot_of, uint8_t* drop, int32_t* expert_rows,
                          const int32_t* expert_offsets, uint16_t* bank) {
    const DispatchWs Lw = dispatch_ws_layout(g);
    uint8_t* w = static_cast<uint8_t*>(ws);
    PackArgs P;
    std::memset(&P, 0, sizeof(P));
    P.z = z;
    P.idx = idx;
    P.send_row = reinterpret_cast<const int64_t*>(w + Lw.send_row_off);
    P.rloc = reinterpret_cast<const int32_t*>(w + Lw.rloc_off);
    P.base_se = reinterpret_cast<const int32_t*>(w + Lw.base_se_off);
    P.pool = pool;
    P.slot_of = slot_of;
    P.drop = drop;
    P.expert_rows = expert_rows;
    if (g.ragged) {
        P.blk_off = reinterpret_cast<const int32_t*>(w + Lw.blk_off_off);
        P.eoff = expert_offsets;
    }
    P.bank = bank;
    return P;
}

static int check_shared_args(const Geom& G, const uint16_t* x, const uint16_t* Wsg,
                             const uint16_t* Wsu, const uint16_t* a) {
    if (G.ns > 0 && G.g.T > 0 &&
        (!x || !Wsg || !Wsu || !a || !aligned16(x) || !aligned16(Wsg) || !aligned16(Wsu) ||
         !aligned16(a)))
        return MOE_EINVAL;
    return MOE_OK;
}

extern "C" {

int moe_dispatch_shared_overlap(const moe_config_t* cfg, const uint16_t* z, const int32_t* idx,
                                void* ws, size_t ws_bytes, uint16_t* pool, int32_t* slot_of,
                                uint8_t* drop, int32_t* expert_rows, int32_t* expert_count,
                                moe_drop_stats_t* stats, uint16_t* bank, const uint16_t* x,
                                const uint16_t* Wsg,
                                const uint16_t* Wsu, uint16_t* a, int32_t* status,
                                void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom(cfg, &G);
    if (rc) return rc;
    const DispatchGeom& g = G.g;
    if (!stats || !expert_count || !status || (g.T > 0 && (!z || !idx || !slot_of || !drop)) ||
        (g.pool_rows > 0 && !pool) || (G.plan.c_recv > 0 && !expert_rows) ||
        (G.plan.ws_dispatch_bytes > 0 && !ws))
        return MOE_EINVAL;
    if ((z && !aligned16(z)) || (pool && !aligned16(pool)) || (ws && !aligned16(ws)))
        return MOE_EINVAL;
    if (ws_bytes < static_cast<size_t>(G.plan.ws_dispatch_bytes)) return MOE_ENOSPC;
    if ((rc = check_shared_args(G, x, Wsg, Wsu, a))) return rc;
    int dev, sms;
    if ((rc = current_device(&dev, &sms))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // without shared experts there is nothing to overlap the pack with
    const bool overlap = G.ns > 0 && g.T > 0 && g.pool_rows > 0;
    if ((rc = launch_dispatch(g, z, idx, ws, pool, slot_of, drop, expert_rows, expert_count, stats,
                              st, -1, !overlap, bank)))
        return rc;
    if (G.ns == 0 || g.T == 0) return MOE_OK;
    const PackArgs P = pack_args(g, ws, z, idx, pool, slot_of, drop, expert_rows, nullptr, bank);
    return shared_gateup(G, overlap ? &P : nullptr, x, Wsg, Wsu, a, status, st);
}

int moe_dispatch_ragged_shared_overlap(const moe_config_t* cfg, const uint16_t* z,
                                       const int32_t* idx, void* ws, size_t ws_bytes,
                                       uint16_t* pool, int32_t* slot_of, uint8_t* drop,
                                       int32_t* expert_offsets, int32_t* expert_rows,
                                       int32_t* expert_count, moe_drop_stats_t* stats,
                                       uint16_t* bank, const uint16_t* x, const uint16_t* Wsg,
                                       const uint16_t* Wsu, uint16_t* a, int32_t* status,
                                       void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom_ragged(cfg, &G);
    if (rc) return rc;
    const DispatchGeom& g = G.g;
    if (!stats || !expert_count || !expert_offsets || !ws || !status ||
        (g.T > 0 && (!z || !idx || !slot_of || !drop || !pool || !expert_rows)))
        return MOE_EINVAL;
    if ((z && !aligned16(z)) || (pool && !aligned16(pool)) || !aligned16(ws) ||
        (bank && (!aligned16(bank) || g.L % 8)))
        return MOE_EINVAL;
    if (ws_bytes < static_cast<size_t>(G.plan.ws_dispatch_bytes)) return MOE_ENOSPC;
    if ((rc = check_shared_args(G, x, Wsg, Wsu, a))) return rc;
    int dev, sms;
    if ((rc = current_device(&dev, &sms))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool overlap = G.ns > 0 && g.T > 0;
    if ((rc = launch_dispatch_ragged(g, z, idx, ws, pool, slot_of, drop, expert_offsets,
                                     expert_rows, expert_count, stats, bank, st, !overlap)))
        return rc;
    if (G.ns == 0 || g.T == 0) return MOE_OK;
    const PackArgs P =
        pack_args(g, ws, z, idx, pool, slot_of, drop, expert_rows, expert_offsets, bank);
    return shared_gateup(G, &P, x, Wsg, Wsu, a, status, st);
}

int moe_balance_update(const moe_config_t* cfg, const int32_t* idx, int64_t* hist, float alpha,
                       float* bias, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom(cfg, &G);
    if (rc) return rc;
    if (!hist || !bias || (G.g.T > 0 && !idx) || !(alpha == alpha)) return MOE_EINVAL;
    if ((reinterpret_cast<uintptr_t>(hist) & 7u) || (reinterpret_cast<uintptr_t>(bias) & 3u))
        return MOE_EINVAL;
    int dev, sms;
    if ((rc = current_device(&dev, &sms))) return rc;
    return launch_balance_update(idx, G.g.T * G.g.k, G.g.E, hist, alpha, bias,
                                 static_cast<cudaStream_t>(stream));
}

int moe_balance_update_window(const moe_config_t* cfg, const int32_t* idx, int64_t* hist,
                              int64_t* ring, int32_t window, int64_t* step, float alpha,
                              float* bias, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom(cfg, &G);
    if (rc) return rc;
    if (!hist || !ring || !step || !bias || window < 1 || (G.g.T > 0 && !idx) || !(alpha == alpha))
        return MOE_EINVAL;
    if ((reinterpret_cast<uintptr_t>(hist) & 7u) || (reinterpret_cast<uintptr_t>(ring) & 7u) ||
        (reinterpret_cast<uintptr_t>(step) & 7u) || (reinterpret_cast<uintptr_t>(bias) & 3u))
        return MOE_EINVAL;
    int dev, sms;
    if ((rc = current_device(&dev, &sms))) return rc;
    return launch_balance_window(idx, G.g.T * G.g.k, G.g.E, hist, ring, window, step, alpha, bias,
                                 static_cast<cudaStream_t>(stream));
}

static void fill_backward_layout(const BackwardWs& w, moe_backward_ws_t* layout) {
    layout->dc = w.dc; layout->da = w.da; layout->dgs = w.dgs; layout->dus = w.dus;
    layout->dw = w.dw; layout->rowinv = w.rowinv; layout->dxpool = w.dxpool; layout->dh = w.dh;
    layout->dg = w.dg; layout->du = w.du; layout->xe = w.xe; layout->dye = w.dye;
    layout->dz = w.dz; layout->dlogits = w.dlogits; layout->tiles = w.tiles;
    layout->hp = w.hp; layout->poff = w.poff;
    layout->total = w.total;
}

int moe_backward_plan(const moe_config_t* cfg, moe_backward_ws_t* layout) {
    if (!layout) return MOE_EINVAL;
    Geom G;
    const int rc = make_geom(cfg, &G);
    if (rc) return rc;
    fill_backward_layout(backward_ws_layout(G.g, G.d, G.H, G.Hs, G.ns), layout);
    return MOE_OK;
}

int moe_backward_plan_ragged(const moe_config_t* cfg, moe_backward_ws_t* layout) {
    if (!layout) return MOE_EINVAL;
    Geom G;
    const int rc = make_geom_ragged(cfg, &G);
    if (rc) return rc;
    fill_backward_layout(backward_ws_layout(G.g, G.d, G.H, G.Hs, G.ns), layout);
    return MOE_OK;
}

static int layer_backward(const Geom& G, const moe_backward_args_t* a, void* stream) {
    if (!a) return MOE_EINVAL;
    if (G.g.T == 0) return MOE_OK;
    const void* need[] = {a->x, a->Wr, a->W_ld, a->Wg, a->Wu, a->Wd, a->W_lu, a->idx, a->w,
                          a->pool, a->slot_of, a->expert_rows, a->expert_count, a->h, a->ypool,
                          a->c, a->dout, a->dx, a->dWr, a->dW_ld, a->dWg, a->dWu, a->dWd,
                          a->dW_lu, a->ws, a->status};
    for (const void* ptr : need)
        if (!ptr) return MOE_EINVAL;
    if (G.ns > 0 && (!a->Wsg || !a->Wsu || !a->Wsd || !a->a || !a->dWsg || !a->dWsu || !a->dWsd))
        return MOE_EINVAL;
    if (G.g.ragged ? !a->expert_offsets : a->expert_offsets != nullptr) return MOE_EINVAL;
    const void* al16[] = {a->x, a->Wr, a->W_ld, a->Wg, a->Wu, a->Wd, a->W_lu, a->pool, a->h,
                          a->ypool, a->c, a->dout, a->dx, a->dWr, a->dW_ld, a->dWg, a->dWu,
                          a->dWd, a->dW_lu, a->ws};
    for (const void* ptr : al16)
        if (!aligned16(ptr)) return MOE_EINVAL;
    if (a->bank && !aligned16(a->bank)) return MOE_EINVAL;
    if (G.g.pool_rows == 0 || G.g.c_recv == 0) return MOE_EINVAL;
    const BackwardWs w = backward_ws_layout(G.g, G.d, G.H, G.Hs, G.ns);
    if (a->ws_bytes < w.total) return MOE_ENOSPC;
    int dev, sms, rc;
    if ((rc = current_device(&dev, &sms))) return rc;
    return launch_backward(G.g, G.d, G.H, G.Hs, G.ns, *a, static_cast<cudaStream_t>(stream));
}

int moe_layer_backward(const moe_config_t* cfg, const moe_backward_args_t* a, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    const int rc = make_geom(cfg, &G);
    if (rc) return rc;
    return layer_backward(G, a, stream);
}

int moe_layer_backward_ragged(const moe_config_t* cfg, const moe_backward_args_t* a,
                              void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    const int rc = make_geom_ragged(cfg, &G);
    if (rc) return rc;
    return layer_backward(G, a, stream);
}

int moe_combine(const moe_config_t* cfg, const uint16_t* ypool, const int32_t* slot_of,
                const float* w, const uint16_t* W_lu, const uint16_t* x, const uint16_t* Wsg,
                const uint16_t* Wsu, const uint16_t* Wsd, uint16_t* c, uint16_t* a,
                uint16_t* out, int32_t* status, void* stream) {
    MOE_NVTX_RANGE();
    Geom G;
    int rc = make_geom(cfg, &G);
    if (rc) return rc;
    const DispatchGeom& g = G.g;
    if (g.T == 0) return MOE_OK;
    if (!slot_of || !w || !W_lu || !c || !out || !status || (g.pool_rows > 0 && !ypool))
        return MOE_EINVAL;
    // Wsg = Wsu = NULL: a already holds the shared activations (computed
    // beside the dispatch by moe_dispatch_shared_overlap)
    const bool a_ready = G.ns > 0 && !Wsg && !Wsu;
    if (G.ns > 0 && (!Wsd || !a || (!a_ready && (!x || !Wsg || !Wsu)))) return MOE_EINVAL;
    if ((ypool && !aligned16(ypool)) || !aligned16(W_lu) || !aligned16(c) || !aligned16(out))
        return MOE_EINVAL;
    if (G.ns > 0 && (!aligned16(Wsd) || !aligned16(a) ||
                     (!a_ready && (!aligned16(x) || !aligned16(Wsg) || !aligned16(Wsu)))))
        return MOE_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((rc = launch_combine(ypool, slot_of, w, g.T, g.k, g.L, c, g.pool_rows, st))) return rc;

    const int d = G.d, Hs = G.Hs, ns = G.ns;
    const int hs_all = ns * Hs;
    if (ns > 0 && !a_ready) {
        GemmDesc s1;
        std::memset(&s1, 0, sizeof(s1));
        s1.a_mode = A_DENSE;
        s1.epi = EPI_SWIGLU;
        s1.bn = 256;
        s1.M = g.T;
        s1.N = hs_all;
        s1.nseg = 1;
        s1.seg[0] = GemmSeg{x, d, Wsg, d, d};
        s1.B_up = Wsu;
        s1.b_rows = hs_all;
        s1.out = a;
        s1.ldo = hs_all;
        s1.status = status;
        s1.name = "gemm_shared_gateup";
        if ((rc = gemm_launch(s1, st))) return rc;
    }
    GemmDesc o;
    std::memset(&o, 0, sizeof(o));
    o.a_mode = A_DENSE;
    o.epi = EPI_BF16;
    o.bn = 256;
    o.M = g.T;
    o.N = d;
    o.nseg = 1 + ns;
    o.seg[0] = GemmSeg{c, g.L, W_lu, g.L, g.L};
    for (int s = 0; s < ns; ++s)
        o.seg[1 + s] = GemmSeg{a + static_cast<size_t>(s) * Hs, hs_all,
                               Wsd + static_cast<size_t>(s) * d * Hs, Hs, Hs};
    o.b_rows = d;
    o.out = out;
    o.ldo = d;
    o.status = status;
    o.name = "gemm_out";
    return gemm_launch(o, st);
}

}  // extern "C"
