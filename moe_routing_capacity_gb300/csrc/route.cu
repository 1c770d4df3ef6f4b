// route.cu -- the bandwidth- and latency-bound steps of the layer:
//   router top-k        one warp per token, rounds of warp max / min
//                       reductions over each lane's earliest entries
//   dispatch            sender slots and receiver ranks (warp-aggregated
//                       counting, deterministic prefix sums), drops counted,
//                       payload rows packed into the fixed pools
//   combine             the return gather: per token, weighted sum of its
//                       kept expert rows
//   tile list           {expert, m0} work items of the grouped expert GEMMs
#include <algorithm>
#include <climits>
#include <cstdio>

#include "common.cuh"
#include "internal.h"
#include "pack.cuh"

namespace moe {

// ==================================================================== top-k

constexpr float kTieEps = 1e-4f;

// The routing order on the logit alone as an unsigned key: a larger logit,
// a larger key (-0 taken as +0, so equal logits give equal keys); 0 marks no
// entry.  Among equal keys the lower expert id ranks first.  Logits are
// finite here (a product of finite inputs); a NaN ranks where its bits put
// it, the one whose bits are all ones as no entry, and routing with NaN
// logits is left unspecified, as for the oracle.
__device__ __forceinline__ uint32_t logit_key(float v) {
    const uint32_t b = __float_as_uint(__fadd_rn(v, 0.0f));
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <int PER>   // logits per lane: E <= 32 * PER
__global__ void __launch_bounds__(256, PER > 16 ? 2 : 5)
    topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k,
                int32_t* __restrict__ idx, float* __restrict__ w, uint8_t* __restrict__ tie) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* row = logits + t * E;
    float v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldg(row + e) : 0.0f;
    }
    // This lane's entries are experts lane + 32 i.  Its two earliest in
    // routing order: head (hk, hi, hv) and second (sk, si, sv); ids ascend
    // with i, so a strict comparison keeps the lower id first on equal keys.
    uint32_t hk = 0, sk = 0;
    int hi = -1, si = -1;
    float hv = 0.0f, sv = 0.0f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        if (lane + 32 * i < E) {
            const uint32_t kk = logit_key(v[i]);
            if (kk > hk) {
                sk = hk; si = hi; sv = hv;
                hk = kk; hi = i; hv = v[i];
            } else if (kk > sk) {
                sk = kk; si = i; sv = v[i];
            }
        }
    }
    // Rounds of selection across the warp: the largest head key, the lowest
    // expert id among the heads that hold it; the winning lane moves on to its
    // second entry, or rescans its unused ones after two wins.
    float my_v = 0.0f;   // lane j holds the j-th entry in routing order
    int my_e = 0;
    float next_v = 0.0f; // the (k+1)-th largest logit
    uint32_t used = 0;   // bit i: entry i of this lane already ranked
    const int rounds = k < E ? k + 1 : k;   // entries to rank
    for (int rd = 0; rd < rounds; ++rd) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, hk);
        const uint32_t mine =
            (hi >= 0 && hk == m) ? static_cast<uint32_t>(lane + 32 * hi) : 0xffffffffu;
        const uint32_t we = __reduce_min_sync(0xffffffffu, mine);
        const int wl = static_cast<int>(we & 31u);
        const float vr = __shfl_sync(0xffffffffu, hv, wl);
        if (rd < k) {
            if (lane == rd) {
                my_v = vr;
                my_e = static_cast<int>(we);
            }
        } else {
            next_v = vr;
        }
        if (lane == wl) {
            used |= 1u << hi;
            if (si >= 0) {
                hk = sk; hi = si; hv = sv;
                sk = 0; si = -1;
            } else {
                hk = 0; hi = -1;
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    if (lane + 32 * i < E && !(used >> i & 1u)) {
                        const uint32_t kk = logit_key(v[i]);
                        if (kk > hk) {
                            hk = kk; hi = i; hv = v[i];
                        }
                    }
                }
            }
        }
    }
    // softmax over the selected logits (lane 0 holds the largest)
    const float vmax = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = lane < k ? expf(my_v - vmax) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    // near ties: exact differences in double against float(1e-4)
    const float nb_v = __shfl_down_sync(0xffffffffu, my_v, 1);
    const bool inner = (lane + 1 < k) &&
                       (static_cast<double>(my_v) - static_cast<double>(nb_v) <
                        static_cast<double>(kTieEps));
    const unsigned inner_any = __ballot_sync(0xffffffffu, inner);
    const float last_v = __shfl_sync(0xffffffffu, my_v, k - 1);
    if (lane < k) {
        idx[t * k + lane] = my_e;
        w[t * k + lane] = ex / sum;
    }
    if (lane == 0) {
        uint8_t f = inner_any ? 2 : 0;
        if (k < E && static_cast<double>(last_v) - static_cast<double>(next_v) <
                         static_cast<double>(kTieEps))
            f |= 1;
        tie[t] = f;
    }
}

int launch_topk(const float* logits, int64_t T, int E, int k, int32_t* idx, float* w,
                uint8_t* tie, cudaStream_t st) {
    if (T == 0) return MOE_OK;
    const int per = (E + 31) / 32;
    const int tpb = 256;
    const unsigned grid = static_cast<unsigned>((T + 7) / 8);
#define MOE_TOPK(P)                                                              \
    topk_kernel<P><<<grid, tpb, 0, st>>>(logits, T, E, k, idx, w, tie);        \
    break;
    switch (per <= 4 ? 4 : per <= 8 ? 8 : per <= 12 ? 12 : per <= 16 ? 16 : 32) {
        case 4: MOE_TOPK(4)
        case 8: MOE_TOPK(8)
        case 12: MOE_TOPK(12)
        case 16: MOE_TOPK(16)
        default: MOE_TOPK(32)
    }
#undef MOE_TOPK
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "router_topk");
    return MOE_OK;
}

// ==================================================================== dispatch

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

DispatchWs dispatch_ws_layout(const DispatchGeom& g) {
    DispatchWs w;
    size_t o = 0;
    const size_t n = static_cast<size_t>(g.T) * g.k;
    w.send_row_off = o;  o = align256(o + n * sizeof(int64_t));
    w.rloc_off = o;      o = align256(o + n * sizeof(int32_t));
    w.cnt_se_off = o;    o = align256(o + static_cast<size_t>(g.S) * g.E * sizeof(int32_t));
    w.base_se_off = o;   o = align256(o + static_cast<size_t>(g.S) * g.E * sizeof(int32_t));
    w.demand_off = o;    o = align256(o + static_cast<size_t>(g.S) * g.D * g.W * sizeof(int32_t));
    w.blk_off_off = o;
    if (g.ragged) o = align256(o + (static_cast<size_t>(g.S) * g.D * g.W + 1) * sizeof(int32_t));
    w.wave_ready_off = o; o = align256(o + static_cast<size_t>(g.W) * sizeof(int32_t));
    w.total = o;
    return w;
}

// Reset the stats and the per-wave copy counters, write the empty tag into
// every pool row and -1 into the expert row lists.
__global__ void dispatch_init_kernel(DispatchGeom g, uint16_t* __restrict__ pool,
                                     int32_t* __restrict__ expert_rows,
                                     moe_drop_stats_t* __restrict__ stats,
                                     int32_t* __restrict__ wave_ready) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (tid < g.W) wave_ready[tid] = 0;
    if (tid == 0) {
        stats->assignments = g.T * g.k;
        stats->kept = 0;
        stats->dropped_send = 0;
        stats->dropped_recv = 0;
        stats->max_send_fill = 0;
        stats->max_expert_rows = 0;
        stats->status = 0;
        stats->reserved = 0;
    }
    if (g.ragged) return;   // every row and every list entry gets written
    const int64_t pitch = pool_pitch(g.L);
    for (int64_t r = tid; r < g.pool_rows; r += nthr)
        *reinterpret_cast<int4*>(pool + r * pitch + g.L) = make_int4(-1, -1, -1, 0);
    const int64_t ne = static_cast<int64_t>(g.E) * g.c_recv;
    for (int64_t i = tid; i < ne; i += nthr) expert_rows[i] = -1;
}

// Sender stage and the per-source half of the receiver stage, one CTA per
// source rank.  The source's assignments are taken in priority order in
// rounds of at most SEND_WARPS x 32 x SEND_PER_LANE; a round is split evenly
// over the warps (in multiples of 32) and warp w holds its contiguous slice in
// registers.  Slots are exact ranks in priority order,
// obtained without atomics on shared counts:
//   pass 1  each warp counts its slice per (destination, wave) key: lanes with
//           the same key find each other with __match_any_sync and the
//           group's lowest lane adds the group size to the warp's counter;
//   scan    per key, an exclusive prefix over warps (plus the rounds before)
//           gives each warp's first slot -- a deterministic prefix sum;
//   pass 2  slot = warp base + rank within the group so far; kept if
//           slot < c_send; kept rows are counted per expert the same way;
//   scan    per expert, prefix over warps;
//   pass 3  each kept row's rank among this source's kept rows for its expert.
constexpr int SEND_WARPS = 16;
constexpr int SEND_PER_LANE = 16;

__global__ void __launch_bounds__(SEND_WARPS * 32) dispatch_send_kernel(
    DispatchGeom g, const int32_t* __restrict__ idx, int64_t* __restrict__ send_row,
    int32_t* __restrict__ rloc, int32_t* __restrict__ cnt_se, int32_t* __restrict__ demand,
    moe_drop_stats_t* __restrict__ stats) {
    extern __shared__ int32_t sh[];
    const int nkey = g.D * g.W;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    int32_t* cnt_key = sh;                              // [SEND_WARPS][nkey]
    int32_t* cnt_e = cnt_key + SEND_WARPS * nkey;       // [SEND_WARPS][E]
    int32_t* run_key = cnt_e + SEND_WARPS * g.E;        // [nkey] totals of earlier rounds
    int32_t* run_e = run_key + nkey;                    // [E]
    for (int i = threadIdx.x; i < nkey + g.E; i += blockDim.x) run_key[i] = 0;

    const int s = blockIdx.x;
    const int64_t n = g.T_s * g.k;
    const int64_t first = static_cast<int64_t>(s) * n;
    int64_t dropped = 0;
    bool bad = false;
    constexpr int ROUND = SEND_WARPS * 32 * SEND_PER_LANE;
    for (int64_t base = 0; base < n; base += ROUND) {
        const int64_t rn = n - base < ROUND ? n - base : ROUND;       // items this round
        const int per_warp = static_cast<int>((rn + SEND_WARPS * 32 - 1) / (SEND_WARPS * 32)) * 32;
        const int64_t wbase = base + static_cast<int64_t>(warp) * per_warp;
        const int64_t wend = (wbase + per_warp < base + rn) ? wbase + per_warp : base + rn;
        int e[SEND_PER_LANE];
#pragma unroll
        for (int i = 0; i < SEND_PER_LANE; ++i) {
            const int64_t a = wbase + 32 * i + lane;
            e[i] = a < wend ? idx[first + a] : -1;
            if (a < wend && (e[i] < 0 || e[i] >= g.E)) {
                bad = true;
                e[i] = 0;
            }
        }
        int32_t* my_key = cnt_key + warp * nkey;
        int32_t* my_e = cnt_e + warp * g.E;
        for (int i = lane; i < nkey; i += 32) my_key[i] = 0;
        for (int i = lane; i < g.E; i += 32) my_e[i] = 0;
        __syncwarp();
        // pass 1: per-warp key counts
#pragma unroll
        for (int i = 0; i < SEND_PER_LANE; ++i) {
            if (i * 32 >= per_warp) break;
            const bool v = e[i] >= 0;
            const int dst = e[i] / g.E_l;
            const int key = dst * g.W + (e[i] - dst * g.E_l) / g.E_w;
            const unsigned peers = __match_any_sync(0xffffffffu, v ? key : -1 - lane);
            if (v && (peers & lt) == 0) my_key[key] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        for (int key = threadIdx.x; key < nkey; key += blockDim.x) {
            int acc = run_key[key];
            for (int w = 0; w < SEND_WARPS; ++w) {
                const int c = cnt_key[w * nkey + key];
                cnt_key[w * nkey + key] = acc;
                acc += c;
            }
            run_key[key] = acc;
        }
        __syncthreads();
        // pass 2: slots, sender decisions, per-warp counts of kept rows per expert
        uint32_t kept_mask = 0;
#pragma unroll
        for (int i = 0; i < SEND_PER_LANE; ++i) {
            if (i * 32 >= per_warp) break;
            const bool v = e[i] >= 0;
            const int dst = e[i] / g.E_l;
            const int key = dst * g.W + (e[i] - dst * g.E_l) / g.E_w;
            const unsigned peers = __match_any_sync(0xffffffffu, v ? key : -1 - lane);
            const int slot = (v ? my_key[key] : 0) + __popc(peers & lt);
            __syncwarp();
            if (v && (peers & lt) == 0) my_key[key] += __popc(peers);
            const bool kept = v && slot < g.c_send;
            const unsigned epeers = __match_any_sync(0xffffffffu, kept ? e[i] : -1 - lane);
            if (kept && (epeers & lt) == 0) my_e[e[i]] += __popc(epeers);
            __syncwarp();
            if (v) {
                const int64_t a = wbase + 32 * i + lane;
                // capped: the pool row; ragged: (block, slot in block), resolved
                // once the block offsets are known
                const int64_t blk = static_cast<int64_t>(key) * g.S + s;
                send_row[first + a] =
                    !kept ? -1 : g.ragged ? (blk << 32) | slot : blk * g.c_send + slot;
                if (!kept) ++dropped;
            }
            kept_mask |= (kept ? 1u : 0u) << i;
        }
        __syncthreads();
        for (int ex = threadIdx.x; ex < g.E; ex += blockDim.x) {
            int acc = run_e[ex];
            for (int w = 0; w < SEND_WARPS; ++w) {
                const int c = cnt_e[w * g.E + ex];
                cnt_e[w * g.E + ex] = acc;
                acc += c;
            }
            run_e[ex] = acc;
        }
        __syncthreads();
        // pass 3: rank among this source's kept rows of the same expert
#pragma unroll
        for (int i = 0; i < SEND_PER_LANE; ++i) {
            if (i * 32 >= per_warp) break;
            const bool kept = kept_mask >> i & 1u;
            const unsigned epeers = __match_any_sync(0xffffffffu, kept ? e[i] : -1 - lane);
            const int r = (kept ? my_e[e[i]] : 0) + __popc(epeers & lt);
            __syncwarp();
            if (kept && (epeers & lt) == 0) my_e[e[i]] += __popc(epeers);
            __syncwarp();
            const int64_t a = wbase + 32 * i + lane;
            if (e[i] >= 0) rloc[first + a] = kept ? r : -1;
        }
        __syncthreads();
    }
    for (int ex = threadIdx.x; ex < g.E; ex += blockDim.x)
        cnt_se[static_cast<int64_t>(s) * g.E + ex] = run_e[ex];
    int maxfill = 0;
    for (int key = threadIdx.x; key < nkey; key += blockDim.x) {
        const int d = run_key[key];
        demand[static_cast<int64_t>(s) * nkey + key] = d;
        maxfill = max(maxfill, min(d, g.c_send));
    }
    for (int off = 16; off > 0; off >>= 1) {
        maxfill = max(maxfill, __shfl_xor_sync(0xffffffffu, maxfill, off));
        dropped += __shfl_xor_sync(0xffffffffu, dropped, off);
    }
    const unsigned any_bad = __ballot_sync(0xffffffffu, bad);
    if (lane == 0) {
        if (dropped)
            atomicAdd(reinterpret_cast<unsigned long long*>(&stats->dropped_send),
                      static_cast<unsigned long long>(dropped));
        atomicMax(&stats->max_send_fill, maxfill);
        if (any_bad) atomicCAS(&stats->status, 0, MOE_EINVAL);
    }
}

// Receiver stage, per expert: exclusive prefix over sources of the kept
// counts (sources hold contiguous token ranges, so source order is priority
// order); count = min(total, c_recv).
__global__ void dispatch_recv_scan_kernel(DispatchGeom g, const int32_t* __restrict__ cnt_se,
                                          int32_t* __restrict__ base_se,
                                          int32_t* __restrict__ expert_count,
                                          moe_drop_stats_t* __restrict__ stats) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    long long kept = 0, over = 0;
    int cnt = 0;
    if (e < g.E) {
        int run = 0;
        for (int s = 0; s < g.S; ++s) {
            base_se[static_cast<int64_t>(s) * g.E + e] = run;
            run += cnt_se[static_cast<int64_t>(s) * g.E + e];
        }
        cnt = min(run, g.c_recv);
        expert_count[e] = cnt;
        kept = cnt;
        over = run - cnt;
    }
    for (int off = 16; off > 0; off >>= 1) {
        kept += __shfl_xor_sync(0xffffffffu, kept, off);
        over += __shfl_xor_sync(0xffffffffu, over, off);
        cnt = max(cnt, __shfl_xor_sync(0xffffffffu, cnt, off));
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(reinterpret_cast<unsigned long long*>(&stats->kept),
                  static_cast<unsigned long long>(kept));
        atomicAdd(reinterpret_cast<unsigned long long*>(&stats->dropped_recv),
                  static_cast<unsigned long long>(over));
        atomicMax(&stats->max_expert_rows, cnt);
    }
}

// Final decisions and the pack, one warp per token (pack_token): the
// token's latent row is read once into registers (16-byte loads) and written
// with 16-byte stores to each of its sender-kept pool rows (all of them, one
// wave's, or none: copy_wave), followed by the row's tag.
template <int CH>   // 16-byte chunks per lane per column block
__global__ void __launch_bounds__(256) dispatch_pack_kernel(
    DispatchGeom g, const uint16_t* __restrict__ z, const int32_t* __restrict__ idx,
    const int64_t* __restrict__ send_row, const int32_t* __restrict__ rloc,
    const int32_t* __restrict__ base_se, uint16_t* __restrict__ pool,
    int32_t* __restrict__ slot_of, uint8_t* __restrict__ drop, int32_t* __restrict__ expert_rows,
    const int32_t* __restrict__ blk_off, const int32_t* __restrict__ eoff, int copy_wave,
    uint16_t* __restrict__ bank) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= g.T) return;
    const PackArgs P{z, idx, send_row, rloc, base_se, pool, slot_of, drop, expert_rows, blk_off, eoff,
                     bank};
    pack_token<CH, false>(g, P, t, lane, true, copy_wave);
}

int launch_dispatch(const DispatchGeom& g, const uint16_t* z, const int32_t* idx, void* ws,
                    uint16_t* pool, int32_t* slot_of, uint8_t* drop, int32_t* expert_rows,
                    int32_t* expert_count, moe_drop_stats_t* stats, cudaStream_t st,
                    int copy_wave, bool run_pack, uint16_t* bank) {
    const DispatchWs L = dispatch_ws_layout(g);
    uint8_t* w = static_cast<uint8_t*>(ws);
    int64_t* send_row = reinterpret_cast<int64_t*>(w + L.send_row_off);
    int32_t* rloc = reinterpret_cast<int32_t*>(w + L.rloc_off);
    int32_t* cnt_se = reinterpret_cast<int32_t*>(w + L.cnt_se_off);
    int32_t* base_se = reinterpret_cast<int32_t*>(w + L.base_se_off);
    int32_t* demand = reinterpret_cast<int32_t*>(w + L.demand_off);
    int32_t* wave_ready = reinterpret_cast<int32_t*>(w + L.wave_ready_off);

    dispatch_init_kernel<<<1024, 256, 0, st>>>(g, pool, expert_rows, stats, wave_ready);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "dispatch_init");
    // per-warp counters plus running totals: (SEND_WARPS + 1) x (D*W + E) ints;
    // D*W <= E <= 1024, so at most 139 KB
    const size_t shm =
        static_cast<size_t>(SEND_WARPS + 1) * (g.D * g.W + g.E) * sizeof(int32_t);
    if (shm > 200 * 1024) return MOE_EINVAL;
    if (shm > 48 * 1024 &&
        ensure_smem_attr(reinterpret_cast<const void*>(dispatch_send_kernel),
                         static_cast<int>(shm)) != MOE_OK)
        return MOE_ECUDA;
    dispatch_send_kernel<<<g.S, SEND_WARPS * 32, shm, st>>>(g, idx, send_row, rloc, cnt_se,
                                                            demand, stats);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "dispatch_send");
    dispatch_recv_scan_kernel<<<(g.E + 127) / 128, 128, 0, st>>>(g, cnt_se, base_se, expert_count,
                                                                  stats);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "dispatch_recv_scan");
    if (g.T == 0 || !run_pack) return MOE_OK;
    const unsigned grid = static_cast<unsigned>((g.T + 7) / 8);
    const int nchunk = g.L / 8;
    if (nchunk <= 32 * 4)
        dispatch_pack_kernel<4><<<grid, 256, 0, st>>>(g, z, idx, send_row, rloc, base_se, pool,
                                                       slot_of, drop, expert_rows, nullptr,
                                                       nullptr, copy_wave, bank);
    else
        dispatch_pack_kernel<12><<<grid, 256, 0, st>>>(g, z, idx, send_row, rloc, base_se, pool,
                                                        slot_of, drop, expert_rows, nullptr,
                                                        nullptr, copy_wave, bank);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "dispatch_pack");
    return MOE_OK;
}

// ==================================================================== ragged offsets

// Exclusive prefix over `n` values read through `get(i)`, written to
// out[0..n] (out[n] = total), by one CTA of 1024 threads in chunks.
template <typename Get>
__device__ void block_exclusive_scan(int n, Get get, int32_t* __restrict__ out) {
    __shared__ int warp_sum[32];
    __shared__ int carry;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += blockDim.x) {
        const int i = i0 + threadIdx.x;
        const int v = i < n ? get(i) : 0;
        int incl = v;
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_sum[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            int ws = lane < static_cast<int>(blockDim.x >> 5) ? warp_sum[lane] : 0;
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, ws, off);
                if (lane >= off) ws += y;
            }
            warp_sum[lane] = ws;
        }
        __syncthreads();
        const int excl = carry + (wid ? warp_sum[wid - 1] : 0) + incl - v;
        if (i < n) out[i] = excl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = excl + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) out[n] = carry;
}

// Ragged pool blocks in (destination, wave, source) order: block b = key*S + s
// holds demand[s][key] rows and starts at the exclusive prefix of the counts;
// expert e's rows start at the prefix of the expert totals.
__global__ void __launch_bounds__(1024) ragged_offsets_kernel(DispatchGeom g,
                                                              const int32_t* __restrict__ demand,
                                                              const int32_t* __restrict__ counts,
                                                              int32_t* __restrict__ blk_off,
                                                              int32_t* __restrict__ eoff) {
    const int nkey = g.D * g.W;
    block_exclusive_scan(nkey * g.S, [&](int b) { return demand[(b % g.S) * nkey + b / g.S]; },
                         blk_off);
    __syncthreads();
    block_exclusive_scan(g.E, [&](int e) { return counts[e]; }, eoff);
}

int launch_dispatch_ragged(const DispatchGeom& g, const uint16_t* z, const int32_t* idx, void* ws,
                           uint16_t* pool, int32_t* slot_of, uint8_t* drop,
                           int32_t* expert_offsets, int32_t* expert_rows, int32_t* expert_count,
                           moe_drop_stats_t* stats, uint16_t* bank, cudaStream_t st,
                           bool run_pack) {
    const DispatchWs L = dispatch_ws_layout(g);
    uint8_t* w = static_cast<uint8_t*>(ws);
    int64_t* send_row = reinterpret_cast<int64_t*>(w + L.send_row_off);
    int32_t* rloc = reinterpret_cast<int32_t*>(w + L.rloc_off);
    int32_t* cnt_se = reinterpret_cast<int32_t*>(w + L.cnt_se_off);
    int32_t* base_se = reinterpret_cast<int32_t*>(w + L.base_se_off);
    int32_t* demand = reinterpret_cast<int32_t*>(w + L.demand_off);
    int32_t* blk_off = reinterpret_cast<int32_t*>(w + L.blk_off_off);
    int32_t* wave_ready = reinterpret_cast<int32_t*>(w + L.wave_ready_off);

    dispatch_init_kernel<<<1, 32, 0, st>>>(g, pool, expert_rows, stats, wave_ready);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "dispatch_init");
    const size_t shm =
        static_cast<size_t>(SEND_WARPS + 1) * (g.D * g.W + g.E) * sizeof(int32_t);
    if (shm > 200 * 1024) return MOE_EINVAL;
    if (shm > 48 * 1024 &&
        ensure_smem_attr(reinterpret_cast<const void*>(dispatch_send_kernel),
                         static_cast<int>(shm)) != MOE_OK)
        return MOE_ECUDA;
    dispatch_send_kernel<<<g.S, SEND_WARPS * 32, shm, st>>>(g, idx, send_row, rloc, cnt_se,
                                                            demand, stats);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "dispatch_send");
    dispatch_recv_scan_kernel<<<(g.E + 127) / 128, 128, 0, st>>>(g, cnt_se, base_se, expert_count,
                                                                  stats);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "dispatch_recv_scan");
    ragged_offsets_kernel<<<1, 1024, 0, st>>>(g, demand, expert_count, blk_off, expert_offsets);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "ragged_offsets");
    if (g.T == 0 || !run_pack) return MOE_OK;
    const unsigned grid = static_cast<unsigned>((g.T + 7) / 8);
    if (g.L / 8 <= 32 * 4)
        dispatch_pack_kernel<4><<<grid, 256, 0, st>>>(g, z, idx, send_row, rloc, base_se, pool,
                                                       slot_of, drop, expert_rows, blk_off,
                                                       expert_offsets, -1, bank);
    else
        dispatch_pack_kernel<12><<<grid, 256, 0, st>>>(g, z, idx, send_row, rloc, base_se, pool,
                                                        slot_of, drop, expert_rows, blk_off,
                                                        expert_offsets, -1, bank);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "dispatch_pack");
    return MOE_OK;
}

// ==================================================================== tile list

// One CTA: per expert ceil(count/bm) row tiles, exclusive prefix over
// experts, entries {e, m0} in expert order.
// wave_El > 0: entries in wave-major order, i.e. the experts of wave 0 on
// every destination (destination by destination), then those of wave 1, ...
// (wave_El local experts a destination, wave_Ew of them a wave).
__global__ void __launch_bounds__(1024) build_tiles_kernel(const int32_t* __restrict__ counts,
                                                           int E, int bm,
                                                           int2* __restrict__ tiles,
                                                           int32_t* __restrict__ tile_count,
                                                           int wave_El, int wave_Ew) {
    __shared__ int warp_sum[32];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int per_wave = wave_El > 0 ? (E / wave_El) * wave_Ew : E;   // experts a wave
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        int e = e0 + threadIdx.x;   // position in the list order
        if (wave_El > 0 && e < E) {
            const int wv = e / per_wave, rem = e - wv * per_wave;
            e = (rem / wave_Ew) * wave_El + wv * wave_Ew + rem % wave_Ew;
        }
        const int mt = e < E ? (counts[e] + bm - 1) / bm : 0;
        int incl = mt;
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_sum[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            int ws = lane < (int)(blockDim.x >> 5) ? warp_sum[lane] : 0;
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, ws, off);
                if (lane >= off) ws += y;
            }
            warp_sum[lane] = ws;
        }
        __syncthreads();
        const int excl = carry + (wid ? warp_sum[wid - 1] : 0) + incl - mt;
        for (int i = 0; i < mt; ++i) tiles[excl + i] = make_int2(e, i * bm);
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = excl + mt;
        __syncthreads();
    }
    if (threadIdx.x == 0) *tile_count = carry;
}

int launch_build_tiles(const int32_t* counts, int E, int bm, int32_t* tile_list,
                       int32_t* tile_count, cudaStream_t st, int wave_El, int wave_Ew) {
    if (wave_El > 0 && (wave_Ew <= 0 || wave_El % wave_Ew || E % wave_El)) return MOE_EINVAL;
    build_tiles_kernel<<<1, 1024, 0, st>>>(counts, E, bm, reinterpret_cast<int2*>(tile_list),
                                           tile_count, wave_El, wave_Ew);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "build_tiles");
    return MOE_OK;
}

// ==================================================================== balancing bias

// Per-expert counts of this batch's top-k selections, added to the caller's
// histogram: a shared-memory histogram per CTA, then one global add per
// expert and CTA (integer adds, so the result does not depend on order).
__global__ void __launch_bounds__(1024) balance_hist_kernel(const int32_t* __restrict__ idx,
                                                            int64_t n, int E,
                                                            unsigned long long* __restrict__ hist) {
    extern __shared__ unsigned int hcount[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hcount[e] = 0;
    __syncthreads();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int e = idx[i];
        if (e >= 0 && e < E) atomicAdd(&hcount[e], 1u);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (hcount[e]) atomicAdd(&hist[e], static_cast<unsigned long long>(hcount[e]));
}

// bias[e] = -alpha * (hist[e] / sum(hist) - 1/E), 0 for an empty histogram.
__global__ void __launch_bounds__(1024) balance_bias_kernel(const int64_t* __restrict__ hist,
                                                            int E, float alpha,
                                                            float* __restrict__ bias) {
    __shared__ long long part[32];
    long long s = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s += hist[e];
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    long long total = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += part[w];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const double f = total > 0 ? static_cast<double>(hist[e]) / static_cast<double>(total)
                                   : 1.0 / E;
        bias[e] = static_cast<float>(-static_cast<double>(alpha) * (f - 1.0 / E));
    }
}

int launch_balance_update(const int32_t* idx, int64_t n, int E, int64_t* hist, float alpha,
                          float* bias, cudaStream_t st) {
    if (n > 0) {
        const int grid = static_cast<int>(std::min<int64_t>((n + 1023) / 1024, 152));
        balance_hist_kernel<<<grid, 1024, E * sizeof(unsigned int), st>>>(
            idx, n, E, reinterpret_cast<unsigned long long*>(hist));
        if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
        trace_after(st, "balance_hist");
    }
    balance_bias_kernel<<<1, 1024, 0, st>>>(hist, E, alpha, bias);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "balance_bias");
    return MOE_OK;
}

// The bias over the past `window` batches, one CTA: this batch's counts
// (shared-memory histogram), the ring row of the batch leaving the window
// swapped for them in H, then the bias as above; the step counter lives on
// the device so that the update needs no host state.
__global__ void __launch_bounds__(1024) balance_window_kernel(
    const int32_t* __restrict__ idx, int64_t n, int E, int64_t* __restrict__ hist,
    int64_t* __restrict__ ring, int window, int64_t* __restrict__ step, float alpha,
    float* __restrict__ bias) {
    extern __shared__ unsigned int cnt[];
    __shared__ long long part[32];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
        const int e = idx[i];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1u);
    }
    __syncthreads();
    const int64_t s = *step;
    int64_t* slot = ring + (s % window) * E;
    long long sum = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const long long h = hist[e] - slot[e] + cnt[e];
        hist[e] = h;
        slot[e] = cnt[e];
        sum += h;
    }
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = sum;
    __syncthreads();
    long long total = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += part[w];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const double f = total > 0 ? static_cast<double>(hist[e]) / static_cast<double>(total)
                                   : 1.0 / E;
        bias[e] = static_cast<float>(-static_cast<double>(alpha) * (f - 1.0 / E));
    }
    if (threadIdx.x == 0) *step = s + 1;   // every thread read it before the barrier above
}

int launch_balance_window(const int32_t* idx, int64_t n, int E, int64_t* hist, int64_t* ring,
                          int window, int64_t* step, float alpha, float* bias, cudaStream_t st) {
    balance_window_kernel<<<1, 1024, E * sizeof(unsigned int), st>>>(idx, n, E, hist, ring, window,
                                                                    step, alpha, bias);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "balance_window");
    return MOE_OK;
}

// ==================================================================== combine

// The return path: c[t] = bf16(sum_j w[t,j] Y[slot_of[t,j]]) over kept j in j
// order, fp32 accumulation, 16-byte loads of the rows.  A warp's unit of
// work is one pass of 32*CH 16-byte chunks of one token's row; the grid
// holds only the blocks that are resident at once and each warp strides over
// the units, so that the last round of work is not left half empty.  Two
// rows' loads are in flight before their products are accumulated.
template <int CH>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ ypool,
                                                      const int32_t* __restrict__ slot_of,
                                                      const float* __restrict__ w, int64_t T,
                                                      int k, int L, uint16_t* __restrict__ c,
                                                      int64_t rows) {
    const int lane = threadIdx.x & 31;
    const int nchunk = L / 8;
    const int npass = (nchunk + 32 * CH - 1) / (32 * CH);
    const int64_t units = T * npass;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         u < units; u += nwarps) {
        const int64_t t = u / npass;
        const int cb = static_cast<int>(u - t * npass) * 32 * CH;
        int32_t my_row = -1;
        float my_w = 0.0f;
        if (lane < k) {
            my_row = slot_of[t * k + lane];
            my_w = w ? w[t * k + lane] : 1.0f;   // no weights: plain sum (gradient return)
            if (!moe_check(my_row < rows, 1003)) my_row = -1;
        }
        float acc[CH][8];
#pragma unroll
        for (int q = 0; q < CH; ++q)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[q][i] = 0.0f;
        auto add = [&](const uint4 (&v)[CH], float wj) {
#pragma unroll
            for (int q = 0; q < CH; ++q) {
                const uint32_t u4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    acc[q][2 * h] = fmaf(wj, bf16_lo(u4[h]), acc[q][2 * h]);
                    acc[q][2 * h + 1] = fmaf(wj, bf16_hi(u4[h]), acc[q][2 * h + 1]);
                }
            }
        };
        auto load = [&](uint4 (&v)[CH], int32_t r) {
            const uint4* src = reinterpret_cast<const uint4*>(ypool + static_cast<int64_t>(r) * L);
#pragma unroll
            for (int q = 0; q < CH; ++q) {
                const int ch = cb + lane + 32 * q;
                v[q] = ch < nchunk ? __ldg(src + ch) : make_uint4(0u, 0u, 0u, 0u);
            }
        };
        for (int j = 0; j < k; j += 2) {
            const int32_t r0 = __shfl_sync(0xffffffffu, my_row, j);
            const float w0 = __shfl_sync(0xffffffffu, my_w, j);
            const int32_t r1 = j + 1 < k ? __shfl_sync(0xffffffffu, my_row, j + 1) : -1;
            const float w1 = j + 1 < k ? __shfl_sync(0xffffffffu, my_w, j + 1) : 0.0f;
            uint4 v0[CH], v1[CH];
            if (r0 >= 0) load(v0, r0);
            if (r1 >= 0) load(v1, r1);
            if (r0 >= 0) add(v0, w0);   // dropped assignments add nothing
            if (r1 >= 0) add(v1, w1);
        }
        uint4* dst = reinterpret_cast<uint4*>(c + t * L);
#pragma unroll
        for (int q = 0; q < CH; ++q) {
            const int ch = cb + lane + 32 * q;
            if (ch < nchunk)
                dst[ch] = make_uint4(pack_bf16x2(acc[q][0], acc[q][1]),
                                     pack_bf16x2(acc[q][2], acc[q][3]),
                                     pack_bf16x2(acc[q][4], acc[q][5]),
                                     pack_bf16x2(acc[q][6], acc[q][7]));
        }
    }
}

int check_status_route() { return moe_check_read_reset(); }

int launch_combine(const uint16_t* ypool, const int32_t* slot_of, const float* w, int64_t T, int k,
                   int L, uint16_t* c, int64_t rows, cudaStream_t st) {
    if (T == 0) return MOE_OK;
    int dev, sms;
    int rc = current_device(&dev, &sms);
    if (rc) return rc;
    // resident blocks of each instance (queried once; no runtime call inside
    // a stream capture after the first launch)
    static int per_sm[2] = {0, 0};
    const bool wide = L / 8 > 32 * 4;
    if (!per_sm[wide]) {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &nb, wide ? combine_kernel<6> : combine_kernel<4>, 256, 0) != cudaSuccess)
            return MOE_ECUDA;
        per_sm[wide] = nb > 0 ? nb : 1;
    }
    const int ch = wide ? 6 : 4;
    const int64_t units = T * ((L / 8 + 32 * ch - 1) / (32 * ch));
    const int64_t need = (units + 7) / 8;   // blocks of 8 warps, one unit each
    const int64_t most = static_cast<int64_t>(sms) * per_sm[wide];
    const unsigned grid = static_cast<unsigned>(need < most ? need : most);
    if (wide)
        combine_kernel<6><<<grid, 256, 0, st>>>(ypool, slot_of, w, T, k, L, c, rows);
    else
        combine_kernel<4><<<grid, 256, 0, st>>>(ypool, slot_of, w, T, k, L, c, rows);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "combine");
    return MOE_OK;
}

}  // namespace moe
