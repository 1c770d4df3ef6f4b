// internal.h -- host-side interfaces between the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moe_pooled_wave.h"

namespace moe {

// ---------------------------------------------------------------- device

// Checks that the current device is an sm_103 part and returns its SM count.
int current_device(int* device, int* num_sms);

// Raises a kernel's dynamic shared-memory limit on the current device to at
// least `bytes`, calling the runtime only the first time a larger value is
// needed (so that launches inside a stream capture make no such call).
int ensure_smem_attr(const void* func, int bytes);

// Kernel timing trace: after each launch the library calls trace_after(),
// which records the next trace event on that stream when tracing is on.
void trace_after(cudaStream_t stream, const char* kernel_name);

// ---------------------------------------------------------------- GEMM engine

enum AMode : int {
    A_DENSE = 0,    // A [M, K] row-major, TMA 2D tiles
    A_GROUPED = 1,  // A [G, rows, K], TMA 3D tiles (group = expert)
    A_GATHER = 2,   // A rows gathered by index from a pitched row store (cp.async)
};

enum EpiMode : int {
    EPI_F32 = 0,      // fp32 out (+ optional per-column bias)
    EPI_BF16 = 1,     // bf16 out
    EPI_SWIGLU = 2,   // accumulator = [gate | up] halves -> bf16(silu(gate) * up)
    EPI_SCATTER = 3,  // bf16 out to rows given by a row map
    EPI_SPLIT = 4,    // column tiles < nsplit: bf16 out (B = seg 0); the rest: fp32
                      // out2 + bias (B = B_up), e.g. latent projection + router
    EPI_SWIGLU_BWD = 5,  // accumulator = [gate | up] (recomputed); with the incoming
                         // gradient dh (aux, bf16): out = dh u silu'(g), out2 = dh silu(g)
};

struct GemmSeg {        // one K segment of the contraction: A_s [M, K_s] . B_s [N, K_s]^T
    const void* A;      // bf16
    int64_t lda;        // elements between A rows
    const void* B;      // bf16
    int64_t ldb;        // elements between B rows
    int K;
};

struct DispatchGeom {
    int64_t T;
    int k, E, S, D, W, E_l, E_w, L;
    int64_t T_s;
    int c_send, c_recv;
    int64_t pool_rows;
    int ragged;   // 1: dropless ragged layout (no caps, pool of T*k rows)
};

// Pointers of one dispatch's pack: what pack_token (pack.cuh) reads and writes.
struct PackArgs {
    const uint16_t* z;          // [T, L] latent rows
    const int32_t* idx;         // [T, k] expert ids
    const int64_t* send_row;    // [T, k] sender-kept pool row (ragged: block | offset), else -1
    const int32_t* rloc;        // [T, k] rank among the source's kept rows of its expert
    const int32_t* base_se;     // [S, E] first receiver rank of each source's rows
    uint16_t* pool;             // [pool_rows, pitch]
    int32_t* slot_of;           // [T, k]
    uint8_t* drop;              // [T, k]
    int32_t* expert_rows;       // [E, c_recv] (ragged: flat, eoff)
    const int32_t* blk_off;     // ragged: first row of each (source, destination, wave) block
    const int32_t* eoff;        // ragged: first row-list entry of each expert
    uint16_t* bank;             // optional [E, c_recv, L]: receiver-kept rows grouped by expert
};

// out = sum_s A_s B_s^T with one of the epilogues above.  For EPI_SWIGLU the
// B operand of segment 0 is the gate weight and B_up the up weight (same
// shape); N then counts hidden units.  Grouped modes take the tile list
// (int2 {group, m0}) and its length from device memory.
struct GemmDesc {
    int a_mode;
    int epi;
    int a_mn;               // 1: A stored [K, M] (M contiguous) instead of [M, K]
    int b_mn;               // 1: B stored [K, N] instead of [N, K]
    int bn;                 // 128, 256, or 384 (fp32 epilogue only: two MMAs, N=256+128)
    int64_t M;              // dense: rows of A/out
    int N;                  // output columns (hidden units for SWIGLU)
    int nseg;
    GemmSeg seg[4];
    const void* B_up;
    // grouped geometry
    int groups;
    int rows_per_group;     // rows of one group in a grouped A / in the row map
    int64_t a_gstride;      // elements between groups of A (A_GROUPED)
    int64_t b_gstride;      // elements between groups of B (and B_up)
    int b_rows;             // rows of one group's B (N extent of the weight)
    const int32_t* tile_list;
    const int32_t* tile_count;
    int max_tiles;          // upper bound of the tile list length
    const int32_t* rowmap;  // [groups, rowmap_ld], or flat with goff
    const int32_t* counts;  // [groups]
    const int32_t* goff;    // optional [groups]: first row of each group in a flat
                            // (ragged) row map, grouped A and grouped SwiGLU output
    int rowmap_ld;
    const uint16_t* gather_src;
    int64_t gather_pitch;   // elements between gathered rows
    int64_t gather_rows;    // rows in the gather source
    // epilogue
    void* out;
    int64_t ldo;
    int64_t out_gstride;    // elements between groups of out (grouped SWIGLU)
    const float* bias;
    int32_t* status;
    const char* name;       // kernel name for the timing trace
    const void* aux;        // EPI_SWIGLU_BWD: incoming gradient, addressed like out
    int uniform_groups;     // > 0: grouped tiles over `groups` groups of M rows each
                            // (no tile list), e.g. per-expert weight gradients
    const int32_t* rmoff;   // optional [groups]: first entry of each group in the row
                            // map, when it differs from goff (row gather, scatter)
    const int32_t* kgoff;   // optional [groups + 1] with uniform_groups: group g
                            // contracts over rows kgoff[g] .. kgoff[g+1] (multiples of
                            // 64) of MN-major operands stored flat; an empty range
                            // writes a zero tile
    int64_t k_rows;         // rows of those flat operands
    const int32_t* kcount;  // optional [groups] with uniform_groups (3-D grouped operands whose
                            // rows past each group's count are zero): group g contracts over
                            // its first ceil(kcount[g] / 64) blocks of 64 rows only
    // EPI_SPLIT: second output (EPI_SWIGLU_BWD: out2 = du, addressed like out)
    int nsplit;             // column tiles of the first output (N = nsplit * bn)
    int N2;                 // columns of the second output
    void* out2;
    int64_t ldo2;
    int b2_rows;            // rows of the second B (B_up)
    // pool fill riding along a GEMM launch (the pack's PackArgs non-null).
    // Wave pipeline (gathered A, wp_ready non-null): extra warps copy the
    // payload rows and tags of waves 1..W-1 into the pool (gather_src) while
    // the launch computes; the row gather of a wave-w tile waits until every
    // CTA has counted wave w in wp_ready[w] (a cooperative launch of one CTA
    // per SM).  Dense products (wp_ready null): extra warps run the whole
    // pack (decisions and every copy), which nothing in the launch waits for.
    int32_t* wp_ready;      // [W] counters, zero at launch
    DispatchGeom wp_g;
    PackArgs wp_a;
};

int gemm_launch(const GemmDesc& d, cudaStream_t stream);

// ---------------------------------------------------------------- routing kernels

int launch_topk(const float* logits, int64_t T, int E, int k, int32_t* idx, float* w,
                uint8_t* tie, cudaStream_t stream);

// Pool row: L bf16 payload, the 16-byte tag, padding to a multiple of 128
// bytes, so that every row (and every 64-element K segment of it) starts on a
// cache-line boundary for the expert GEMM's row gather.  In uint16 elements.
__host__ __device__ inline int64_t pool_pitch(int L) { return ((2ll * L + 16 + 127) / 128 * 128) / 2; }

// Scratch layout of moe_dispatch_pooled (and of the ragged dispatch, which
// adds the block offsets).
struct DispatchWs {
    size_t send_row_off, rloc_off, cnt_se_off, base_se_off, demand_off, blk_off_off,
        wave_ready_off, total;
};
DispatchWs dispatch_ws_layout(const DispatchGeom& g);

// copy_wave >= 0: every decision is made, but only the payload rows (and
// tags) of that wave are written; -1: all.  run_pack false: the sender and
// receiver counts only, the pack (decisions and copies) left to a GEMM
// launch that carries it.
// bank (optional, [E, c_recv, L]): the pack also writes each receiver-kept
// row there, at its expert's receiver rank.
int launch_dispatch(const DispatchGeom& g, const uint16_t* z, const int32_t* idx, void* ws,
                    uint16_t* pool, int32_t* slot_of, uint8_t* drop, int32_t* expert_rows,
                    int32_t* expert_count, moe_drop_stats_t* stats, cudaStream_t stream,
                    int copy_wave = -1, bool run_pack = true, uint16_t* bank = nullptr);

// bank (optional): [T*k, L], each row also written at its position in the
// flat expert row list.  run_pack = false stops after the offsets (the pack
// then runs inside the shared experts' gate/up launch).
int launch_dispatch_ragged(const DispatchGeom& g, const uint16_t* z, const int32_t* idx, void* ws,
                           uint16_t* pool, int32_t* slot_of, uint8_t* drop,
                           int32_t* expert_offsets, int32_t* expert_rows, int32_t* expert_count,
                           moe_drop_stats_t* stats, uint16_t* bank, cudaStream_t stream,
                           bool run_pack = true);

// The capped layout's expert FFN on CTA pairs with the expert's rows on the
// MMA's N axis (expert_pair.cu): chunk list, gate/up from the per-expert
// bank into h [E, c_recv, H], down from h scattered to the pool rows of
// ypool.  chunk_ws: expert_pair_chunks_bytes(E, c_recv), 16-byte aligned.
size_t expert_pair_chunks_bytes(int E, int c_recv);
int expert_ffn_pair(int E, int c_recv, int L, int H, const uint16_t* bank,
                    const int32_t* expert_rows, const int32_t* expert_count, const uint16_t* Wg,
                    const uint16_t* Wu, const uint16_t* Wd, void* chunk_ws, uint16_t* h,
                    uint16_t* ypool, int64_t pool_rows, int32_t* status, cudaStream_t stream);
int check_status_expert_pair();

// The dropless layout's expert FFN on CTA pairs over row groups
// (expert_pair.cu): gate/up from the flat bank [rows, L] (expert e's rows at
// expert_offsets[e]) into the flat h [rows, H], down from h scattered to the
// pool rows of ypool (expert_rows, flat).  list_ws:
// expert_pair_lists_bytes_ragged(E, rows), 16-byte aligned.  MOE_EINVAL,
// having enqueued nothing, when the widths or tensors do not allow it.
size_t expert_pair_lists_bytes_ragged(int E, int64_t rows);
int expert_ffn_pair_ragged(int E, int64_t rows, int L, int H, const uint16_t* bank,
                           const int32_t* expert_offsets, const int32_t* expert_rows,
                           const int32_t* expert_count, const uint16_t* Wg, const uint16_t* Wu,
                           const uint16_t* Wd, void* list_ws, uint16_t* h, uint16_t* ypool,
                           int32_t* status, cudaStream_t stream);

// The routed experts' products of the backward over row groups on CTA pairs
// (expert_pair.cu), capped layout, per-expert row layouts [E, c_recv, .]:
//  expert_group_list: the row groups of every expert from expert_count, in
//    `ws` (expert_pair_chunks_bytes(E, c_recv) bytes, 16-byte aligned; kept
//    until the products below have run);
//  expert_dh_group: dh = dY Wd_e (dY rows from dye, zero past each count);
//  expert_swiglu_bwd_group: g, u recomputed from X (xe), dg = dh u silu'(g),
//    du = dh silu(g), each expert's first expert_count rows (the rest
//    untouched);
//  expert_dx_group: dX = dg Wg_e + du Wu_e, each row to its pool row of
//    dxpool (expert_rows).
// The dropless layout (roff given, c_recv ignored): the per-expert buffers
// are flat [rows, .] with expert e's rows from row roff[e] (padded to whole
// 64-row blocks), the group list from expert_group_list_ragged (its `ws`:
// expert_pair_lists_bytes_ragged(E, kept rows) bytes), and dX's row list is
// the flat one with expert e's entries from rmoff[e].
// Each returns MOE_EINVAL, having enqueued nothing, when the widths or the
// tensors do not allow its path (the caller then takes the grouped GEMM).
struct ExpertGroups {
    const int4* groups;
    const int32_t* ngroups;
};
int expert_group_list(int E, int c_recv, const int32_t* expert_count, void* ws, ExpertGroups* out,
                      cudaStream_t stream);
int expert_group_list_ragged(int E, int64_t rows, const int32_t* expert_count, void* ws,
                             ExpertGroups* out, cudaStream_t stream);
int expert_dh_group(int E, int c_recv, int L, int H, const uint16_t* dye, const uint16_t* Wd,
                    const ExpertGroups& groups, uint16_t* dh, int32_t* status, cudaStream_t stream,
                    const int32_t* roff = nullptr, int64_t rows = 0);
int expert_swiglu_bwd_group(int E, int c_recv, int L, int H, const uint16_t* xe,
                            const uint16_t* Wg, const uint16_t* Wu, const uint16_t* dh,
                            const ExpertGroups& groups, uint16_t* dg, uint16_t* du,
                            int32_t* status, cudaStream_t stream, const int32_t* roff = nullptr,
                            int64_t rows = 0);
int expert_dx_group(int E, int c_recv, int L, int H, const uint16_t* dg, const uint16_t* du,
                    const uint16_t* Wg, const uint16_t* Wu, const ExpertGroups& groups,
                    const int32_t* expert_rows, uint16_t* dxpool, int64_t pool_rows,
                    int32_t* status, cudaStream_t stream, const int32_t* roff = nullptr,
                    int64_t rows = 0, const int32_t* rmoff = nullptr);

// Tile list {expert, m0} of the grouped expert GEMMs, from the expert counts.
// Checked builds: the site code recorded by each translation unit's index
// checks since the last call (0: none), reset on reading.
int check_status_route();
int check_status_gemm();
// Checked builds: the limit of the wave pipeline's cross-CTA wait (MOE_EINVAL otherwise).
int set_wave_wait_limit(unsigned long long ns);
int check_status_backward();

// wave_El > 0: wave-major entry order (wave_El local experts a destination,
// wave_Ew a wave); else expert order.
int launch_build_tiles(const int32_t* counts, int E, int bm, int32_t* tile_list,
                       int32_t* tile_count, cudaStream_t stream, int wave_El = 0,
                       int wave_Ew = 0);

// Backward pass: scratch layout (byte offsets) and launch sequence.
struct BackwardWs {
    size_t dc, da, dgs, dus, dw, rowinv, dxpool, dh, dg, du, xe, dye, dz, dlogits, tiles, hp, poff,
        total;
};
BackwardWs backward_ws_layout(const DispatchGeom& g, int d, int H, int Hs, int ns);
int launch_backward(const DispatchGeom& g, int d, int H, int Hs, int ns,
                    const moe_backward_args_t& a, cudaStream_t stream);

// Quantile-balancing bias update: hist += counts of idx; bias from hist.
int launch_balance_update(const int32_t* idx, int64_t n, int E, int64_t* hist, float alpha,
                          float* bias, cudaStream_t stream);
int launch_balance_window(const int32_t* idx, int64_t n, int E, int64_t* hist, int64_t* ring,
                          int window, int64_t* step, float alpha, float* bias, cudaStream_t st);

// c[t] = bf16(sum over kept j of w[t,j] ypool[slot_of[t,j]]); w == nullptr: weights 1.
int launch_combine(const uint16_t* ypool, const int32_t* slot_of, const float* w, int64_t T, int k,
                   int L, uint16_t* c, int64_t rows, cudaStream_t stream);

}  // namespace moe
