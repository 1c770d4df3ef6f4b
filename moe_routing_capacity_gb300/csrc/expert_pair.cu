// expert_pair.cu -- the routed experts' two products on CTA pairs, with an
// expert's received rows on the MMA's N axis.
//
//   gate/up:  [Wg_e ; Wu_e] . X_e^T  ->  h_e = bf16(silu(g) * u)
//   down:     Wd_e . h_e^T           ->  Y = bf16(.), each row scattered to its pool row
//
// The weight rows sit on M: a pair tile is 256 weight rows, 128 staged by each
// CTA of a two-CTA cluster (tcgen05.mma.cta_group::2, issued by the even
// CTA).  For gate/up a CTA's 128 rows are the gate and the up rows of the
// same 64 hidden units, so its SwiGLU epilogue needs only its own TMEM.  The
// expert's rows sit on N in chunks of at most 256 rows (an M x N x 16 MMA
// costs N/2 cycles for N >= 128, measured on this part), sized evenly over
// the expert's count and rounded up to 16, each CTA staging half of them.
// Both operands arrive by TMA: the weights from their [E, rows, K] tensors,
// the expert's rows from a per-expert bank [E, c_recv, K] (the received rows
// grouped by local expert, written by the dispatch's pack; for the down
// product, h itself).  Bank rows past an expert's count hold stale values:
// each one reaches only its own column of the accumulator, which the
// epilogue never stores.
//
// Two kernels:
//  * expert_group_kernel (both products): a tile is a group of up to 416 of
//    an expert's rows in one or two chunks that share each weight block
//    staged in shared memory; see its section below.
//  * expert_pair_kernel: a tile is one chunk, two accumulators of 256
//    columns in turn; gate/up when the two weight tensors cannot share one
//    tensor map, and either product when built with MOE_XPAIR_TM=0 or
//    MOE_XPAIR_DGROUP=0.
// Warp roles per CTA: 0 TMA producer, 1 MMA issuer (even CTA) or the wait
// for the pair's last MMA (odd CTA), 2 TMEM allocation, 4 and up epilogue.
// expert_pair_kernel's epilogue moves each 32-column block of its
// accumulator through shared memory (gate/up: fp32 across the four warps,
// 132 floats a column; down: bf16 within each warp, 64 bytes a row; both free
// of bank conflicts), then each thread writes whole 16- or 32-byte pieces of
// one output row.
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int XBK = 64;                              // K block: one 128-byte swizzle row
constexpr int XA_BYTES = 128 * XBK * 2;              // this CTA's weight rows: 16 KB
constexpr int XB_ROWS = 128;                         // this CTA's half of at most 256 rows
constexpr int XB_BYTES = XB_ROWS * XBK * 2;          // 16 KB
constexpr int XSTAGE = XA_BYTES + XB_BYTES;          // 32 KB a ring stage
#ifndef MOE_XPAIR_STAGES
#define MOE_XPAIR_STAGES 6
#endif
constexpr int XST = MOE_XPAIR_STAGES;
constexpr int XSTG_LD = 132;                         // gate/up: floats a staged column
constexpr int XSTG_BYTES = 32 * XSTG_LD * 4;           // (down: 4 warps x 32 x 32 bf16, less)
constexpr int XBAR_BYTES = ((2 * XST + 5) * 8 + 2 * 4 + 63) / 64 * 64;
constexpr int XSMEM = 1024 + XST * XSTAGE + XSTG_BYTES + XBAR_BYTES;
static_assert(XSMEM <= 232448, "shared memory budget");
constexpr int XCHUNK = 256;                          // most rows a chunk (the MMA's N)
#ifndef MOE_XPAIR_GRAN
#define MOE_XPAIR_GRAN 16
#endif
constexpr int XGRAN = MOE_XPAIR_GRAN;                // chunk N: a multiple of this (N/2 rows a CTA)
static_assert(XGRAN == 16 || XGRAN == 32, "chunk granularity");
// A CTA loads its half of a chunk (XGRAN/2 .. 128 rows, a multiple of
// XGRAN/2, whole 8-row swizzle atoms) with one box of exactly that height:
// one tensor map per height.  Every extra box a stage costs the TMA unit
// time, every row loaded but not used costs shared-memory bandwidth.
constexpr int XHSTEP = XGRAN / 2;
constexpr int XNMAP = XB_ROWS / XHSTEP;
// gate/up over row groups (expert_group_kernel); 0: the chunk-tile kernel
#ifndef MOE_XPAIR_TM
#define MOE_XPAIR_TM 1
#endif
static_assert(!MOE_XPAIR_TM || XGRAN == 16, "gate/up groups split into halves of 16-row multiples");

struct XParams {
    CUtensorMap mapW0;     // gate/up: Wg [E, H, L], box {64, 64} (or, wpair, both: see below);
                           // down: Wd [E, L, H], box {64, 128}
    CUtensorMap mapW1;     // gate/up: Wu [E, H, L], box {64, 64}
    CUtensorMap mapX[XNMAP];   // the rows: bank [E, c_recv, L] or h [E, c_recv, H], box {64, XHSTEP (i+1)}
    const int4* chunks;    // {expert, first row, rows, N}
    const int* nchunks;
    int n_mb;              // 256-row weight blocks a chunk (gate/up: H / 128; down: L / 256)
    int wpair;             // gate/up: mapW0 is [2][E*H/64][64][L] over the lower-addressed of
                           // Wg, Wu and the other, one box {64, 64, 1, 2} fetching both halves
    int gate_hi;           // gate/up: the gate rows are the second half (Wu below Wg)
    int hblk;              // gate/up: H / 64
    int kb;                // K blocks
    int c_recv;
    uint16_t* out;         // h [E, c_recv, H] (gate/up) or ypool [pool_rows, L] (down)
    long long ldo;         // H or L
    const int* rowmap;     // down: expert_rows [E, c_recv]
    long long out_rows;    // down: pool rows (checked builds)
    int* status;
};

template <int EPI>
__global__ void __launch_bounds__(256, 1) expert_pair_kernel(const __grid_constant__ XParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sbase = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sStage = sbase;                                        // XST x (A 16 KB | B 16 KB)
    float* stg = reinterpret_cast<float*>(sbase + XST * XSTAGE);    // epilogue staging
    uint64_t* bars = reinterpret_cast<uint64_t*>(sbase + XST * XSTAGE + XSTG_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = full + XST;
    uint64_t* tfull = empty + XST;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const bool leader = crank == 0;
    const int pair = static_cast<int>(blockIdx.x >> 1);
    const int npairs = static_cast<int>(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < XST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 256);   // both CTAs' 128 epilogue threads
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&p.mapW0);
        if (EPI == EPI_SWIGLU && !p.wpair) tma_prefetch_map(&p.mapW1);
        for (int i = 0; i < XNMAP; ++i) tma_prefetch_map(&p.mapX[i]);
    }
    if (warp == 2) {
        tmem_alloc_pair(tmem_slot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();   // the peer's barriers exist before any remote arrival
    const uint32_t tmem_base = *tmem_slot;
    const int ntiles = *reinterpret_cast<const volatile int*>(p.nchunks) * p.n_mb;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t s = 0, ph = 0;
            uint32_t armed = 0, par = 0;   // stages armed by the even CTA (for unwinding)
            bool ok = true;
            for (int tile = pair; ok && tile < ntiles; tile += npairs) {
                const int ci = tile / p.n_mb;
                const int mb = tile - ci * p.n_mb;
                const int4 ch = p.chunks[ci];
                const int e = ch.x, half = ch.w >> 1;
                const int xrow = ch.y + static_cast<int>(crank) * half;   // this CTA's first row
                const CUtensorMap* xmap = &p.mapX[half / XHSTEP - 1];
                const uint32_t bytes = XA_BYTES + static_cast<uint32_t>(half) * XBK * 2;
                for (int kb = 0; kb < p.kb; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    if (leader) {
                        mbar_arrive_expect_tx(&full[s], 2u * bytes);
                        armed |= 1u << s;
                        par = (par & ~(1u << s)) | (ph << s);
                    }
                    const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
                    const uint32_t a_dst = smem_u32(sStage + s * XSTAGE);
                    const uint32_t b_dst = a_dst + XA_BYTES;
                    const int kx = kb * XBK;
                    if (EPI == EPI_SWIGLU) {   // gate then up rows of 64 hidden units
                        const int u = mb * 128 + static_cast<int>(crank) * 64;
                        if (p.wpair) {
                            tma_load_4d_pair(a_dst, &p.mapW0, fb, kx, 0, e * p.hblk + u / 64, 0);
                        } else {
                            tma_load_3d_pair(a_dst, &p.mapW0, fb, kx, u, e);
                            tma_load_3d_pair(a_dst + XA_BYTES / 2, &p.mapW1, fb, kx, u, e);
                        }
                    } else {                   // 128 output features
                        tma_load_3d_pair(a_dst, &p.mapW0, fb, kx,
                                         mb * 256 + static_cast<int>(crank) * 128, e);
                    }
                    tma_load_3d_pair(b_dst, xmap, fb, kx, xrow, e);
                    if (++s == XST) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok || *abort_flag) {
                // Unwinding: every armed stage's loads (both CTAs') land before
                // the pair may exit.
                volatile int no_abort = 0;
                for (int i = 0; i < XST; ++i)
                    if (armed >> i & 1u)
                        mbar_wait(&full[i], (par >> i) & 1u, &no_abort, nullptr, 20000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && !leader) {
            // the even CTA issues the pair's MMAs, which read this CTA's shared
            // memory and write its TMEM: wait until the last one is done
            volatile int no_abort = 0;
            mbar_wait(done, 0, &no_abort, p.status);
        } else if (lane == 0) {
            uint32_t s = 0, ph = 0, acc = 0, acc_ph = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < ntiles; tile += npairs) {
                const int4 ch = p.chunks[tile / p.n_mb];
                const uint32_t idesc = idesc_bf16_f32(256, ch.w);
                if (!mbar_wait(&tempty[acc], acc_ph ^ 1u, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * 256;
                for (int kb = 0; kb < p.kb; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_s = smem_u32(sStage + s * XSTAGE);
                    const uint64_t ad = sdesc_k_sw128(a_s);
                    const uint64_t bd = sdesc_k_sw128(a_s + XA_BYTES);
#pragma unroll
                    for (int kk = 0; kk < XBK / 16; ++kk)
                        mma_bf16_pair(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc,
                                      (kb | kk) != 0 ? 1u : 0u);
                    mma_commit_pair(&empty[s]);   // the stage is free in both CTAs
                    if (++s == XST) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_ph ^= 1u;
                }
            }
            // every MMA issued must finish before either CTA releases TMEM
            mma_commit_pair(done);
            volatile int no_abort = 0;
            mbar_wait(done, 0, &no_abort, p.status);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp - 4;
        const int t = threadIdx.x - 128;          // 0..127
        const uint32_t tempty_c0 = mapa_shared(smem_u32(&tempty[0]), 0);
        uint32_t acc = 0, acc_ph = 0;
        for (int tile = pair; tile < ntiles; tile += npairs) {
            const int ci = tile / p.n_mb;
            const int mb = tile - ci * p.n_mb;
            const int4 ch = p.chunks[ci];
            const int e = ch.x, row0 = ch.y, nrows = ch.z, N = ch.w;
            if (EPI == EPI_SWIGLU) {
                if (!mbar_wait(&tfull[acc], acc_ph, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * 256;
                // gate rows at lanes go .. go+63, up rows at uo .. uo+63
                const int go = p.gate_hi ? 64 : 0, uo = 64 - go;
#pragma unroll 1
                for (int c0 = 0; c0 < N; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tl + c0, r);
                    // column j of this block, TMEM lane 32q + lane
#pragma unroll
                    for (int j = 0; j < 32; ++j) stg[j * XSTG_LD + q * 32 + lane] = __uint_as_float(r[j]);
                    named_bar_sync(1, 128);
                    // thread t: row j = t % 32 of the block, units 16 (t / 32) .. +15
                    const int j = t & 31, grp = t >> 5;
                    const int rr = c0 + j;            // row within the chunk
                    if (rr < nrows) {
                        const float* col = stg + j * XSTG_LD;
                        uint32_t pk[8];
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const float4 g4 = *reinterpret_cast<const float4*>(col + go + 16 * grp + 4 * v);
                            const float4 u4 = *reinterpret_cast<const float4*>(col + uo + 16 * grp + 4 * v);
                            pk[2 * v] = pack_bf16x2(silu_fast(g4.x) * u4.x, silu_fast(g4.y) * u4.y);
                            pk[2 * v + 1] = pack_bf16x2(silu_fast(g4.z) * u4.z, silu_fast(g4.w) * u4.w);
                        }
                        const long long hrow = static_cast<long long>(e) * p.c_recv + row0 + rr;
                        uint16_t* dst = p.out + hrow * p.ldo + mb * 128 +
                                        static_cast<int>(crank) * 64 + 16 * grp;
                        *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        *reinterpret_cast<uint4*>(dst + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                    named_bar_sync(1, 128);   // the staging is rewritten by the next block
                }
            } else {
                // The pool row of each of the tile's rows, loaded before the
                // accumulator is ready: lane j holds rows j, 32 + j, ...
                long long prow[XCHUNK / 32];
#pragma unroll
                for (int c = 0; c < XCHUNK / 32; ++c) {
                    const int rr = 32 * c + lane;
                    prow[c] = -1;
                    if (rr < nrows) {
                        const long long v =
                            p.rowmap[static_cast<long long>(e) * p.c_recv + row0 + rr];
                        if (moe_check(v >= 0 && v < p.out_rows, 1101)) prow[c] = v;
                    }
                }
                if (!mbar_wait(&tfull[acc], acc_ph, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * 256;
                // each warp transposes its own 32 features x 32 rows through
                // its part of the staging, already rounded to bf16 (the
                // output's rounding): row-major, 64 bytes a row
                uint16_t* w = reinterpret_cast<uint16_t*>(stg) + q * 32 * 32;
                uint16_t* obase = p.out + mb * 256 + static_cast<int>(crank) * 128 + 32 * q;
#pragma unroll
                for (int c = 0; c < XCHUNK / 32; ++c) {
                    if (32 * c < N) {                 // warp-uniform
                        uint32_t r[32];
                        tmem_ld32(tl + 32 * c, r);    // feature 32q + lane, rows 32c ..
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            w[j * 32 + lane] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[j])));
                        __syncwarp();
                        // four lanes a row, 16 bytes (8 features) each: one
                        // store instruction writes 8 rows x 64 contiguous bytes
                        const int sub = lane & 3;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int j = 8 * i + (lane >> 2);     // row 32c + j
                            const long long pr = __shfl_sync(0xffffffffu, prow[c], j);
                            const uint4 y = *reinterpret_cast<const uint4*>(w + j * 32 + 8 * sub);
                            if (pr >= 0) *reinterpret_cast<uint4*>(obase + pr * p.ldo + 8 * sub) = y;
                        }
                        __syncwarp();                 // before the next block overwrites w
                    }
                }
            }
            tc_fence_before();
            mbar_arrive_cluster_relaxed(tempty_c0 + acc * 8u);
            if (++acc == 2) {
                acc = 0;
                acc_ph ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // neither CTA leaves while the other may still arrive on its barriers or
    // the pair's MMAs may touch its memory
    cluster_sync();
    if (warp == 2) tmem_dealloc_pair(tmem_base, 512);
}

// ---------------------------------------------------------------- both products over row groups
//
// With one tile a chunk, an expert's second chunk streams the same 48 weight
// blocks through shared memory again: at N = 160 a CTA's shared memory moves
// 52 KB a K block (TMA writes and MMA reads of 16 KB of weights and 10 KB of
// rows) for 320 MMA cycles, more than it sustains.  Here a tile is a group of
// up to 416 of an expert's rows in one or two chunks (an MMA's N is at most
// 256): each weight block is loaded once and read by both chunks' MMAs, 36 KB
// written and 52 KB read a K block for 640 MMA cycles.
//
// A group's accumulator takes S = N0 + N1 TMEM columns.  Consecutive tiles of
// a CTA pair sit at the two ends of the 512 columns (even tiles from column
// 0, odd tiles ending at column 511, every start a multiple of 32), so the
// next tile's MMAs start while the previous tile drains unless the two
// overlap; then the epilogue drains the overlapping columns first (both
// warp groups, from the end facing the other tile) and releases them before
// the rest.  The MMA issuer waits for the overlap of the tile before and for
// the whole of the tile two before (the same end).
//
// Gate/up (forward, and its recomputation in the backward): a CTA's 128
// weight rows arrive by one TMA box that interleaves the two tensors by 16
// rows: lanes 32q .. 32q+15 hold 16 hidden units of the lower-addressed
// tensor, lanes 32q+16 .. 32q+31 the same units of the other, so a lane's
// SwiGLU partner is lane ^ 16 of its own warp (one shuffle, no shared-memory
// exchange); the forward writes h, the backward reads dh and writes dg, du.
// Scatter (the forward's down product; the backward's dh and dX): a CTA's
// 128 weight rows are 128 output features; lanes pair adjacent features by a
// shuffle into 32-bit stores to each row's output row (its pool row, or its
// row of the per-expert layout).  The backward's products read their weights
// MN-major (stored [K, M]), dX's K in two segments (gate, then up).  Sixteen
// epilogue warps, four a lane quarter, take every fourth 32-column block, so
// the columns the next tile needs drain in a quarter of the blocks' time.
constexpr int GACC = 416;                      // most rows (accumulator columns) a group
constexpr int GB_BYTES = GACC / 2 * XBK * 2;   // this CTA's rows a stage: at most 208
constexpr int GSTAGE = XA_BYTES + GB_BYTES;    // 42 KB
#ifndef MOE_XGATE_STAGES
#define MOE_XGATE_STAGES 5
#endif
constexpr int GST = MOE_XGATE_STAGES;
constexpr int GBAR_BYTES = ((2 * GST + 7) * 8 + 2 * 4 + 63) / 64 * 64;
constexpr int GSMEM = 1024 + GST * GSTAGE + GBAR_BYTES;
static_assert(GSMEM <= 232448, "shared memory budget");
constexpr int GEPI_WARPS = 16;                    // epilogue warps, GEPQ a TMEM lane quarter
constexpr int GEPQ = GEPI_WARPS / 4;
static_assert(GEPI_WARPS % 4 == 0, "whole lane quarters");
constexpr int GMAXB = (GACC / 32 + GEPQ - 1) / GEPQ;   // most 32-column blocks a warp drains a tile
constexpr int GTHREADS = 128 + 32 * GEPI_WARPS;

struct GParams {
    CUtensorMap mapW;          // gate/up: [Wg ; Wu] as dims {L, 16, 2, E*H/16}, box {64, 16, 2, 4};
                               // down: Wd [E, L, H], box {64, 128}
    CUtensorMap mapX[XNMAP];   // the rows: bank [E, c_recv, L] or h [E, c_recv, H], box {64, XHSTEP (i+1)}
    const int4* groups;        // {expert, first row, rows, N0 | N1 << 16}
    const int* ngroups;
    int n_mb;                  // 256-row weight blocks a group (gate/up: H / 128; down: L / 256)
    int zpe;                   // gate/up: H / 16, 16-unit blocks an expert
    int gate_hi;               // gate/up: the gate tensor is the higher-addressed one
    int kb;                    // K blocks
    int c_recv;
    uint16_t* out;             // h [E, c_recv, H] (gate/up), ypool [pool_rows, L] (down),
                               // dg [E, c_recv, H] (SwiGLU backward)
    uint16_t* out2;            // SwiGLU backward: du [E, c_recv, H]
    const uint16_t* aux;       // SwiGLU backward: dh [E, c_recv, H]
    long long ldo;             // H or L
    const int* rowmap;         // scatter: the output row of each group row, [E, c_recv]
                               // (NULL: row e * c_recv + r, the per-expert layout)
    long long out_rows;        // scatter: output rows (checked builds)
    int a_mn;                  // scatter: the weights are MN-major (stored [K, M]): two
                               // 64 x 64 boxes a stage, 8 KB apart
    int kseg;                  // scatter: K in two segments of this many (0: one); mapW
                               // and mapX then have a 4th dimension stepping between two
                               // tensors, aseg / bseg giving each segment's index in it
    int aseg[2], bseg[2];
    const int32_t* roff;       // dropless layout: expert e's rows start at row roff[e] of the
                               // flat bank, h and row list (mapX one group of all rows);
                               // NULL: at e * c_recv, mapX [E, c_recv, K]
    const int32_t* rmoff;      // scatter, dropless backward: expert e's first entry in
                               // rowmap, where it differs from roff[e] (padded operands,
                               // unpadded row list); NULL: the same row as the operand
    int* status;
};

struct GTile {
    int e, row0, rows, n0, n1, mb;
    long long rbase;   // the expert's first row in the flat row space (e * c_recv or roff[e])
};

__device__ __forceinline__ GTile gate_tile(const GParams& p, int tile) {
    const int gi = tile / p.n_mb;
    const int4 g = p.groups[gi];
    GTile t;
    t.e = g.x;
    t.row0 = g.y;
    t.rows = g.z;
    t.n0 = g.w & 0xffff;
    t.n1 = static_cast<int>(static_cast<uint32_t>(g.w) >> 16);
    t.mb = tile - gi * p.n_mb;
    t.rbase = p.roff ? static_cast<long long>(p.roff[t.e])
                     : static_cast<long long>(t.e) * p.c_recv;
    return t;
}

// First TMEM column of the k-th tile of a pair whose accumulator has S columns.
__device__ __forceinline__ int gate_base(int k, int S) { return (k & 1) ? (512 - S) & ~31 : 0; }

__device__ __forceinline__ int gate_cols(const GParams& p, int tile) {
    const int w = p.groups[tile / p.n_mb].w;
    return (w & 0xffff) + static_cast<int>(static_cast<uint32_t>(w) >> 16);
}

template <int EPI>
__global__ void __launch_bounds__(GTHREADS, 1) expert_group_kernel(const __grid_constant__ GParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sbase = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sStage = sbase;                                   // GST x (W 16 KB | rows 26 KB)
    uint64_t* bars = reinterpret_cast<uint64_t*>(sbase + GST * GSTAGE);
    uint64_t* full = bars;
    uint64_t* empty = full + GST;
    uint64_t* tfull = empty + GST;   // [2]: a tile at that end is accumulated
    uint64_t* ovl = tfull + 2;       // [2]: its columns the next tile needs are drained
    uint64_t* fdone = ovl + 2;       // [2]: all its columns are drained
    uint64_t* done = fdone + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const bool leader = crank == 0;
    const int pair = static_cast<int>(blockIdx.x >> 1);
    const int npairs = static_cast<int>(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < GST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&ovl[a], 2 * GEPI_WARPS);     // one arrival a warp, both CTAs
            mbar_init(&fdone[a], 2 * GEPI_WARPS);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&p.mapW);
        for (int i = 0; i < XNMAP; ++i) tma_prefetch_map(&p.mapX[i]);
    }
    if (warp == 2) {
        tmem_alloc_pair(tmem_slot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();
    const uint32_t tmem_base = *tmem_slot;
    const int ntiles = *reinterpret_cast<const volatile int*>(p.ngroups) * p.n_mb;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t s = 0, ph = 0;
            uint32_t armed = 0, par = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < ntiles; tile += npairs) {
                const GTile t = gate_tile(p, tile);
                const int h0 = t.n0 >> 1, h1 = t.n1 >> 1;      // this CTA's rows of each chunk
                const int xrow0 = t.row0 + static_cast<int>(crank) * h0;
                const int xrow1 = t.row0 + t.n0 + static_cast<int>(crank) * h1;
                const uint32_t bytes = XA_BYTES + static_cast<uint32_t>(h0 + h1) * XBK * 2;
                const int z = t.e * p.zpe + t.mb * 8 + static_cast<int>(crank) * 4;
                for (int kb = 0; kb < p.kb; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    if (leader) {
                        mbar_arrive_expect_tx(&full[s], 2u * bytes);
                        armed |= 1u << s;
                        par = (par & ~(1u << s)) | (ph << s);
                    }
                    const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
                    const uint32_t a_dst = smem_u32(sStage + s * GSTAGE);
                    const uint32_t b_dst = a_dst + XA_BYTES;
                    const int kx = kb * XBK;
                    const int m0 = t.mb * 256 + static_cast<int>(crank) * 128;
                    const int sg = p.kseg ? kx / p.kseg : 0, kin = kx - sg * p.kseg;
                    if (EPI != EPI_SCATTER) {
                        tma_load_4d_pair(a_dst, &p.mapW, fb, kx, 0, 0, z);
                    } else if (!p.a_mn) {
                        tma_load_3d_pair(a_dst, &p.mapW, fb, kx, m0, t.e);
                    } else if (p.kseg) {
                        tma_load_4d_pair(a_dst, &p.mapW, fb, m0, kin, t.e, p.aseg[sg]);
                        tma_load_4d_pair(a_dst + 8192, &p.mapW, fb, m0 + 64, kin, t.e, p.aseg[sg]);
                    } else {
                        tma_load_3d_pair(a_dst, &p.mapW, fb, m0, kx, t.e);
                        tma_load_3d_pair(a_dst + 8192, &p.mapW, fb, m0 + 64, kx, t.e);
                    }
                    // rows: [E, c_recv] by expert, or (dropless) one flat group
                    const int by = p.roff ? static_cast<int>(t.rbase) : 0;
                    const int bz = p.roff ? 0 : t.e;
                    if (p.kseg) {
                        tma_load_4d_pair(b_dst, &p.mapX[h0 / XHSTEP - 1], fb, kin, by + xrow0, bz,
                                         p.bseg[sg]);
                        if (h1)
                            tma_load_4d_pair(b_dst + h0 * XBK * 2, &p.mapX[h1 / XHSTEP - 1], fb, kin,
                                             by + xrow1, bz, p.bseg[sg]);
                    } else {
                        tma_load_3d_pair(b_dst, &p.mapX[h0 / XHSTEP - 1], fb, kx, by + xrow0, bz);
                        if (h1)
                            tma_load_3d_pair(b_dst + h0 * XBK * 2, &p.mapX[h1 / XHSTEP - 1], fb, kx,
                                             by + xrow1, bz);
                    }
                    if (++s == GST) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok || *abort_flag) {
                volatile int no_abort = 0;
                for (int i = 0; i < GST; ++i)
                    if (armed >> i & 1u)
                        mbar_wait(&full[i], (par >> i) & 1u, &no_abort, nullptr, 20000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && !leader) {
            volatile int no_abort = 0;
            mbar_wait(done, 0, &no_abort, p.status);
        } else if (lane == 0) {
            uint32_t s = 0, ph = 0;
            bool ok = true;
            int k = 0;   // this pair's tiles so far
            for (int tile = pair; ok && tile < ntiles; tile += npairs, ++k) {
                const GTile t = gate_tile(p, tile);
                const uint32_t end = static_cast<uint32_t>(k & 1);
                // the tile two before (same end) fully drained, the tile
                // before drained where this one's columns lie
                if (k >= 2)
                    ok = mbar_wait(&fdone[end], static_cast<uint32_t>((k - 2) >> 1) & 1u, abort_flag,
                                   p.status);
                if (ok && k >= 1)
                    ok = mbar_wait(&ovl[end ^ 1u], static_cast<uint32_t>((k - 1) >> 1) & 1u,
                                   abort_flag, p.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(gate_base(k, t.n0 + t.n1));
                const uint32_t d1 = d0 + static_cast<uint32_t>(t.n0);
                const bool amn = EPI == EPI_SCATTER && p.a_mn;
                const uint32_t id0 = idesc_bf16_f32(256, t.n0, amn);
                const uint32_t id1 = idesc_bf16_f32(256, t.n1 ? t.n1 : 16, amn);
                const uint32_t boff1 = static_cast<uint32_t>(t.n0 >> 1) * XBK * 2;
                // descriptor step per 16-wide K slice: 32 B along a K-major row,
                // 16 rows of 128 B down an MN-major box
                const uint32_t a_step = amn ? (2048u >> 4) : (32u >> 4);
                for (int kb = 0; kb < p.kb; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_s = smem_u32(sStage + s * GSTAGE);
                    const uint64_t ad = amn ? sdesc_mn_sw128(a_s) : sdesc_k_sw128(a_s);
                    const uint64_t bd0 = sdesc_k_sw128(a_s + XA_BYTES);
                    const uint64_t bd1 = sdesc_k_sw128(a_s + XA_BYTES + boff1);
#pragma unroll
                    for (int kk = 0; kk < XBK / 16; ++kk) {
                        const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                        mma_bf16_pair(d0, ad + a_step * kk, bd0 + 2u * kk, id0, acc);
                        if (t.n1) mma_bf16_pair(d1, ad + a_step * kk, bd1 + 2u * kk, id1, acc);
                    }
                    mma_commit_pair(&empty[s]);
                    if (++s == GST) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair(&tfull[end]);
            }
            mma_commit_pair(done);
            volatile int no_abort = 0;
            mbar_wait(done, 0, &no_abort, p.status);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 4;
        const int q = ew & 3;                     // TMEM lane quarter (= warp % 4)
        const int grp = ew >> 2;                  // order positions grp, grp + GEPQ, ...
        const bool hi = lane >= 16;               // lanes of the higher-addressed tensor
        const int y = lane & 15;
        const bool odd = (y & 1) != 0;
        const uint32_t bar_c0 = mapa_shared(smem_u32(&ovl[0]), 0);
        const uint32_t fdone_c0 = mapa_shared(smem_u32(&fdone[0]), 0);
        int k = 0;
        for (int tile = pair; tile < ntiles; tile += npairs, ++k) {
            const GTile t = gate_tile(p, tile);
            const uint32_t end = static_cast<uint32_t>(k & 1);
            const int S = t.n0 + t.n1;
            const int base = gate_base(k, S);
            const int nblk = (S + 31) >> 5;
            // columns the next tile (other end) needs: blocks met first in
            // this tile's drain order (from the end facing it)
            int n_ov = 0;
            if (tile + npairs < ntiles) {
                const int S2 = gate_cols(p, tile + npairs);
                const int b2 = gate_base(k + 1, S2);
                const int lo = base > b2 ? base : b2;
                const int hi_c = base + S < b2 + S2 ? base + S : b2 + S2;
                if (lo < hi_c)
                    n_ov = end ? (hi_c - base + 31) >> 5                 // ascending: blocks below hi_c
                               : nblk - ((lo - base) >> 5);              // descending: blocks from lo up
            }
            const int my_ov = n_ov > grp ? (n_ov - grp + GEPQ - 1) / GEPQ : 0;
            if (my_ov == 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(bar_c0 + end * 8u);
            }
            const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                static_cast<uint32_t>(base);
            if (EPI == EPI_SCATTER) {
                // The pool row of each row of this warp's blocks, loaded before
                // the accumulator is ready: lane j holds row 32 b + j of its
                // i-th block b.
                int prow[GMAXB];
#pragma unroll
                for (int i = 0; i < GMAXB; ++i) {
                    const int pos = grp + GEPQ * i;
                    const int b = end ? pos : nblk - 1 - pos;
                    const int rr = 32 * b + lane;
                    prow[i] = -1;
                    if (pos < nblk && rr < t.rows) {
                        const int rm = p.rmoff ? p.rmoff[t.e] : static_cast<int>(t.rbase);
                        const int r = rm + t.row0 + rr;
                        const int v = p.rowmap ? p.rowmap[r] : static_cast<int>(t.rbase) + t.row0 + rr;
                        if (moe_check(v >= 0 && v < p.out_rows, 1102)) prow[i] = v;
                    }
                }
                if (!mbar_wait(&tfull[end], static_cast<uint32_t>(k >> 1) & 1u, abort_flag, p.status))
                    break;
                tc_fence_after();
                // lane f: output feature 32 q + f of this CTA's 128
                uint16_t* ob = p.out + t.mb * 256 + static_cast<int>(crank) * 128 + 32 * q + (lane & ~1);
                const bool fodd = (lane & 1) != 0;
#pragma unroll
                for (int i = 0; i < GMAXB; ++i) {
                    const int pos = grp + GEPQ * i;
                    if (pos >= nblk) break;   // warp-uniform
                    const int b = end ? pos : nblk - 1 - pos;
                    uint32_t r[32];
                    if (S - 32 * b >= 32) {
                        tmem_ld32(tl + 32 * b, r);
                    } else {
                        uint32_t r16[16];
                        tmem_ld16(tl + 32 * b, r16);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            r[j] = r16[j];
                            r[16 + j] = 0u;
                        }
                    }
                    if (i + 1 == my_ov) {   // this warp's share of the overlap is out of TMEM
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster_relaxed(bar_c0 + end * 8u);
                    }
                    // pairs of features to 32-bit stores: even lanes rows 0-15,
                    // odd lanes rows 16-31 of the block
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float v = __uint_as_float(fodd ? r[j] : r[16 + j]);
                        const float other = __shfl_xor_sync(0xffffffffu, v, 1);
                        const int rl = fodd ? 16 + j : j;
                        const int pr = __shfl_sync(0xffffffffu, prow[i], rl);
                        const uint32_t word =
                            fodd ? pack_bf16x2(other, __uint_as_float(r[16 + j]))
                                 : pack_bf16x2(__uint_as_float(r[j]), other);
                        if (pr >= 0)
                            *reinterpret_cast<uint32_t*>(ob + static_cast<long long>(pr) * p.ldo) = word;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_relaxed(fdone_c0 + end * 8u);
                continue;
            }
            if (!mbar_wait(&tfull[end], static_cast<uint32_t>(k >> 1) & 1u, abort_flag, p.status))
                break;
            tc_fence_after();
            // column c of the tile is the group's row row0 + c (chunk 0 is full)
            const int unit = t.mb * 128 + static_cast<int>(crank) * 64 + q * 16 + (y & ~1);
            uint16_t* hb = p.out + (t.rbase + t.row0) * p.ldo + unit;
            int drained = 0;
#pragma unroll 1
            for (int pos = grp; pos < nblk; pos += GEPQ) {
                const int b = end ? pos : nblk - 1 - pos;
                uint32_t r[32];
                if (S - 32 * b >= 32) {
                    tmem_ld32(tl + 32 * b, r);
                } else {
                    uint32_t r16[16];
                    tmem_ld16(tl + 32 * b, r16);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        r[j] = r16[j];
                        r[16 + j] = 0u;
                    }
                }
                if (++drained == my_ov) {   // this warp's share of the overlap is out of TMEM
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(bar_c0 + end * 8u);
                }
                if (EPI == EPI_SWIGLU_BWD) {
                    // recomputed g, u of this lane's unit for rows 0-15 (lanes < 16)
                    // or 16-31 of the block, then pairs of units per lane: even
                    // lanes rows 0-7, odd lanes 8-15; incoming dh, dg = dh u
                    // silu'(g), du = dh silu(g); 32-bit loads and stores
                    float gv[16], uv[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint32_t mine = hi ? r[16 + j] : r[j];
                        const uint32_t give = hi ? r[j] : r[16 + j];
                        const float oth = __uint_as_float(__shfl_xor_sync(0xffffffffu, give, 16));
                        const float own = __uint_as_float(mine);
                        const float lo_t = hi ? oth : own, hi_t = hi ? own : oth;
                        gv[j] = p.gate_hi ? hi_t : lo_t;
                        uv[j] = p.gate_hi ? lo_t : hi_t;
                    }
                    const long long gbase = (t.rbase + t.row0) * p.ldo + unit;
                    const int rb = 32 * b + (hi ? 16 : 0) + (odd ? 8 : 0);   // this lane's first row
                    // the eight rows' dh first (independent loads), then the
                    // partner's g, u, then the arithmetic
                    uint32_t hw[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        hw[j] = rb + j < t.rows
                                    ? *reinterpret_cast<const uint32_t*>(
                                          p.aux + gbase + static_cast<long long>(rb + j) * p.ldo)
                                    : 0u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float og = __shfl_xor_sync(0xffffffffu, odd ? gv[j] : gv[8 + j], 1);
                        const float ou = __shfl_xor_sync(0xffffffffu, odd ? uv[j] : uv[8 + j], 1);
                        const int row = rb + j;
                        if (row < t.rows) {
                            const float g2[2] = {odd ? og : gv[j], odd ? gv[8 + j] : og};
                            const float u2[2] = {odd ? ou : uv[j], odd ? uv[8 + j] : ou};
                            const long long off = gbase + static_cast<long long>(row) * p.ldo;
                            float dg2[2], du2[2];
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const float gg = g2[e2], uu = u2[e2];
                                const float dh = e2 ? bf16_hi(hw[j]) : bf16_lo(hw[j]);
                                const float sig = 1.0f / (1.0f + expf(-gg));
                                dg2[e2] = dh * uu * (sig * (1.0f + gg * (1.0f - sig)));
                                du2[e2] = dh * (gg * sig);
                            }
                            *reinterpret_cast<uint32_t*>(p.out + off) = pack_bf16x2(dg2[0], dg2[1]);
                            *reinterpret_cast<uint32_t*>(p.out2 + off) = pack_bf16x2(du2[0], du2[1]);
                        }
                    }
                } else {
                // lanes < 16 finish rows 0-15 of the block, lanes >= 16 rows 16-31
                float hv[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t mine = hi ? r[16 + j] : r[j];
                    const uint32_t give = hi ? r[j] : r[16 + j];
                    const float oth = __uint_as_float(__shfl_xor_sync(0xffffffffu, give, 16));
                    const float own = __uint_as_float(mine);
                    const float lo_t = hi ? oth : own, hi_t = hi ? own : oth;
                    const float g = p.gate_hi ? hi_t : lo_t, u = p.gate_hi ? lo_t : hi_t;
                    hv[j] = silu_fast(g) * u;
                }
                // pairs of units to 32-bit stores: even lanes rows 0-7, odd lanes 8-15
                const int rb = 32 * b + (hi ? 16 : 0);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float other = __shfl_xor_sync(0xffffffffu, odd ? hv[j] : hv[8 + j], 1);
                    const int row = rb + (odd ? 8 + j : j);
                    const uint32_t word = odd ? pack_bf16x2(other, hv[8 + j]) : pack_bf16x2(hv[j], other);
                    if (row < t.rows)
                        *reinterpret_cast<uint32_t*>(hb + static_cast<long long>(row) * p.ldo) = word;
                }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(fdone_c0 + end * 8u);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();
    if (warp == 2) tmem_dealloc_pair(tmem_base, 512);
}

// Block-wide exclusive prefix of v over the CTA's threads, plus the running
// total carried across calls (all threads call it; blockDim a multiple of 32).
__device__ __forceinline__ int block_excl_scan(int v, int* warp_sum, int* carry) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
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
    const int excl = *carry + (wid ? warp_sum[wid - 1] : 0) + incl - v;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) *carry = excl + v;
    __syncthreads();
    return excl;
}

__device__ __forceinline__ int round_gran(int n) { return (n + XGRAN - 1) / XGRAN * XGRAN; }

// Pieces of at most `cap` rows covering n rows, sized evenly and rounded up to
// XGRAN (the last one takes the rest): the piece size, and their number.
__device__ __forceinline__ int piece_rows(int n, int cap, int* count) {
    if (n <= 0) {
        *count = 0;
        return 0;
    }
    const int per = round_gran((n + (n + cap - 1) / cap - 1) / ((n + cap - 1) / cap));
    *count = (n + per - 1) / per;
    return per;
}

// For every expert with rows:
//  chunks {expert, first row, rows, N}: pieces of at most 256 rows, N = the
//    rows rounded up to XGRAN (the down product's tiles);
//  groups {expert, first row, rows, N0 | N1 << 16}: pieces of at most 416 rows
//    (the gate/up product's tiles), each one chunk (N0 = rows rounded up,
//    N1 = 0) up to 256 rows, else two: N0 = half the rows rounded up to 32
//    (chunk 0 exactly full), N1 = the rest rounded up to XGRAN; N0 + N1 is at
//    most the rows rounded up to XGRAN, so at most 416.
// One CTA; block-wide exclusive prefixes over the experts' counts.
__global__ void __launch_bounds__(1024) chunk_list_kernel(const int32_t* __restrict__ counts,
                                                          int E, int c_recv, int4* __restrict__ chunks,
                                                          int32_t* __restrict__ nchunks,
                                                          int4* __restrict__ groups,
                                                          int32_t* __restrict__ ngroups) {
    __shared__ int warp_sum[32];
    __shared__ int carry_c, carry_g;
    if (threadIdx.x == 0) carry_c = carry_g = 0;
    __syncthreads();
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        int n = e < E ? counts[e] : 0;
        n = n < 0 ? 0 : (n > c_recv ? c_recv : n);
        int nch, ngr;
        const int per = piece_rows(n, XCHUNK, &nch);
        const int pg = piece_rows(n, GACC, &ngr);
        const int exc = block_excl_scan(nch, warp_sum, &carry_c);
        const int exg = block_excl_scan(ngr, warp_sum, &carry_g);
        for (int i = 0; i < nch; ++i) {
            const int r0 = i * per;
            const int rows = (n - r0 < per) ? n - r0 : per;
            chunks[exc + i] = make_int4(e, r0, rows, round_gran(rows));
        }
        for (int i = 0; i < ngr; ++i) {
            const int r0 = i * pg;
            const int rows = (n - r0 < pg) ? n - r0 : pg;
            int n0, n1;
            if (rows <= XCHUNK) {
                n0 = round_gran(rows);
                n1 = 0;
            } else {   // chunk 0: half the rows rounded up to 32 (at most 224)
                n0 = ((rows + 1) / 2 + 31) / 32 * 32;
                n1 = round_gran(rows - n0);
            }
            groups[exg + i] = make_int4(e, r0, rows, n0 | (n1 << 16));
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        *nchunks = carry_c;
        *ngroups = carry_g;
    }
}

typedef CUresult (*EncodeTiledFnX)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnX encode_x() {
    static EncodeTiledFnX fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFnX>(f);
    }();
    return fn;
}

// bf16 [groups, rows, cols] (row pitch ld, group stride gs elements), box
// {64, box_rows, 1}, 128-byte swizzle; reads past the rows give zeros.
int map3(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t groups,
         uint64_t ld, uint64_t gs, uint32_t box_rows) {
    EncodeTiledFnX enc = encode_x();
    if (!enc) return MOE_ECUDA;
    const cuuint64_t gdim[3] = {cols, rows, groups};
    const cuuint64_t gstr[2] = {ld * 2, gs * 2};
    const cuuint32_t box[3] = {XBK, box_rows, 1}, est[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstr,
                     box, est, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ECUDA;
}

// bf16 4-D map of dims {d0, d1, d2, d3} (d0 contiguous) with byte strides
// {s1, s2, s3} of dims 1..3, box {64, box1, 1, 1}, 128-byte swizzle: two
// tensors of the same shape as the two values of the outermost dimension,
// s3 the distance from the lower-addressed to the other.  MOE_EINVAL when the
// driver refuses it (a distance of 0, not a multiple of 16, ...).
int map4(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
         uint64_t s1, uint64_t s2, uint64_t s3, uint32_t box1) {
    EncodeTiledFnX enc = encode_x();
    if (!enc) return MOE_ECUDA;
    if (s3 == 0 || (s3 & 15) || s3 >= (1ull << 40)) return MOE_EINVAL;
    const cuuint64_t gdim[4] = {d0, d1, d2, d3};
    const cuuint64_t gstr[3] = {s1, s2, s3};
    const cuuint32_t box[4] = {XBK, box1, 1, 1}, est[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gdim, gstr,
                     box, est, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_EINVAL;
}

// One map over both gate/up weight tensors, so that one box brings a CTA's
// 64 gate rows and the 64 up rows of the same units: dims {L, 64, E*H/64,
// 2}, the outermost one stepping from the lower-addressed tensor to the
// other (strides grow outward only when the two do not overlap), box
// {64, 64, 1, 2}: rows 0-63 of the box from the lower tensor, 64-127 from
// the other.  MOE_EINVAL when the tensors' distance does not allow it.
int map_gateup(CUtensorMap* m, const void* Wg, const void* Wu, int E, int H, int L,
               int* gate_hi) {
    EncodeTiledFnX enc = encode_x();
    if (!enc) return MOE_ECUDA;
    const uintptr_t g = reinterpret_cast<uintptr_t>(Wg), u = reinterpret_cast<uintptr_t>(Wu);
    const uintptr_t lo = g < u ? g : u, hi = g < u ? u : g;
    const uint64_t span = static_cast<uint64_t>(E) * H * L * 2;   // bytes of one tensor
    const uint64_t dist = hi - lo;
    if (dist < span || (dist & 15) || dist >= (1ull << 40) || H % 64) return MOE_EINVAL;
    const cuuint64_t gdim[4] = {static_cast<cuuint64_t>(L), 64,
                                static_cast<cuuint64_t>(E) * (H / 64), 2};
    const cuuint64_t gstr[3] = {static_cast<cuuint64_t>(L) * 2, 64ull * L * 2, dist};
    const cuuint32_t box[4] = {XBK, 64, 1, 2}, est[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, reinterpret_cast<void*>(lo), gdim, gstr,
                     box, est, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return MOE_EINVAL;
    *gate_hi = g > u ? 1 : 0;
    return MOE_OK;
}

template <int EPI>
int launch_pair(const XParams& p, int sms, cudaStream_t st, const char* name) {
    auto kern = expert_pair_kernel<EPI>;
    if (ensure_smem_attr(reinterpret_cast<const void*>(kern), XSMEM) != MOE_OK) return MOE_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = XSMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return MOE_ECUDA;
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, name);
    return MOE_OK;
}

// [Wg ; Wu] for the TMEM-held gate/up product: dims {L, 16, 2, E*H/16} with
// strides {row, distance from the lower-addressed tensor to the other, 16
// rows}, box {64, 16, 2, 4}: a box of 128 rows holds, for each of 4 blocks of
// 16 hidden units, the 16 rows of the lower tensor then the 16 of the other.
// MOE_EINVAL when the two tensors' distance cannot be a stride.
int map_gateup_il(CUtensorMap* m, const void* Wg, const void* Wu, int E, int H, int L,
                  int* gate_hi) {
    EncodeTiledFnX enc = encode_x();
    if (!enc) return MOE_ECUDA;
    const uintptr_t g = reinterpret_cast<uintptr_t>(Wg), u = reinterpret_cast<uintptr_t>(Wu);
    const uintptr_t lo = g < u ? g : u, hi = g < u ? u : g;
    const uint64_t dist = hi - lo;
    if (dist == 0 || (dist & 15) || dist >= (1ull << 40) || H % 64 || (lo & 15)) return MOE_EINVAL;
    const cuuint64_t gdim[4] = {static_cast<cuuint64_t>(L), 16, 2,
                                static_cast<cuuint64_t>(E) * (H / 16)};
    const cuuint64_t gstr[3] = {static_cast<cuuint64_t>(L) * 2, dist, 16ull * L * 2};
    const cuuint32_t box[4] = {XBK, 16, 2, 4}, est[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, reinterpret_cast<void*>(lo), gdim, gstr,
                     box, est, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return MOE_EINVAL;
    *gate_hi = g > u ? 1 : 0;
    return MOE_OK;
}

template <int EPI>
int launch_group(const GParams& p, int sms, cudaStream_t st, const char* name) {
    auto kern = expert_group_kernel<EPI>;
    if (ensure_smem_attr(reinterpret_cast<const void*>(kern), GSMEM) != MOE_OK) return MOE_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
    cfg.blockDim = dim3(GTHREADS, 1, 1);
    cfg.dynamicSmemBytes = GSMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return MOE_ECUDA;
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, name);
    return MOE_OK;
}

// The down product: over the row groups (expert_group_kernel), or with
// MOE_XPAIR_DGROUP=0 over the chunk list (expert_pair_kernel).
#ifndef MOE_XPAIR_DGROUP
#define MOE_XPAIR_DGROUP 1
#endif
int launch_down(int E, int c_recv, int L, int H, const uint16_t* Wd, const int4* chunks,
                const int32_t* nchunks, const int4* groups, const int32_t* ngroups, uint16_t* h,
                const int32_t* expert_rows, uint16_t* ypool, int64_t pool_rows, int32_t* status,
                int sms, cudaStream_t st) {
    int rc;
    if (MOE_XPAIR_DGROUP) {
        GParams g;
        std::memset(&g, 0, sizeof(g));
        if ((rc = map3(&g.mapW, Wd, H, L, E, H, static_cast<uint64_t>(L) * H, 128))) return rc;
        for (int i = 0; i < XNMAP; ++i)
            if ((rc = map3(&g.mapX[i], h, H, c_recv, E, H, static_cast<uint64_t>(c_recv) * H,
                           XHSTEP * (i + 1))))
                return rc;
        g.groups = groups;
        g.ngroups = ngroups;
        g.n_mb = L / 256;
        g.kb = H / XBK;
        g.c_recv = c_recv;
        g.out = ypool;
        g.ldo = L;
        g.rowmap = expert_rows;
        g.out_rows = pool_rows;
        g.status = status;
        return launch_group<EPI_SCATTER>(g, sms, st, "gemm_expert_down");
    }
    XParams b;
    std::memset(&b, 0, sizeof(b));
    if ((rc = map3(&b.mapW0, Wd, H, L, E, H, static_cast<uint64_t>(L) * H, 128))) return rc;
    for (int i = 0; i < XNMAP; ++i)
        if ((rc = map3(&b.mapX[i], h, H, c_recv, E, H, static_cast<uint64_t>(c_recv) * H,
                       XHSTEP * (i + 1))))
            return rc;
    b.chunks = chunks;
    b.nchunks = nchunks;
    b.n_mb = L / 256;
    b.kb = (H + XBK - 1) / XBK;
    b.c_recv = c_recv;
    b.out = ypool;
    b.ldo = L;
    b.rowmap = expert_rows;
    b.out_rows = pool_rows;
    b.status = status;
    return launch_pair<EPI_SCATTER>(b, sms, st, "gemm_expert_down");
}

}  // namespace

int check_status_expert_pair() { return moe_check_read_reset(); }

static size_t chunk_list_bytes(int E, int c_recv);

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t expert_pair_lists_bytes_ragged(int E, int64_t rows) {
    // every expert's chunks and groups: at most E + rows / 256 and E + rows / 416
    const size_t nc = static_cast<size_t>(E) + static_cast<size_t>(rows / XCHUNK) + 1;
    const size_t ng = static_cast<size_t>(E) + static_cast<size_t>(rows / GACC) + 1;
    return (nc + ng) * sizeof(int4) + 16;
}

int expert_ffn_pair_ragged(int E, int64_t rows, int L, int H, const uint16_t* bank,
                           const int32_t* expert_offsets, const int32_t* expert_rows,
                           const int32_t* expert_count, const uint16_t* Wg, const uint16_t* Wu,
                           const uint16_t* Wd, void* list_ws, uint16_t* h, uint16_t* ypool,
                           int32_t* status, cudaStream_t st) {
    int dev, sms;
    int rc = current_device(&dev, &sms);
    if (rc) return rc;
    if (!MOE_XPAIR_TM || sms < 2 || E <= 0 || rows <= 0 || rows > INT32_MAX / 2 || L % 256 ||
        H % 128 || !al16(bank) || !al16(h) || !al16(list_ws))
        return MOE_EINVAL;
    GParams g;
    std::memset(&g, 0, sizeof(g));
    if (map_gateup_il(&g.mapW, Wg, Wu, E, H, L, &g.gate_hi) != MOE_OK) return MOE_EINVAL;
    for (int i = 0; i < XNMAP; ++i)   // the flat bank [rows, L] as one group
        if ((rc = map3(&g.mapX[i], bank, L, rows, 1, L, static_cast<uint64_t>(rows) * L,
                       XHSTEP * (i + 1))))
            return rc;
    const size_t nc = static_cast<size_t>(E) + static_cast<size_t>(rows / XCHUNK) + 1;
    uint8_t* w = static_cast<uint8_t*>(list_ws);
    int4* chunks = reinterpret_cast<int4*>(w);
    int4* groups = chunks + nc;
    int32_t* counts = reinterpret_cast<int32_t*>(w + expert_pair_lists_bytes_ragged(E, rows) - 16);
    chunk_list_kernel<<<1, 1024, 0, st>>>(expert_count, E, INT32_MAX, chunks, counts, groups,
                                          counts + 1);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "build_chunks");
    g.groups = groups;
    g.ngroups = counts + 1;
    g.n_mb = H / 128;
    g.zpe = H / 16;
    g.kb = L / XBK;
    g.out = h;
    g.ldo = H;
    g.roff = expert_offsets;
    g.status = status;
    if ((rc = launch_group<EPI_SWIGLU>(g, sms, st, "gemm_expert_gateup"))) return rc;
    GParams d;
    std::memset(&d, 0, sizeof(d));
    if ((rc = map3(&d.mapW, Wd, H, L, E, H, static_cast<uint64_t>(L) * H, 128))) return rc;
    for (int i = 0; i < XNMAP; ++i)   // the flat h [rows, H] as one group
        if ((rc = map3(&d.mapX[i], h, H, rows, 1, H, static_cast<uint64_t>(rows) * H,
                       XHSTEP * (i + 1))))
            return rc;
    d.groups = groups;
    d.ngroups = counts + 1;
    d.n_mb = L / 256;
    d.kb = H / XBK;
    d.out = ypool;
    d.ldo = L;
    d.rowmap = expert_rows;
    d.out_rows = rows;
    d.roff = expert_offsets;
    d.status = status;
    return launch_group<EPI_SCATTER>(d, sms, st, "gemm_expert_down");
}

int expert_group_list(int E, int c_recv, const int32_t* expert_count, void* ws, ExpertGroups* out,
                      cudaStream_t st) {
    if (E <= 0 || c_recv <= 0 || (reinterpret_cast<uintptr_t>(ws) & 15)) return MOE_EINVAL;
    uint8_t* w = static_cast<uint8_t*>(ws);
    int4* chunks = reinterpret_cast<int4*>(w);
    int4* groups = reinterpret_cast<int4*>(w + chunk_list_bytes(E, c_recv));
    int32_t* counts = reinterpret_cast<int32_t*>(w + expert_pair_chunks_bytes(E, c_recv) - 16);
    chunk_list_kernel<<<1, 1024, 0, st>>>(expert_count, E, c_recv, chunks, counts, groups,
                                          counts + 1);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "bwd_build_groups");
    out->groups = groups;
    out->ngroups = counts + 1;
    return MOE_OK;
}

int expert_group_list_ragged(int E, int64_t rows, const int32_t* expert_count, void* ws,
                             ExpertGroups* out, cudaStream_t st) {
    if (E <= 0 || rows <= 0 || rows > INT32_MAX / 2 || (reinterpret_cast<uintptr_t>(ws) & 15))
        return MOE_EINVAL;
    const size_t nc = static_cast<size_t>(E) + static_cast<size_t>(rows / XCHUNK) + 1;
    uint8_t* w = static_cast<uint8_t*>(ws);
    int4* chunks = reinterpret_cast<int4*>(w);
    int4* groups = chunks + nc;
    int32_t* counts = reinterpret_cast<int32_t*>(w + expert_pair_lists_bytes_ragged(E, rows) - 16);
    chunk_list_kernel<<<1, 1024, 0, st>>>(expert_count, E, INT32_MAX, chunks, counts, groups,
                                          counts + 1);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "bwd_build_groups");
    out->groups = groups;
    out->ngroups = counts + 1;
    return MOE_OK;
}

// The rows of a backward product's operand X [K wide]: per expert [E, c_recv,
// K], or (roff) one flat group of `rows`, expert e's from row roff[e].
static int map_rows(CUtensorMap* m, const void* X, int K, int c_recv, int E,
                    const int32_t* roff, int64_t rows, int i) {
    if (roff)
        return map3(m, X, K, rows, 1, K, static_cast<uint64_t>(rows) * K, XHSTEP * (i + 1));
    return map3(m, X, K, c_recv, E, K, static_cast<uint64_t>(c_recv) * K, XHSTEP * (i + 1));
}

static bool bwd_rows_ok(int sms, int E, int c_recv, const int32_t* roff, int64_t rows) {
    return sms >= 2 && E > 0 && (roff ? rows > 0 && rows <= INT32_MAX / 2 : c_recv > 0);
}

int expert_dh_group(int E, int c_recv, int L, int H, const uint16_t* dye, const uint16_t* Wd,
                    const ExpertGroups& gl, uint16_t* dh, int32_t* status, cudaStream_t st,
                    const int32_t* roff, int64_t rows) {
    int dev, sms;
    int rc = current_device(&dev, &sms);
    if (rc) return rc;
    if (!MOE_XPAIR_TM || !bwd_rows_ok(sms, E, c_recv, roff, rows) || H % 256 || L % 64 ||
        !al16(dye) || !al16(Wd) || !al16(dh))
        return MOE_EINVAL;
    GParams g;
    std::memset(&g, 0, sizeof(g));
    // Wd [E, L, H] is the weights' [K, M]: MN-major boxes of 64 units x 64 K
    if ((rc = map3(&g.mapW, Wd, H, L, E, H, static_cast<uint64_t>(L) * H, 64))) return rc;
    for (int i = 0; i < XNMAP; ++i)
        if ((rc = map_rows(&g.mapX[i], dye, L, c_recv, E, roff, rows, i))) return rc;
    g.roff = roff;
    g.groups = gl.groups;
    g.ngroups = gl.ngroups;
    g.n_mb = H / 256;
    g.kb = L / XBK;
    g.c_recv = c_recv;
    g.out = dh;
    g.ldo = H;
    g.rowmap = nullptr;   // dh in the operand's row layout
    g.out_rows = roff ? rows : static_cast<long long>(E) * c_recv;
    g.a_mn = 1;
    g.status = status;
    return launch_group<EPI_SCATTER>(g, sms, st, "bwd_gemm_dh");
}

int expert_swiglu_bwd_group(int E, int c_recv, int L, int H, const uint16_t* xe,
                            const uint16_t* Wg, const uint16_t* Wu, const uint16_t* dh,
                            const ExpertGroups& gl, uint16_t* dg, uint16_t* du, int32_t* status,
                            cudaStream_t st, const int32_t* roff, int64_t rows) {
    int dev, sms;
    int rc = current_device(&dev, &sms);
    if (rc) return rc;
    if (!MOE_XPAIR_TM || !bwd_rows_ok(sms, E, c_recv, roff, rows) || L % 256 || H % 128 ||
        !al16(xe) || !al16(dh) || !al16(dg) || !al16(du))
        return MOE_EINVAL;
    GParams g;
    std::memset(&g, 0, sizeof(g));
    if (map_gateup_il(&g.mapW, Wg, Wu, E, H, L, &g.gate_hi) != MOE_OK) return MOE_EINVAL;
    for (int i = 0; i < XNMAP; ++i)
        if ((rc = map_rows(&g.mapX[i], xe, L, c_recv, E, roff, rows, i))) return rc;
    g.roff = roff;
    g.groups = gl.groups;
    g.ngroups = gl.ngroups;
    g.n_mb = H / 128;
    g.zpe = H / 16;
    g.kb = L / XBK;
    g.c_recv = c_recv;
    g.out = dg;
    g.out2 = du;
    g.aux = dh;
    g.ldo = H;
    g.status = status;
    return launch_group<EPI_SWIGLU_BWD>(g, sms, st, "bwd_gemm_expert_swiglu");
}

int expert_dx_group(int E, int c_recv, int L, int H, const uint16_t* dg, const uint16_t* du,
                    const uint16_t* Wg, const uint16_t* Wu, const ExpertGroups& gl,
                    const int32_t* expert_rows, uint16_t* dxpool, int64_t pool_rows,
                    int32_t* status, cudaStream_t st, const int32_t* roff, int64_t rows,
                    const int32_t* rmoff) {
    int dev, sms;
    int rc = current_device(&dev, &sms);
    if (rc) return rc;
    if (!MOE_XPAIR_TM || !bwd_rows_ok(sms, E, c_recv, roff, rows) || L % 256 || H % 64 ||
        !al16(dg) || !al16(du) || !al16(Wg) || !al16(Wu) || !al16(dxpool))
        return MOE_EINVAL;
    GParams g;
    std::memset(&g, 0, sizeof(g));
    // K in two segments, gate then up: the weights Wg, Wu [E, H, L] as [K, M]
    // (MN-major), the rows dg, du [E, c_recv, H]; each pair through one 4-D
    // map whose outer dimension steps from the lower-addressed tensor to the
    // other
    const uintptr_t wg = reinterpret_cast<uintptr_t>(Wg), wu = reinterpret_cast<uintptr_t>(Wu);
    const uintptr_t xg = reinterpret_cast<uintptr_t>(dg), xu = reinterpret_cast<uintptr_t>(du);
    const void* wlo = reinterpret_cast<const void*>(wg < wu ? wg : wu);
    const void* xlo = reinterpret_cast<const void*>(xg < xu ? xg : xu);
    if ((rc = map4(&g.mapW, wlo, L, H, E, 2, static_cast<uint64_t>(L) * 2,
                   static_cast<uint64_t>(H) * L * 2, wg < wu ? wu - wg : wg - wu, 64)))
        return rc;
    const uint64_t xrows = roff ? static_cast<uint64_t>(rows) : static_cast<uint64_t>(c_recv);
    const uint64_t xgroups = roff ? 1u : static_cast<uint64_t>(E);
    for (int i = 0; i < XNMAP; ++i)
        if ((rc = map4(&g.mapX[i], xlo, H, xrows, xgroups, 2, static_cast<uint64_t>(H) * 2,
                       xrows * H * 2, xg < xu ? xu - xg : xg - xu, XHSTEP * (i + 1))))
            return rc;
    g.roff = roff;
    g.rmoff = rmoff;
    g.aseg[0] = wg < wu ? 0 : 1;
    g.aseg[1] = 1 - g.aseg[0];
    g.bseg[0] = xg < xu ? 0 : 1;
    g.bseg[1] = 1 - g.bseg[0];
    g.kseg = H;
    g.groups = gl.groups;
    g.ngroups = gl.ngroups;
    g.n_mb = L / 256;
    g.kb = 2 * H / XBK;
    g.c_recv = c_recv;
    g.out = dxpool;
    g.ldo = L;
    g.rowmap = expert_rows;
    g.out_rows = pool_rows;
    g.a_mn = 1;
    g.status = status;
    return launch_group<EPI_SCATTER>(g, sms, st, "bwd_gemm_dX");
}

static size_t chunk_list_bytes(int E, int c_recv) {
    const size_t per = static_cast<size_t>((c_recv + XCHUNK - 1) / XCHUNK);
    return static_cast<size_t>(E) * (per > 0 ? per : 1) * sizeof(int4);
}

static size_t group_list_bytes(int E, int c_recv) {
    const size_t per = static_cast<size_t>((c_recv + GACC - 1) / GACC);
    return static_cast<size_t>(E) * (per > 0 ? per : 1) * sizeof(int4);
}

size_t expert_pair_chunks_bytes(int E, int c_recv) {
    return chunk_list_bytes(E, c_recv) + group_list_bytes(E, c_recv) + 16;
}

int expert_ffn_pair(int E, int c_recv, int L, int H, const uint16_t* bank,
                    const int32_t* expert_rows, const int32_t* expert_count, const uint16_t* Wg,
                    const uint16_t* Wu, const uint16_t* Wd, void* chunk_ws, uint16_t* h,
                    uint16_t* ypool, int64_t pool_rows, int32_t* status, cudaStream_t st) {
    int dev, sms;
    int rc = current_device(&dev, &sms);
    if (rc) return rc;
    if (sms < 2 || E <= 0 || c_recv <= 0 || L % 256 || H % 128 || L < 64 || H < 64) return MOE_EINVAL;
    if ((reinterpret_cast<uintptr_t>(chunk_ws) & 15) || (reinterpret_cast<uintptr_t>(bank) & 15) ||
        (reinterpret_cast<uintptr_t>(h) & 15))
        return MOE_EINVAL;
    uint8_t* ws = static_cast<uint8_t*>(chunk_ws);
    int4* chunks = reinterpret_cast<int4*>(ws);
    int4* groups = reinterpret_cast<int4*>(ws + chunk_list_bytes(E, c_recv));
    int32_t* nchunks = reinterpret_cast<int32_t*>(ws + expert_pair_chunks_bytes(E, c_recv) - 16);
    int32_t* ngroups = nchunks + 1;
    chunk_list_kernel<<<1, 1024, 0, st>>>(expert_count, E, c_recv, chunks, nchunks, groups,
                                          ngroups);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
    trace_after(st, "build_chunks");

    if (MOE_XPAIR_TM) {
        GParams g;
        std::memset(&g, 0, sizeof(g));
        if (map_gateup_il(&g.mapW, Wg, Wu, E, H, L, &g.gate_hi) == MOE_OK) {
            for (int i = 0; i < XNMAP; ++i)
                if ((rc = map3(&g.mapX[i], bank, L, c_recv, E, L, static_cast<uint64_t>(c_recv) * L,
                               XHSTEP * (i + 1))))
                    return rc;
            g.groups = groups;
            g.ngroups = ngroups;
            g.n_mb = H / 128;
            g.zpe = H / 16;
            g.kb = L / XBK;
            g.c_recv = c_recv;
            g.out = h;
            g.ldo = H;
            g.status = status;
            if ((rc = launch_group<EPI_SWIGLU>(g, sms, st, "gemm_expert_gateup"))) return rc;
            return launch_down(E, c_recv, L, H, Wd, chunks, nchunks, groups, ngroups, h, expert_rows,
                               ypool, pool_rows, status, sms, st);
        }
    }
    XParams a;
    std::memset(&a, 0, sizeof(a));
#ifndef MOE_XPAIR_ONE_WLOAD
#define MOE_XPAIR_ONE_WLOAD 1
#endif
    if (MOE_XPAIR_ONE_WLOAD && map_gateup(&a.mapW0, Wg, Wu, E, H, L, &a.gate_hi) == MOE_OK) {
        a.wpair = 1;
    } else {   // two boxes a stage: the gate rows, then the up rows
        if ((rc = map3(&a.mapW0, Wg, L, H, E, L, static_cast<uint64_t>(H) * L, 64))) return rc;
        if ((rc = map3(&a.mapW1, Wu, L, H, E, L, static_cast<uint64_t>(H) * L, 64))) return rc;
        a.wpair = 0;
        a.gate_hi = 0;
    }
    a.hblk = H / 64;
    for (int i = 0; i < XNMAP; ++i)
        if ((rc = map3(&a.mapX[i], bank, L, c_recv, E, L, static_cast<uint64_t>(c_recv) * L,
                       XHSTEP * (i + 1))))
            return rc;
    a.chunks = chunks;
    a.nchunks = nchunks;
    a.n_mb = H / 128;
    a.kb = (L + XBK - 1) / XBK;
    a.c_recv = c_recv;
    a.out = h;
    a.ldo = H;
    a.status = status;
    if ((rc = launch_pair<EPI_SWIGLU>(a, sms, st, "gemm_expert_gateup"))) return rc;
    return launch_down(E, c_recv, L, H, Wd, chunks, nchunks, groups, ngroups, h, expert_rows, ypool,
                       pool_rows, status, sms, st);
}

}  // namespace moe
