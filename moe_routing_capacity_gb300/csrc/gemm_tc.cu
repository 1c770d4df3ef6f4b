// gemm_tc.cu -- the layer's dense contractions on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in TMEM, operands staged in shared memory
// by TMA or, for gathered expert rows, by cp.async).
//
// One persistent kernel template serves every contraction of the layer:
//   router logits      x [T,d] . Wr [E,d]^T               -> fp32 (+ bias)
//   latent down-proj   x [T,d] . W_ld [L,d]^T             -> bf16 z
//   shared gate/up     x [T,d] . [Wsg | Wsu]^T            -> bf16 silu(g)*u
//   up-proj + shared   [c | a_0 | a_1] . [W_lu | Wsd_0 | Wsd_1]^T -> bf16 out
//   expert gate/up     pool rows of expert e (gathered) . [Wg_e | Wu_e]^T -> h_e
//   expert down        h_e . Wd_e^T  -> Y, scattered back to the pool rows
//
// CTA = 128 x BN output tile, K in blocks of 64 (one 128-byte swizzle row).
// Warp roles: warp 0 issues TMA loads (one elected lane), warp 1 issues
// tcgen05.mma (one lane), warp 2 owns the TMEM allocation, warps 4-7 run the
// epilogue (warp 4+q reads TMEM lanes 32q..32q+31), and for gathered A
// warps 8-11 copy the tile's 128 rows (indices from the expert's row list)
// with cp.async, eight threads per 128-byte row segment so every global
// access is a full, coalesced line.  Two TMEM accumulators let the epilogue
// of tile i overlap the main loop of tile i+1.  In the wave-pipelined
// dispatch, warps 12-15 of the gathered-A kernel copy the payload rows of
// waves 1.. into the pool while the tiles of wave 0 compute; the row gather
// of a later wave's tile first waits for every CTA's copies of that wave.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "pack.cuh"

namespace moe {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_STAGE_BYTES = BM * BK * 2;   // 16 KB

// Shared-memory rings: A stages (128 x 64 bf16, 16 KB) and B stages (BN x 64
// bf16) have their own depths.  Gathered A (cp.async, latency-bound) gets a
// deeper ring than the TMA-fed B.
// ring depth of the CTA-pair products without fp32 staging (32 KB a stage)
#ifndef MOE_PAIR_STAGES
#define MOE_PAIR_STAGES 7
#endif
#ifndef MOE_GATHER_A_STAGES
#define MOE_GATHER_A_STAGES 6
#endif
#ifndef MOE_GATHER_B_STAGES
#define MOE_GATHER_B_STAGES 4
#endif
#ifndef MOE_GROUPED_A_STAGES
#define MOE_GROUPED_A_STAGES 4
#endif
#ifndef MOE_GROUPED_B_STAGES
#define MOE_GROUPED_B_STAGES 4
#endif

// CG2: the tile is computed by a CTA pair (cta_group::2, M = 256); each CTA
// stages its 128 rows of A and half (BN/2 rows) of the B tile.
template <int BN, int AMODE, int EPI, bool CG2 = false>
struct TileCfg {
    static constexpr int B_ROWS = CG2 ? BN / 2 : BN;   // B rows staged by this CTA
    static constexpr int B_STAGE_BYTES = B_ROWS * BK * 2;
    static constexpr int B_STAGES = CG2                      ? (EPI == EPI_F32 ? 6 : MOE_PAIR_STAGES)
                                    : (BN == 384)            ? 3
                                    : (BN != 256)            ? 6
                                    : (AMODE == A_GATHER)    ? MOE_GATHER_B_STAGES
                                    : (AMODE == A_GROUPED)   ? (EPI == EPI_F32 ? 4 : MOE_GROUPED_B_STAGES)
                                                             : 4;
    static constexpr int A_STAGES = CG2                    ? (EPI == EPI_F32 ? 6 : MOE_PAIR_STAGES)
                                    : (AMODE == A_GATHER)  ? MOE_GATHER_A_STAGES
                                    : (AMODE == A_GROUPED) ? (EPI == EPI_F32 ? 4 : MOE_GROUPED_A_STAGES)
                                                           : B_STAGES;
    static_assert(AMODE != A_GATHER || A_STAGES >= 2, "the row gather needs two stages");
    // two accumulators (double buffering) when they fit in the 512 TMEM
    // columns; the 384-wide router tile gets one
    static constexpr int NACC = (2 * BN <= 512) ? 2 : 1;
    static constexpr int TMEM_COLS = (BN <= 256) ? 2 * BN : 512;
    // barriers (full/empty per stage, two accumulator pairs, done) and the
    // words after them (TMEM slot, abort flag, gather wave, two pace words),
    // rounded up to 64 bytes
    static constexpr int BAR_BYTES = ((2 * (A_STAGES + B_STAGES) + 5) * 8 + 5 * 4 + 63) / 64 * 64;
    // fp32 output: each epilogue warp stages 32 x 32 blocks in shared memory
    // (two, so one can be written while the other is being stored)
    static constexpr int STG_BYTES = (EPI == EPI_F32) ? 2 * 4 * 32 * 32 * 4 : 0;
    static constexpr int SMEM_BYTES =
        1024 + A_STAGES * A_STAGE_BYTES + B_STAGES * B_STAGE_BYTES + STG_BYTES + BAR_BYTES;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct KParams {
    CUtensorMap mapA[4];
    CUtensorMap mapB[4];
    CUtensorMap mapBup;
    CUtensorMap omap;       // fp32 output, box 32 x 32, 128-byte swizzle
    int omap_rank;          // 2 (dense), 3 (per-group), or 0: plain stores
    int nseg;
    int seg_kb[5];          // k-block prefix over segments
    long long M;
    int N;
    int K0;                 // K of segment 0 (gather bound)
    int n_tiles_n;
    int m_tiles;            // dense tile rows
    const int2* tile_list;
    const int* tile_count;
    const int* rowmap;
    const int* counts;
    const int* goff;        // optional per-group first row (ragged groups)
    const int* rmoff;       // optional per-group first row-map entry (else goff)
    const int* kgoff;       // optional per-group K row range (uniform groups)
    const int* kcount;      // optional per-group rows contracted (uniform groups, 3-D
                            // operands whose rows past the count are zero)
    int rowmap_ld;
    const uint16_t* gather_src;
    long long gather_pitch;
    long long gather_rows;  // rows of the gather source / scatter destination (checks)
    void* out;
    long long ldo;
    long long out_gstride;
    const float* bias;
    int* status;
    int nsplit;
    int N2;
    void* out2;
    long long ldo2;
    const uint16_t* aux;
    int uniform_groups;
    // pool fill riding along (wp_a.pool non-null): wave pipeline (gathered
    // A, wp_ready non-null: warps 12-15 copy waves 1..W-1 while the tiles of
    // earlier waves compute) or the whole pack in a dense product (warps 8-11)
    int* wp_ready;
    DispatchGeom wp_g;
    PackArgs wp_a;
    int raster_gn;          // dense tiles: column blocks a band (0: row tile by row tile)
};

// Limit of the wave pipeline's wait for every CTA's count of a wave.  In
// checked builds a test can shorten it from the host, so that the wait runs
// out on legitimate work and the unwinding path is exercised; only this wait
// reads it (the waits that drain copies and MMAs keep their own limits).
#if MOE_CHECK
static __device__ unsigned long long g_wave_wait_limit_ns = kWaitTimeoutNs;
__device__ __forceinline__ uint64_t wave_wait_limit() { return g_wave_wait_limit_ns; }
#else
__device__ __forceinline__ uint64_t wave_wait_limit() { return kWaitTimeoutNs; }
#endif

int set_wave_wait_limit(unsigned long long ns) {
#if MOE_CHECK
    return cudaMemcpyToSymbol(g_wave_wait_limit_ns, &ns, sizeof(ns)) == cudaSuccess ? MOE_OK
                                                                                    : MOE_ECUDA;
#else
    (void)ns;
    return MOE_EINVAL;
#endif
}

// The pack run by extra warps of a GEMM launch (pack_token), tokens dealt
// out over the grid's copy warps (cw of ncw in this CTA): the receiver
// decisions (decide) and the copies of wave w (every wave if w < 0), with
// streaming loads and stores so the product's tiles keep their L2 lines.
// pace (optional): token i of this warp's n goes once the CTA has started
// i * tiles / (n + 1) of its tiles (pace[0]: tiles started, pace[1]: this
// CTA's tile count), spreading the copy over the product.
__device__ __forceinline__ void pack_tokens(const KParams& p, bool decide, int w, int cw, int ncw,
                                            int lane, const volatile int* pace = nullptr,
                                            const volatile int* abort_flag = nullptr) {
    const long long nwarps = static_cast<long long>(ncw) * gridDim.x;
    const long long first = static_cast<long long>(ncw) * blockIdx.x + cw;
    const long long ntok = first < p.wp_g.T ? (p.wp_g.T - first + nwarps - 1) / nwarps : 0;
    long long i = 0;
    for (long long t = first; t < p.wp_g.T; t += nwarps, ++i) {
        if (pace) {
            const long long need = i * pace[1] / (ntok + 1);
            if (pace[0] <= need) {
                const uint64_t t0 = globaltimer_ns();
                while (pace[0] <= need && !*abort_flag && globaltimer_ns() - t0 < kWaitTimeoutNs)
                    __nanosleep(1000);
            }
        }
        pack_token<4, true>(p.wp_g, p.wp_a, t, lane, decide, w);
    }
}

template <int AMODE>
__device__ __forceinline__ int num_tiles(const KParams& p) {
    if (AMODE == A_DENSE) return p.m_tiles * p.n_tiles_n;
    if (p.uniform_groups) return p.uniform_groups * p.m_tiles * p.n_tiles_n;
    return (*reinterpret_cast<const volatile int*>(p.tile_count)) * p.n_tiles_n;
}

template <int AMODE>
__device__ __forceinline__ void decode_tile(const KParams& p, int tile, int& g, int& m0, int& nb) {
    const int entry = tile / p.n_tiles_n;
    nb = tile - entry * p.n_tiles_n;
    if (AMODE == A_DENSE) {
        g = 0;
        int m = entry;
        if (p.raster_gn > 0) {
            // bands of raster_gn column blocks: every row tile crosses one band
            // before the next band starts, so the band's B stays in L2 while
            // A streams (A is read once a band instead of B once a row tile)
            const int gn = p.raster_gn;
            const int full = (p.n_tiles_n / gn) * gn * p.m_tiles;   // tiles in whole bands
            int band, r, width;
            if (tile < full) {
                band = tile / (gn * p.m_tiles);
                r = tile - band * gn * p.m_tiles;
                width = gn;
            } else {
                band = p.n_tiles_n / gn;
                r = tile - full;
                width = p.n_tiles_n - band * gn;
            }
            m = r / width;
            nb = band * gn + (r - m * width);
        }
        m0 = m * BM;
    } else if (p.uniform_groups) {
        g = entry / p.m_tiles;
        m0 = (entry - g * p.m_tiles) * BM;
    } else {
        const int2 te = p.tile_list[entry];
        g = te.x;
        m0 = te.y;
    }
}

__device__ __forceinline__ float silu_f(float g) { return silu_fast(g); }

// First row-map entry of group g.
__device__ __forceinline__ long long rowmap_base(const KParams& p, int g) {
    if (p.rmoff) return p.rmoff[g];
    if (p.goff) return p.goff[g];
    return static_cast<long long>(g) * p.rowmap_ld;
}

// K blocks of a tile of group g: the whole contraction, or the group's own
// row range of flat MN-major operands.
__device__ __forceinline__ int tile_kblocks(const KParams& p, int g, int kb_total) {
    if (p.kgoff) return (p.kgoff[g + 1] - p.kgoff[g]) / 64;
    if (p.kcount) {
        const int kb = (p.kcount[g] + BK - 1) / BK;
        return kb < kb_total ? kb : kb_total;
    }
    return kb_total;
}

// MAJ bit 0: A is MN-major (stored [K, M], M contiguous); bit 1: B is
// MN-major (stored [K, N]).  MN-major tiles arrive as 64 x 64 TMA boxes, one
// per 64 M/N elements, 8 KB apart.
// CG2: launched in clusters of two; the pair computes 256 x BN tiles with
// tcgen05.mma.cta_group::2 issued by the even CTA.  Both CTAs' TMA loads count
// on the even CTA's full barriers; the MMA commits arrive on the empty, full
// and done barriers of both CTAs; both CTAs' epilogues arrive on the even
// CTA's accumulator-free barriers.
template <int BN, int AMODE, int EPI, int MAJ, bool CG2>
__global__ void __launch_bounds__(AMODE == A_GATHER ? 512 : 384, 1)
    gemm_tc_kernel(const __grid_constant__ KParams p) {
    using C = TileCfg<BN, AMODE, EPI, CG2>;
    static_assert(!CG2 || (AMODE == A_DENSE && BN == 256 &&
                           (EPI == EPI_BF16 || EPI == EPI_F32 || (EPI == EPI_SPLIT && MAJ == 0) ||
                            ((EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) && !(MAJ & 2)))),
                  "CTA pairs: dense tiles; bf16, fp32, split, SwiGLU (K-major B) epilogues");
    constexpr int AST = C::A_STAGES;
    constexpr int BST = C::B_STAGES;
    constexpr bool B3D = (AMODE != A_DENSE);
    constexpr bool A_MN = (MAJ & 1) != 0;
    constexpr bool B_MN = (MAJ & 2) != 0;
    static_assert(!A_MN || AMODE != A_GATHER, "MN-major A: TMA tiles only");
    static_assert(!B_MN || (BN <= 256 && EPI != EPI_SPLIT), "MN-major B: plain tiles only");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sbase = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sA = sbase;
    uint8_t* sB = sbase + AST * A_STAGE_BYTES;
    uint8_t* sStg = sB + BST * C::B_STAGE_BYTES;   // 1024-aligned fp32 staging
    uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + C::STG_BYTES);
    uint64_t* fullA = bars;
    uint64_t* emptyA = fullA + AST;
    uint64_t* fullB = emptyA + AST;
    uint64_t* emptyB = fullB + BST;
    uint64_t* tfull = emptyB + BST;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // wave pipeline: the wave of the tiles this CTA's row gather has reached
    // (W once it has no more), which paces the copies of the later waves
    volatile int* gather_wave = abort_flag + 1;
    // dense products carrying the pool fill: tiles this CTA's producer has
    // started, and this CTA's tile count (the copy's pace)
    volatile int* tiles_pace = gather_wave + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA pairs: rank in the pair; tiles are dealt out per pair
    const uint32_t crank = CG2 ? cluster_ctarank() : 0u;
    const bool leader = crank == 0;
    const int cta0 = CG2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int ncta = CG2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < AST; ++s) {
            mbar_init(&fullA[s], AMODE == A_GATHER ? 128 : 1);
            mbar_init(&emptyA[s], 1);
        }
        for (int s = 0; s < BST; ++s) {
            mbar_init(&fullB[s], 1);
            mbar_init(&emptyB[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], CG2 ? 256 : 128);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        *gather_wave = 0;
        tiles_pace[0] = 0;
        {
            const int nt = num_tiles<AMODE>(p);
            tiles_pace[1] = nt > cta0 ? (nt - cta0 + ncta - 1) / ncta : 0;
        }
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < p.nseg; ++s) {
            tma_prefetch_map(&p.mapB[s]);
            if (AMODE != A_GATHER) tma_prefetch_map(&p.mapA[s]);
        }
    }
    if (warp == 2) {
        if constexpr (CG2) {
            tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (CG2) cluster_sync();   // the peer's barriers exist before any remote arrival
    const uint32_t tmem_base = *tmem_slot;
    const int kb_total = p.seg_kb[p.nseg];

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const int ntiles = num_tiles<AMODE>(p);
            uint32_t sa = 0, pa = 0, sb = 0, pb = 0;
            uint32_t armedA = 0, parA = 0, armedB = 0, parB = 0;   // for unwinding
            bool ok = true;
            int started = 0;
            for (int tile = cta0; ok && tile < ntiles; tile += ncta) {
                tiles_pace[0] = ++started;
                int g, m0, nb;
                decode_tile<AMODE>(p, tile, g, m0, nb);
                if (CG2) m0 = 2 * m0 + static_cast<int>(crank) * BM;
                const int kbt = tile_kblocks(p, g, kb_total);
                const int k0 = p.kgoff ? p.kgoff[g] : 0;   // first K row (flat operands)
                int seg = 0;
                for (int kb = 0; kb < kbt; ++kb) {
                    while (kb >= p.seg_kb[seg + 1]) ++seg;
                    const int kx = (kb - p.seg_kb[seg]) * BK;
                    if (AMODE != A_GATHER) {
                        if (!mbar_wait(&emptyA[sa], pa ^ 1u, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        const uint32_t a_dst = smem_u32(sA + sa * A_STAGE_BYTES);
                        if constexpr (CG2) {   // both halves count on the even CTA's barrier
                            if (leader) mbar_arrive_expect_tx(&fullA[sa], 2 * A_STAGE_BYTES);
                            const uint32_t fa = mapa_shared(smem_u32(&fullA[sa]), 0);
                            if (A_MN) {   // two 64-row boxes of the MN-major A
                                tma_load_2d_pair(a_dst, &p.mapA[seg], fa, m0, kx);
                                tma_load_2d_pair(a_dst + 8192, &p.mapA[seg], fa, m0 + 64, kx);
                            } else {
                                tma_load_2d_pair(a_dst, &p.mapA[seg], fa, kx, m0);
                            }
                        } else {
                            mbar_arrive_expect_tx(&fullA[sa], A_STAGE_BYTES);
                        }
                        if (!CG2 || leader) {
                            armedA |= 1u << sa;
                            parA = (parA & ~(1u << sa)) | (pa << sa);
                        }
                        if constexpr (CG2) {
                        } else if (A_MN && AMODE == A_DENSE) {
                            tma_load_2d(a_dst, &p.mapA[seg], &fullA[sa], m0, kx);
                            tma_load_2d(a_dst + 8192, &p.mapA[seg], &fullA[sa], m0 + 64, kx);
                        } else if (A_MN && p.kgoff) {
                            tma_load_2d(a_dst, &p.mapA[seg], &fullA[sa], m0, k0 + kx);
                            tma_load_2d(a_dst + 8192, &p.mapA[seg], &fullA[sa], m0 + 64, k0 + kx);
                        } else if (A_MN) {
                            tma_load_3d(a_dst, &p.mapA[seg], &fullA[sa], m0, kx, g);
                            tma_load_3d(a_dst + 8192, &p.mapA[seg], &fullA[sa], m0 + 64, kx, g);
                        } else if (AMODE == A_DENSE)
                            tma_load_2d(a_dst, &p.mapA[seg], &fullA[sa], kx, m0);
                        else if (p.goff)   // ragged groups: rows of one flat 2-D matrix
                            tma_load_2d(a_dst, &p.mapA[seg], &fullA[sa], kx, p.goff[g] + m0);
                        else
                            tma_load_3d(a_dst, &p.mapA[seg], &fullA[sa], kx, m0, g);
                        if (++sa == AST) {
                            sa = 0;
                            pa ^= 1u;
                        }
                    }
                    if (!mbar_wait(&emptyB[sb], pb ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t b_dst = smem_u32(sB + sb * C::B_STAGE_BYTES);
                    if constexpr (CG2) {
                        if (leader) mbar_arrive_expect_tx(&fullB[sb], 2 * C::B_STAGE_BYTES);
                    } else {
                        mbar_arrive_expect_tx(&fullB[sb], C::B_STAGE_BYTES);
                    }
                    if (!CG2 || leader) {
                        armedB |= 1u << sb;
                        parB = (parB & ~(1u << sb)) | (pb << sb);
                    }
                    if constexpr (CG2) {
                        // this CTA's half of the B tile: SwiGLU gate rows (even
                        // CTA) or up rows (odd CTA); otherwise rows crank*BN/2..
                        const uint32_t fb = mapa_shared(smem_u32(&fullB[sb]), 0);
                        if (B_MN) {   // two 64-column boxes of the MN-major B
                            const int n = nb * BN + static_cast<int>(crank) * (BN / 2);
                            tma_load_2d_pair(b_dst, &p.mapB[seg], fb, n, kx);
                            tma_load_2d_pair(b_dst + 8192, &p.mapB[seg], fb, n + 64, kx);
                        } else if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD)
                            tma_load_2d_pair(b_dst, crank ? &p.mapBup : &p.mapB[0], fb, kx,
                                             nb * (BN / 2));
                        else if (EPI == EPI_SPLIT && nb >= p.nsplit)
                            tma_load_2d_pair(b_dst, &p.mapBup, fb, kx,
                                             (nb - p.nsplit) * BN + static_cast<int>(crank) * (BN / 2));
                        else
                            tma_load_2d_pair(b_dst, &p.mapB[seg], fb, kx,
                                             nb * BN + static_cast<int>(crank) * (BN / 2));
                    } else if (B_MN) {
                        // BN/64 boxes of 64 N x 64 K; SwiGLU: gate then up halves
#pragma unroll
                        for (int h = 0; h < BN / 64; ++h) {
                            constexpr bool PAIR = EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD;
                            const bool up = PAIR && h >= BN / 128;
                            const int n = PAIR ? nb * (BN / 2) + (h % (BN / 128)) * 64
                                               : nb * BN + h * 64;
                            const CUtensorMap* mp = up ? &p.mapBup : &p.mapB[seg];
                            if (B3D && p.kgoff)
                                tma_load_2d(b_dst + h * 8192, mp, &fullB[sb], n, k0 + kx);
                            else if (B3D)
                                tma_load_3d(b_dst + h * 8192, mp, &fullB[sb], n, kx, g);
                            else
                                tma_load_2d(b_dst + h * 8192, mp, &fullB[sb], n, kx);
                        }
                    } else if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) {
                        const int n_half = nb * (BN / 2);
                        const uint32_t b_dst2 = b_dst + (BN / 2) * BK * 2;
                        if (B3D) {
                            tma_load_3d(b_dst, &p.mapB[0], &fullB[sb], kx, n_half, g);
                            tma_load_3d(b_dst2, &p.mapBup, &fullB[sb], kx, n_half, g);
                        } else {
                            tma_load_2d(b_dst, &p.mapB[0], &fullB[sb], kx, n_half);
                            tma_load_2d(b_dst2, &p.mapBup, &fullB[sb], kx, n_half);
                        }
                    } else if (EPI == EPI_SPLIT) {
                        if (nb < p.nsplit)
                            tma_load_2d(b_dst, &p.mapB[0], &fullB[sb], kx, nb * BN);
                        else
                            tma_load_2d(b_dst, &p.mapBup, &fullB[sb], kx, (nb - p.nsplit) * BN);
                    } else if (BN == 384) {
#pragma unroll
                        for (int h = 0; h < 3; ++h)
                            tma_load_2d(b_dst + h * 128 * BK * 2, &p.mapB[seg], &fullB[sb], kx,
                                        nb * BN + h * 128);
                    } else {
                        if (B3D)
                            tma_load_3d(b_dst, &p.mapB[seg], &fullB[sb], kx, nb * BN, g);
                        else
                            tma_load_2d(b_dst, &p.mapB[seg], &fullB[sb], kx, nb * BN);
                    }
                    if (++sb == BST) {
                        sb = 0;
                        pb ^= 1u;
                    }
                }
            }
            tiles_pace[0] = 1 << 30;   // no more tiles: the copy may finish
            if (!ok || *abort_flag) {
                // Unwinding: let every armed TMA load land before the CTA exits.
                volatile int no_abort = 0;
                for (int s = 0; s < BST; ++s)
                    if (armedB >> s & 1u)
                        mbar_wait(&fullB[s], (parB >> s) & 1u, &no_abort, nullptr, 20000000ull);
                for (int s = 0; s < AST; ++s)
                    if (armedA >> s & 1u)
                        mbar_wait(&fullA[s], (parA >> s) & 1u, &no_abort, nullptr, 20000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        bool issuer = lane == 0;
        if constexpr (CG2) {
            if (!leader && lane == 0) {
                // the even CTA issues the pair's MMAs; wait until they are all
                // done (they write this CTA's TMEM and read its shared memory)
                volatile int no_abort = 0;
                mbar_wait(done, 0, &no_abort, p.status);
                issuer = false;
            }
        }
        if (issuer) {
            const int ntiles = num_tiles<AMODE>(p);
            constexpr int N0 = BN <= 256 ? BN : 256;          // first MMA's N
            constexpr uint32_t idesc = idesc_bf16_f32(CG2 ? 2 * BM : BM, N0, A_MN, B_MN);
            constexpr uint32_t idesc_hi = idesc_bf16_f32(BM, BN > 256 ? BN - 256 : 16);
            // descriptor step per 16-wide K slice: 32 B along a K-major row,
            // 16 rows of 128 B down an MN-major box
            constexpr uint32_t a_step = A_MN ? (2048u >> 4) : (32u >> 4);
            constexpr uint32_t b_step = B_MN ? (2048u >> 4) : (32u >> 4);
            uint32_t sa = 0, pa = 0, sb = 0, pb = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool ok = true;
            for (int tile = cta0; ok && tile < ntiles; tile += ncta) {
                int kbt = kb_total;
                if (p.kgoff || p.kcount) {
                    int g, m0, nb;
                    decode_tile<AMODE>(p, tile, g, m0, nb);
                    kbt = tile_kblocks(p, g, kb_total);
                }
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < kbt; ++kb) {
                    if (!mbar_wait(&fullA[sa], pa, abort_flag, p.status) ||
                        !mbar_wait(&fullB[sb], pb, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    // gathered rows came through cp.async (generic proxy): make
                    // them visible to the tensor core's reads
                    if constexpr (AMODE == A_GATHER) fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t a_s = smem_u32(sA + sa * A_STAGE_BYTES);
                    const uint32_t b_s = smem_u32(sB + sb * C::B_STAGE_BYTES);
                    const uint64_t ad = A_MN ? sdesc_mn_sw128(a_s) : sdesc_k_sw128(a_s);
                    const uint64_t bd = B_MN ? sdesc_mn_sw128(b_s) : sdesc_k_sw128(b_s);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        if constexpr (CG2) {
                            mma_bf16_pair(d_tmem, ad + a_step * kk, bd + b_step * kk, idesc,
                                          (kb | kk) != 0 ? 1u : 0u);
                        } else {
                            mma_bf16(d_tmem, ad + a_step * kk, bd + b_step * kk, idesc,
                                     (kb | kk) != 0 ? 1u : 0u);
                        }
                        if constexpr (BN > 256)   // columns 256.. from B rows 256.. (32 KB further)
                            mma_bf16(d_tmem + 256, ad + 2u * kk, bd + (32768u >> 4) + 2u * kk,
                                     idesc_hi, (kb | kk) != 0 ? 1u : 0u);
                    }
                    if constexpr (CG2) {   // both CTAs' stages are free once these MMAs finish
                        mma_commit_pair(&emptyA[sa]);
                        mma_commit_pair(&emptyB[sb]);
                    } else {
                        mma_commit(&emptyA[sa]);
                        mma_commit(&emptyB[sb]);
                    }
                    if (++sa == AST) {
                        sa = 0;
                        pa ^= 1u;
                    }
                    if (++sb == BST) {
                        sb = 0;
                        pb ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (CG2)
                    mma_commit_pair(&tfull[acc]);
                else
                    mma_commit(&tfull[acc]);
                if (++acc == C::NACC) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Every MMA this CTA issued must finish before TMEM is released.
            if constexpr (CG2)
                mma_commit_pair(done);
            else
                mma_commit(done);
            volatile int no_abort = 0;
            mbar_wait(done, 0, &no_abort, p.status);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ epilogue
        const int q = warp - 4;
        const int r_local = q * 32 + lane;
        const int ntiles = num_tiles<AMODE>(p);
        uint32_t acc = 0, acc_phase = 0;
        uint32_t nstore = 0;   // fp32 tile stores this warp committed (lane 0)
        // the pair's accumulator-free barrier lives in the even CTA
        const uint32_t tempty_c0 = CG2 ? mapa_shared(smem_u32(&tempty[0]), 0) : 0u;
        for (int tile = cta0; tile < ntiles; tile += ncta) {
            int g, m0, nb;
            decode_tile<AMODE>(p, tile, g, m0, nb);
            if (CG2) m0 = 2 * m0 + static_cast<int>(crank) * BM;
            if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status)) break;
            tc_fence_after();
            const uint32_t tl = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            const int m = m0 + r_local;
            bool row_ok;
            long long orow;
            if (AMODE == A_DENSE || p.uniform_groups) {
                row_ok = m < p.M;
                orow = m;
            } else {
                row_ok = m < p.counts[g];
                orow = m;
                if (EPI == EPI_SCATTER && row_ok) {
                    orow = p.rowmap[rowmap_base(p, g) + m];
                    if (!moe_check(orow >= 0 && orow < p.gather_rows, 1006)) row_ok = false;
                }
            }
            // element offset of this row in the output (and in aux / out2):
            // dense or scattered rows, or row m of group g
            const long long obase =
                (AMODE == A_DENSE || EPI == EPI_SCATTER)
                    ? orow * p.ldo
                    : (p.goff ? (p.goff[g] + orow) * p.ldo
                              : static_cast<long long>(g) * p.out_gstride + orow * p.ldo);
            if (EPI == EPI_SPLIT && nb >= p.nsplit) {
                float* out = reinterpret_cast<float*>(p.out2) + orow * p.ldo2;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tl + c * 32, r);
                    const int col0 = (nb - p.nsplit) * BN + c * 32;
                    if (row_ok && col0 < p.N2) {
                        if (col0 + 32 <= p.N2 && (p.ldo2 & 3) == 0) {
#pragma unroll
                            for (int v = 0; v < 8; ++v) {
                                float4 f;
                                f.x = __uint_as_float(r[4 * v]);
                                f.y = __uint_as_float(r[4 * v + 1]);
                                f.z = __uint_as_float(r[4 * v + 2]);
                                f.w = __uint_as_float(r[4 * v + 3]);
                                if (p.bias) {
                                    const float4 b = *reinterpret_cast<const float4*>(p.bias + col0 + 4 * v);
                                    f.x += b.x; f.y += b.y; f.z += b.z; f.w += b.w;
                                }
                                *reinterpret_cast<float4*>(out + col0 + 4 * v) = f;
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int col = col0 + i;
                                if (col < p.N2) {
                                    float v = __uint_as_float(r[i]);
                                    if (p.bias) v += p.bias[col];
                                    out[col] = v;
                                }
                            }
                        }
                    }
                }
            } else if (EPI == EPI_F32) {
                // a group with an empty K range contributes a zero tile
                const bool zero_tile = (p.kgoff || p.kcount) && tile_kblocks(p, g, kb_total) == 0;
                if (p.omap_rank) {
                    // Lane i holds row 32q + i.  Each 32 x 32 block is written
                    // to shared memory in the 128-byte-swizzled layout of the
                    // output map (16-byte chunk v of row i at chunk v ^ (i % 8):
                    // conflict-free) and stored by one TMA tile store; two
                    // buffers per warp let the next block be written while
                    // the previous one is still being read out.
                    const int row0 = m0 + q * 32;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tl + c * 32, r);
                        const int col0 = nb * BN + c * 32;
                        float4* buf = reinterpret_cast<float4*>(sStg) + (q * 2 + (nstore & 1)) * 256;
                        if (lane == 0 && nstore >= 2) bulk_wait_read1();
                        __syncwarp();
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            float4 f = make_float4(__uint_as_float(r[4 * v]),
                                                   __uint_as_float(r[4 * v + 1]),
                                                   __uint_as_float(r[4 * v + 2]),
                                                   __uint_as_float(r[4 * v + 3]));
                            if (zero_tile) f = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (p.bias) {
                                const int cc = col0 + 4 * v;
                                if (cc + 0 < p.N) f.x += p.bias[cc + 0];
                                if (cc + 1 < p.N) f.y += p.bias[cc + 1];
                                if (cc + 2 < p.N) f.z += p.bias[cc + 2];
                                if (cc + 3 < p.N) f.w += p.bias[cc + 3];
                            }
                            buf[lane * 8 + (v ^ (lane & 7))] = f;
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (col0 < p.N && row0 < p.M) {   // warp-uniform
                            if (lane == 0) {
                                if (p.omap_rank == 3)
                                    tma_store_3d(&p.omap, smem_u32(buf), col0, row0, g);
                                else
                                    tma_store_2d(&p.omap, smem_u32(buf), col0, row0);
                                bulk_commit();
                            }
                            ++nstore;   // every lane: the buffer choice stays uniform
                        }
                    }
                } else {
                // Lane i holds row 32q + i.  Each 32-column block goes through
                // shared memory (16-byte chunks XOR-swizzled by row, so both
                // the row-wise writes and the column-wise reads are free of
                // bank conflicts); then lane l stores columns 4(l%8)..+3 of
                // rows 4j + l/8: one warp store covers four whole rows.
                float4* stg = reinterpret_cast<float4*>(sStg) + q * 256;
                float* out = reinterpret_cast<float*>(p.out);
                const int rsub = lane >> 3, csub = lane & 7;
                long long rbase[8];
                uint32_t rok = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    rbase[j] = __shfl_sync(0xffffffffu, obase, 4 * j + rsub);
                    rok |= (__shfl_sync(0xffffffffu, row_ok ? 1 : 0, 4 * j + rsub) ? 1u : 0u) << j;
                }
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tl + c * 32, r);
                    if (zero_tile) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = 0u;
                    }
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        stg[lane * 8 + (v ^ (lane & 7))] =
                            make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                        __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                    __syncwarp();
                    const int col = nb * BN + c * 32 + 4 * csub;
                    float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (p.bias) {
                        if (col + 0 < p.N) bv.x = p.bias[col + 0];
                        if (col + 1 < p.N) bv.y = p.bias[col + 1];
                        if (col + 2 < p.N) bv.z = p.bias[col + 2];
                        if (col + 3 < p.N) bv.w = p.bias[col + 3];
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int rr = 4 * j + rsub;
                        float4 f = stg[rr * 8 + (csub ^ (rr & 7))];
                        f.x += bv.x; f.y += bv.y; f.z += bv.z; f.w += bv.w;
                        if (!(rok >> j & 1u) || col >= p.N) continue;
                        float* dst = out + rbase[j] + col;
                        if (col + 4 <= p.N && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                            *reinterpret_cast<float4*>(dst) = f;
                        } else {
                            dst[0] = f.x;
                            if (col + 1 < p.N) dst[1] = f.y;
                            if (col + 2 < p.N) dst[2] = f.z;
                            if (col + 3 < p.N) dst[3] = f.w;
                        }
                    }
                    __syncwarp();
                }
                }
            } else if (EPI == EPI_SWIGLU_BWD) {
                // recomputed g (columns 0..BN/2) and u (BN/2..BN) of hidden units
                // nb*BN/2 + c; incoming dh; dg = dh u silu'(g), du = dh silu(g)
                uint16_t* dgo = reinterpret_cast<uint16_t*>(p.out) + obase;
                uint16_t* duo = reinterpret_cast<uint16_t*>(p.out2) + obase;
                const uint16_t* dhi = p.aux + obase;
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t gr[32], ur[32];
                    tmem_ld32(tl + c * 32, gr);
                    tmem_ld32(tl + BN / 2 + c * 32, ur);
                    const int col0 = nb * (BN / 2) + c * 32;
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int col = col0 + 8 * v;
                            if (col >= p.N) continue;
                            const uint4 hv = *reinterpret_cast<const uint4*>(dhi + col);
                            const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
                            uint32_t pg[4], pu[4];
#pragma unroll
                            for (int q2 = 0; q2 < 4; ++q2) {
                                float dg2[2], du2[2];
#pragma unroll
                                for (int e2 = 0; e2 < 2; ++e2) {
                                    const int i = 8 * v + 2 * q2 + e2;
                                    const float gg = __uint_as_float(gr[i]);
                                    const float uu = __uint_as_float(ur[i]);
                                    const float dh = e2 ? bf16_hi(hw[q2]) : bf16_lo(hw[q2]);
                                    const float sig = 1.0f / (1.0f + expf(-gg));
                                    dg2[e2] = dh * uu * (sig * (1.0f + gg * (1.0f - sig)));
                                    du2[e2] = dh * (gg * sig);
                                }
                                pg[q2] = pack_bf16x2(dg2[0], dg2[1]);
                                pu[q2] = pack_bf16x2(du2[0], du2[1]);
                            }
                            *reinterpret_cast<uint4*>(dgo + col) = make_uint4(pg[0], pg[1], pg[2], pg[3]);
                            *reinterpret_cast<uint4*>(duo + col) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
                        }
                    } else if (AMODE == A_GATHER &&
                               m < (p.goff ? p.goff[g + 1] - p.goff[g] : p.out_gstride / p.ldo)) {
                        // a padding row inside the group's slab: zeros, which
                        // the weight gradients contract over
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int col = col0 + 8 * v;
                            if (col >= p.N) continue;
                            *reinterpret_cast<uint4*>(dgo + col) = make_uint4(0u, 0u, 0u, 0u);
                            *reinterpret_cast<uint4*>(duo + col) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
            } else if (EPI == EPI_SWIGLU) {
                uint16_t* out = reinterpret_cast<uint16_t*>(p.out) + obase;
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t gr[32], ur[32];
                    tmem_ld32(tl + c * 32, gr);
                    tmem_ld32(tl + BN / 2 + c * 32, ur);
                    const int col0 = nb * (BN / 2) + c * 32;
                    if (row_ok) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float h0 = silu_f(__uint_as_float(gr[2 * i])) *
                                             __uint_as_float(ur[2 * i]);
                            const float h1 = silu_f(__uint_as_float(gr[2 * i + 1])) *
                                             __uint_as_float(ur[2 * i + 1]);
                            pk[i] = pack_bf16x2(h0, h1);
                        }
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            if (col0 + 8 * v < p.N)
                                *reinterpret_cast<uint4*>(out + col0 + 8 * v) =
                                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2],
                                               pk[4 * v + 3]);
                    } else if (AMODE == A_GATHER && !p.goff && m < p.out_gstride / p.ldo) {
                        // a padding row of the expert's last tile (inside its
                        // slab of h): zeros, so the down-projection's padded
                        // MMAs multiply zeros instead of a stale row
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            if (col0 + 8 * v < p.N)
                                *reinterpret_cast<uint4*>(out + col0 + 8 * v) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            } else {   // EPI_BF16 / EPI_SCATTER
                uint16_t* out = reinterpret_cast<uint16_t*>(p.out) + obase;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tl + c * 32, r);
                    const int col0 = nb * BN + c * 32;
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            if (col0 + 8 * v < p.N) {
                                const uint4 pk = make_uint4(
                                    pack_bf16x2(__uint_as_float(r[8 * v]), __uint_as_float(r[8 * v + 1])),
                                    pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                                    pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                                    pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
                                *reinterpret_cast<uint4*>(out + col0 + 8 * v) = pk;
                            }
                        }
                    }
                }
            }
            // the accumulator's columns are read (tcgen05.wait::ld): hand them
            // back without waiting for this tile's stores to be visible
            tc_fence_before();
            if constexpr (CG2)
                mbar_arrive_cluster_relaxed(tempty_c0 + acc * 8u);
            else
                mbar_arrive_relaxed(&tempty[acc]);
            if (++acc == C::NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (EPI == EPI_F32 && lane == 0) bulk_wait_all();   // the last tile stores land
    } else if (AMODE == A_GATHER && warp >= 8 && warp < 12) {
        // ------------------------------------------------------------ row gather (A)
        // Thread t copies 16-byte chunk c = t % 8 of tile rows t/8 + 16 i,
        // i = 0..7: a warp instruction moves four whole 128-byte row segments.
        // Each thread's copies of a stage arrive on the stage's full barrier by
        // themselves once they land (cp.async.mbarrier.arrive.noinc, 128
        // arrivals a phase), so the thread moves on to the next free stage
        // at once; the MMA thread fences them into the async proxy after its
        // wait.  The next tile's row indices are fetched while this tile
        // streams.
        const int t = threadIdx.x - 256;
        const int c = t & 7;
        const int rg = t >> 3;
        const int ntiles = num_tiles<AMODE>(p);
        uint32_t sa = 0, pa = 0;
        bool ok = true;
        int nxt_row[8];
        int nxt_cnt = 0, nxt_g = 0;
        uint32_t waves_seen = 1u;   // wave 0's rows were written before this launch
        auto fetch_rows = [&](int tile) {
            int g, m0, nb;
            decode_tile<AMODE>(p, tile, g, m0, nb);
            nxt_g = g;
            nxt_cnt = p.counts[g] - m0;   // valid rows of the tile, from its first
            const int* rl = p.rowmap + m0 + rowmap_base(p, g);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int m = rg + 16 * i;
                nxt_row[i] = m < nxt_cnt ? rl[m] : 0;
                if (!moe_check(nxt_row[i] >= 0 && nxt_row[i] < p.gather_rows, 1004)) nxt_row[i] = 0;
            }
        };
        if (cta0 < ntiles) fetch_rows(cta0);
        for (int tile = cta0; ok && tile < ntiles; tile += ncta) {
            if (p.wp_ready) {   // the tile's wave: its pool rows filled by every CTA
                const int wv = (nxt_g % p.wp_g.E_l) / p.wp_g.E_w;
                if (!(waves_seen >> wv & 1u)) {
                    if (t == 0) *gather_wave = wv;   // lets this CTA copy wave wv + 1
                    if (!wait_count(p.wp_ready + wv, static_cast<int>(gridDim.x), abort_flag,
                                    p.status, wave_wait_limit())) {
                        ok = false;
                        break;
                    }
                    waves_seen |= 1u << wv;
                }
            }
            const uint16_t* src[8];
            uint32_t valid = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const bool v = rg + 16 * i < nxt_cnt;
                valid |= (v ? 1u : 0u) << i;
                src[i] = p.gather_src + static_cast<long long>(nxt_row[i]) * p.gather_pitch + c * 8;
            }
            if (tile + ncta < ntiles) fetch_rows(tile + ncta);
            for (int kb = 0; kb < kb_total; ++kb) {
                if (!mbar_wait(&emptyA[sa], pa ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                const uint32_t dst = smem_u32(sA + sa * A_STAGE_BYTES) + ((c ^ (rg & 7)) << 4);
                const int kc = kb * BK;
                const bool kin = kc + c * 8 < p.K0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t nbytes = ((valid >> i & 1u) && kin) ? 16u : 0u;
                    cp_async_16(dst + (rg + 16 * i) * 128, src[i] + (nbytes ? kc : 0), nbytes);
                }
                cp_async_arrive_noinc(&fullA[sa]);   // arrives when these copies land
                if (++sa == AST) {
                    sa = 0;
                    pa ^= 1u;
                }
            }
        }
        if (t == 0) *gather_wave = 1 << 30;   // no more tiles: copy what is left
        cp_async_commit();    // every copy (none were grouped) lands before the CTA may exit
        cp_async_wait<0>();
    } else if (AMODE == A_GATHER && warp >= 12 && p.wp_ready) {
        // ------------------------------------------------------------ pool fill, waves 1..
        // Wave by wave; after wave w the CTA's four copy warps meet and one
        // thread releases the CTA's count in wp_ready[w].  Wave w >= 2 is
        // copied once this CTA's row gather has reached wave w-1, so that
        // the extra memory traffic spreads over the compute of the earlier
        // waves instead of piling onto wave 0's.  This wait only paces the
        // copy: on expiry the copy goes ahead and nothing is reported, since
        // the results do not depend on it.
        const int cw = warp - 12;
        for (int w = 1; w < p.wp_g.W; ++w) {
            if (w >= 2 && *gather_wave < w - 1) {
                const uint64_t t0 = globaltimer_ns();
                while (*gather_wave < w - 1 && !*abort_flag && globaltimer_ns() - t0 < kWaitTimeoutNs)
                    __nanosleep(500);
            }
            pack_tokens(p, false, w, cw, 4, lane);
            named_bar_sync(1, 128);
            if (cw == 0 && lane == 0) {
                __threadfence();
                atomicAdd(p.wp_ready + w, 1);
            }
        }
    } else if (AMODE != A_GATHER && warp >= 8 && p.wp_a.pool) {
        // ------------------------------------------------------------ the pack
        // The dispatch's final decisions and every copy, overlapped with this
        // product (the shared experts' gate/up, which does not depend on the
        // routing); nothing in this launch reads what they write, the next
        // launch on the stream does.
        pack_tokens(p, true, -1, warp - 8, 4, lane, tiles_pace, abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // neither CTA of a pair leaves while the other may still arrive on its
    // barriers or the pair's MMAs may touch its memory
    if constexpr (CG2) cluster_sync();
    if (warp == 2) {
        if constexpr (CG2)
            tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ==================================================================== host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// bf16 tensor map, 128-byte swizzle, box {64, box_rows[, 1]}; out-of-range
// elements read as zero.  dims/strides in elements (innermost first).
static int make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_el, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return MOE_ECUDA;
    cuuint64_t gdim[3], gstr[2];
    cuuint32_t box[3], est[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) gdim[i] = dims[i];
    for (int i = 0; i + 1 < rank; ++i) gstr[i] = strides_el[i] * 2;
    box[0] = BK;
    box[1] = box_rows;
    box[2] = 1;
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gdim, gstr,
                     box, est, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ECUDA;
}

static int map2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld,
                 uint32_t box_rows) {
    const uint64_t dims[2] = {cols, rows};
    const uint64_t str[1] = {ld};
    return make_map(m, base, 2, dims, str, box_rows);
}

static int map3d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t groups,
                 uint64_t ld, uint64_t gstride, uint32_t box_rows) {
    const uint64_t dims[3] = {cols, rows, groups};
    const uint64_t str[2] = {ld, gstride};
    return make_map(m, base, 3, dims, str, box_rows);
}

template <int BN, int AMODE, int EPI, int MAJ = 0, bool CG2 = false>
static int launch_inst(const KParams& p, int grid, cudaStream_t st) {
    using C = TileCfg<BN, AMODE, EPI, CG2>;
    auto kern = gemm_tc_kernel<BN, AMODE, EPI, MAJ, CG2>;
    if (ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES) != MOE_OK)
        return MOE_ECUDA;
    if (CG2) {   // clusters of two CTAs (grid is even)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid, 1, 1);
        cfg.blockDim = dim3(p.wp_a.pool ? 384 : 256, 1, 1);   // + 4 copy warps
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return MOE_ECUDA;
    } else if (AMODE == A_GATHER && p.wp_ready) {
        // the copy warps' counters are waited on by every CTA: all resident
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid, 1, 1);
        cfg.blockDim = dim3(512, 1, 1);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return MOE_ECUDA;
    } else {
        // gathered A: warps 8-11 gather (12-15 copy only in the wave pipeline,
        // launched cooperatively above); dense products carrying the pack: 8-11
        const int threads = (AMODE == A_GATHER || p.wp_a.pool) ? 384 : 256;
        kern<<<grid, threads, C::SMEM_BYTES, st>>>(p);
    }
    return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

template <int BN, int AMODE, int EPI, int MAJ = 0, bool CG2 = false>
static int launch_traced(const KParams& p, int grid, cudaStream_t st, const char* name) {
    const int rc = launch_inst<BN, AMODE, EPI, MAJ, CG2>(p, grid, st);
    if (rc == MOE_OK) trace_after(st, name ? name : "gemm");
    return rc;
}

int check_status_gemm() { return moe_check_read_reset(); }

// fp32 output map, box 32 x 32 with the 128-byte swizzle (rank 2: [rows, cols]
// with row pitch ld; rank 3: groups of rows, gstride apart).
static int map_f32(CUtensorMap* m, const void* base, int rank, uint64_t cols, uint64_t rows,
                   uint64_t groups, uint64_t ld, uint64_t gstride) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return MOE_ECUDA;
    cuuint64_t gdim[3] = {cols, rows, groups};
    cuuint64_t gstr[2] = {ld * 4, gstride * 4};
    cuuint32_t box[3] = {32, 32, 1}, est[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<void*>(base), gdim, gstr,
                     box, est, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ECUDA;
}

int gemm_launch(const GemmDesc& d, cudaStream_t st) {
    int dev, sms;
    int rc = current_device(&dev, &sms);
    if (rc) return rc;
    if (d.nseg < 1 || d.nseg > 4 || (d.bn != 128 && d.bn != 256 && d.bn != 384))
        return MOE_EINVAL;
    if (d.bn == 384 && (d.epi != EPI_F32 || d.a_mode != A_DENSE)) return MOE_EINVAL;

    KParams p;
    std::memset(&p, 0, sizeof(p));
    // CTA pairs (cta_group::2, 256-row tiles) for the dense K-major products
    // with the bf16, SwiGLU and split epilogues
    const bool cg2 = d.a_mode == A_DENSE && d.bn == 256 && sms >= 2 &&
                     (d.epi == EPI_BF16 || d.epi == EPI_F32 || (d.epi == EPI_SPLIT && !d.b_mn) ||
                      ((d.epi == EPI_SWIGLU || d.epi == EPI_SWIGLU_BWD) && !d.b_mn));
    // gate/up pairs load two 128-row halves, the 384-wide router tile three
    // 128-row thirds; everything else one box of bn rows (K-major B); a CTA
    // of a pair loads one 128-row half of the B tile
    const bool pair = d.epi == EPI_SWIGLU || d.epi == EPI_SWIGLU_BWD;
    const uint32_t b_box = (cg2 || pair || d.bn == 384) ? 128 : d.bn;
    {   // every stage must receive exactly the bytes its barrier expects
        const uint32_t loads = cg2 ? (d.b_mn ? 2 : 1)
                               : d.b_mn ? d.bn / 64 : pair ? 2 : d.bn == 384 ? 3 : 1;
        const uint32_t box_rows = d.b_mn ? 64 : b_box;
        const uint32_t rows = cg2 ? d.bn / 2 : d.bn;
        if (loads * box_rows * BK * 2 != rows * BK * 2) return MOE_EINVAL;
    }
    p.nseg = d.nseg;
    p.seg_kb[0] = 0;
    for (int s = 0; s < d.nseg; ++s) {
        const GemmSeg& g = d.seg[s];
        // the row gather copies 16-byte chunks of K; TMA tiles take any K
        if (g.K <= 0 || (d.a_mode == A_GATHER && g.K % 8)) return MOE_EINVAL;
        p.seg_kb[s + 1] = p.seg_kb[s] + (g.K + BK - 1) / BK;
        // A: [M, K] K-major or [K, M] MN-major; grouped: one such matrix per group
        if (d.a_mode == A_DENSE)
            rc = d.a_mn ? map2d(&p.mapA[s], g.A, d.M, g.K, g.lda, 64)
                        : map2d(&p.mapA[s], g.A, g.K, d.M, g.lda, BM);
        else if (d.a_mode == A_GROUPED && d.kgoff)   // flat [k_rows, M] operand
            rc = d.a_mn ? map2d(&p.mapA[s], g.A, d.M, d.k_rows, g.lda, 64) : MOE_EINVAL;
        else if (d.a_mode == A_GROUPED && d.goff)
            rc = d.a_mn ? MOE_EINVAL : map2d(&p.mapA[s], g.A, g.K, d.rows_per_group, g.lda, BM);
        else if (d.a_mode == A_GROUPED)
            rc = d.a_mn ? map3d(&p.mapA[s], g.A, d.M, g.K, d.groups, g.lda, d.a_gstride, 64)
                        : map3d(&p.mapA[s], g.A, g.K, d.rows_per_group, d.groups, g.lda,
                                d.a_gstride, BM);
        else
            rc = d.a_mn ? MOE_EINVAL : MOE_OK;   // gathered rows: no map
        if (rc) return rc;
        // B: [N, K] K-major or [K, N] MN-major; grouped modes: per group
        if (d.a_mode == A_DENSE)
            rc = d.b_mn ? map2d(&p.mapB[s], g.B, d.b_rows, g.K, g.ldb, 64)
                        : map2d(&p.mapB[s], g.B, g.K, d.b_rows, g.ldb, b_box);
        else if (d.kgoff)   // flat [k_rows, N] operand
            rc = d.b_mn ? map2d(&p.mapB[s], g.B, d.b_rows, d.k_rows, g.ldb, 64) : MOE_EINVAL;
        else
            rc = d.b_mn ? map3d(&p.mapB[s], g.B, d.b_rows, g.K, d.groups, g.ldb, d.b_gstride, 64)
                        : map3d(&p.mapB[s], g.B, g.K, d.b_rows, d.groups, g.ldb, d.b_gstride,
                                b_box);
        if (rc) return rc;
    }
    if (d.epi == EPI_SPLIT) {
        if (d.nseg != 1 || !d.B_up || d.a_mode != A_DENSE || d.N != d.nsplit * d.bn)
            return MOE_EINVAL;
        if ((rc = map2d(&p.mapBup, d.B_up, d.seg[0].K, d.b2_rows, d.seg[0].ldb, b_box))) return rc;
    }
    if (d.epi == EPI_SWIGLU || d.epi == EPI_SWIGLU_BWD) {
        if (d.nseg != 1 || !d.B_up) return MOE_EINVAL;
        if (d.epi == EPI_SWIGLU_BWD && (!d.aux || !d.out2)) return MOE_EINVAL;
        if (d.b_mn && d.a_mode == A_DENSE)
            rc = map2d(&p.mapBup, d.B_up, d.b_rows, d.seg[0].K, d.seg[0].ldb, 64);
        else if (d.b_mn)
            rc = map3d(&p.mapBup, d.B_up, d.b_rows, d.seg[0].K, d.groups, d.seg[0].ldb,
                       d.b_gstride, 64);
        else if (d.a_mode == A_DENSE)
            rc = map2d(&p.mapBup, d.B_up, d.seg[0].K, d.b_rows, d.seg[0].ldb, b_box);
        else
            rc = map3d(&p.mapBup, d.B_up, d.seg[0].K, d.b_rows, d.groups, d.seg[0].ldb,
                       d.b_gstride, b_box);
        if (rc) return rc;
    }
    p.M = d.M;
    p.N = d.N;
    p.K0 = d.seg[0].K;
    const int n_per_tile = (d.epi == EPI_SWIGLU || d.epi == EPI_SWIGLU_BWD) ? d.bn / 2 : d.bn;
    p.n_tiles_n = (d.N + n_per_tile - 1) / n_per_tile;
    if (d.epi == EPI_SPLIT) {
        p.nsplit = d.nsplit;
        p.N2 = d.N2;
        p.out2 = d.out2;
        p.ldo2 = d.ldo2;
        p.n_tiles_n = d.nsplit + (d.N2 + d.bn - 1) / d.bn;
    }
    const int bm_tile = cg2 ? 2 * BM : BM;
    p.m_tiles = static_cast<int>((d.M + bm_tile - 1) / bm_tile);
#ifndef MOE_RASTER_MB
#define MOE_RASTER_MB 48
#endif
    // dense products whose whole B does not fit comfortably in L2 walk the
    // tiles in bands of column blocks whose B spans about MOE_RASTER_MB
    if (d.a_mode == A_DENSE && MOE_RASTER_MB > 0 && p.n_tiles_n > 1) {
        long long ktot = 0;
        for (int s = 0; s < d.nseg; ++s) ktot += d.seg[s].K;
        const long long bblk = static_cast<long long>(d.bn) * ktot * 2;   // B bytes a column block
        long long gn = (static_cast<long long>(MOE_RASTER_MB) << 20) / (bblk > 0 ? bblk : 1);
        if (gn < 1) gn = 1;
        if (gn < p.n_tiles_n) {
            const long long nb_ = (p.n_tiles_n + gn - 1) / gn;   // bands, then even widths
            p.raster_gn = static_cast<int>((p.n_tiles_n + nb_ - 1) / nb_);
        }
    }
    p.tile_list = reinterpret_cast<const int2*>(d.tile_list);
    p.tile_count = d.tile_count;
    p.rowmap = d.rowmap;
    p.counts = d.counts;
    // fp32 tile stores by TMA for the dense products (measured: ~3 % faster on
    // the backward's dense weight gradients); the per-expert weight gradients
    // (short K, write-bound) stay on the warps' own stores, which measured
    // ~4 % faster there
    if (d.epi == EPI_F32 && d.a_mode == A_DENSE && d.ldo % 4 == 0 &&
        (reinterpret_cast<uintptr_t>(d.out) & 15) == 0) {
        if (map_f32(&p.omap, d.out, 2, d.N, d.M, 1, d.ldo, 0) == MOE_OK) p.omap_rank = 2;
    }
    p.goff = d.goff;
    p.rmoff = d.rmoff;
    p.kgoff = d.kgoff;
    if (d.kgoff && (!d.uniform_groups || !d.a_mn || !d.b_mn || d.nseg != 1 || d.epi != EPI_F32 ||
                    d.k_rows <= 0))
        return MOE_EINVAL;
    p.kcount = d.kcount;
    if (d.kcount && (!d.uniform_groups || d.kgoff || d.a_mode != A_GROUPED)) return MOE_EINVAL;
    p.rowmap_ld = d.rowmap_ld;
    p.gather_src = d.gather_src;
    p.gather_pitch = d.gather_pitch;
    p.gather_rows = d.gather_rows;
    p.out = d.out;
    p.ldo = d.ldo;
    p.out_gstride = d.out_gstride;
    p.bias = d.bias;
    p.status = d.status;
    p.aux = static_cast<const uint16_t*>(d.aux);
    p.uniform_groups = d.uniform_groups;
    if (d.epi == EPI_SWIGLU_BWD) p.out2 = d.out2;
    if (d.wp_a.pool) {   // the dispatch's pack rides along (waves pipeline or dense overlap)
        const DispatchGeom& g = d.wp_g;
        // the dropless layout rides along only with the dense overlap, with
        // its block and expert offsets
        if (g.ragged && (d.wp_ready || !d.wp_a.blk_off || !d.wp_a.eoff)) return MOE_EINVAL;
        if (!d.wp_a.z || !d.wp_a.idx || !d.wp_a.send_row || g.k < 1 || g.k > 32 ||
            g.W < 1 || g.W > 32 || g.E_w < 1 || g.E_l != g.E_w * g.W || g.E % g.E_l || g.L < 8 ||
            g.L % 8 || (reinterpret_cast<uintptr_t>(d.wp_a.z) & 15) ||
            (reinterpret_cast<uintptr_t>(d.wp_a.pool) & 15))
            return MOE_EINVAL;
        if (d.wp_ready && (d.a_mode != A_GATHER || d.nseg != 1 || d.wp_a.pool != d.gather_src ||
                           g.L != d.seg[0].K || pool_pitch(g.L) != d.gather_pitch))
            return MOE_EINVAL;
        if (!d.wp_ready && (d.a_mode == A_GATHER || !d.wp_a.rloc || !d.wp_a.base_se ||
                            !d.wp_a.slot_of || !d.wp_a.drop || !d.wp_a.expert_rows))
            return MOE_EINVAL;
        p.wp_ready = d.wp_ready;
        p.wp_g = g;
        p.wp_a = d.wp_a;
    } else if (d.wp_ready) {
        return MOE_EINVAL;
    }

    int tiles = (d.a_mode == A_DENSE) ? p.m_tiles * p.n_tiles_n
                : d.uniform_groups     ? d.uniform_groups * p.m_tiles * p.n_tiles_n
                                       : d.max_tiles * p.n_tiles_n;
    if (tiles <= 0) return MOE_OK;
    int grid = tiles < sms ? tiles : sms;
    if (cg2) grid = 2 * (tiles < sms / 2 ? tiles : sms / 2);
    if (p.wp_ready) grid = sms;   // every SM copies its share of the later waves

    if ((d.a_mn || d.b_mn) && (d.bn != 256 || d.epi == EPI_SPLIT)) return MOE_EINVAL;
    const int maj = (d.a_mn ? 1 : 0) | (d.b_mn ? 2 : 0);
    const int key = ((d.bn * 10 + d.a_mode) * 10 + d.epi) * 10 + maj;
#define MOE_K(BN_, AM_, EP_, MJ_) ((((BN_) * 10 + (AM_)) * 10 + (EP_)) * 10 + (MJ_))
    switch (key) {
        case MOE_K(128, A_DENSE, EPI_F32, 0): return launch_traced<128, A_DENSE, EPI_F32>(p, grid, st, d.name);
        case MOE_K(384, A_DENSE, EPI_F32, 0): return launch_traced<384, A_DENSE, EPI_F32>(p, grid, st, d.name);
        case MOE_K(256, A_DENSE, EPI_SPLIT, 0):
            return cg2 ? launch_traced<256, A_DENSE, EPI_SPLIT, 0, true>(p, grid, st, d.name)
                       : launch_traced<256, A_DENSE, EPI_SPLIT>(p, grid, st, d.name);
        case MOE_K(256, A_DENSE, EPI_BF16, 0):
            return cg2 ? launch_traced<256, A_DENSE, EPI_BF16, 0, true>(p, grid, st, d.name)
                       : launch_traced<256, A_DENSE, EPI_BF16>(p, grid, st, d.name);
        case MOE_K(256, A_DENSE, EPI_SWIGLU, 0):
            return cg2 ? launch_traced<256, A_DENSE, EPI_SWIGLU, 0, true>(p, grid, st, d.name)
                       : launch_traced<256, A_DENSE, EPI_SWIGLU>(p, grid, st, d.name);
        case MOE_K(256, A_GATHER, EPI_SWIGLU, 0): return launch_traced<256, A_GATHER, EPI_SWIGLU>(p, grid, st, d.name);
        case MOE_K(256, A_GROUPED, EPI_SCATTER, 0): return launch_traced<256, A_GROUPED, EPI_SCATTER>(p, grid, st, d.name);
        // MN-major operands (general products, the backward pass)
#define MOE_PAIRED(EP_, MJ_)                                                                  \
    case MOE_K(256, A_DENSE, EP_, MJ_):                                                       \
        return cg2 ? launch_traced<256, A_DENSE, EP_, MJ_, true>(p, grid, st, d.name)         \
                   : launch_traced<256, A_DENSE, EP_, MJ_>(p, grid, st, d.name);
        MOE_PAIRED(EPI_BF16, 1)
        MOE_PAIRED(EPI_BF16, 2)
        MOE_PAIRED(EPI_BF16, 3)
        MOE_PAIRED(EPI_F32, 0)
        MOE_PAIRED(EPI_F32, 1)
        MOE_PAIRED(EPI_F32, 2)
        MOE_PAIRED(EPI_F32, 3)
        MOE_PAIRED(EPI_SWIGLU_BWD, 0)
#undef MOE_PAIRED
        // backward pass
        case MOE_K(256, A_GATHER, EPI_SWIGLU_BWD, 0): return launch_traced<256, A_GATHER, EPI_SWIGLU_BWD, 0>(p, grid, st, d.name);
        case MOE_K(256, A_GROUPED, EPI_BF16, 2): return launch_traced<256, A_GROUPED, EPI_BF16, 2>(p, grid, st, d.name);
        case MOE_K(256, A_GROUPED, EPI_SCATTER, 2): return launch_traced<256, A_GROUPED, EPI_SCATTER, 2>(p, grid, st, d.name);
        case MOE_K(256, A_GROUPED, EPI_F32, 3): return launch_traced<256, A_GROUPED, EPI_F32, 3>(p, grid, st, d.name);
#undef MOE_K
        default: return MOE_EINVAL;
    }
}

}  // namespace moe
