// pack.cuh -- one token's share of the dispatch (final decisions and the
// pool fill), shared by the pack kernel and the GEMM launches that carry the
// pool fill.
#pragma once
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace moe {

// Token t by one warp (lane j holds assignment (t, j)).  decide: make the
// receiver decisions -- expert row list entry, slot_of, drop code (0 kept,
// 1 dropped by the sender, 2 by the receiver).  copy_wave: copy the latent
// row and write the tag into the pool rows of every sender-kept assignment
// (-1), of those of one wave (>= 0), or of none (< -1); with a bank and
// decide, each receiver-kept row copied is also written to the bank at its
// position in its expert's row list (e * c_recv + r capped, offset[e] + r
// ragged).  The latent row is read once, CH 16-byte
// chunks a lane at a time, and written to each row.
// STREAM: streaming (evict-first) loads and stores, for a copy that runs
// beside a product whose tiles should stay in L2.
template <int CH, bool STREAM>
__device__ __forceinline__ void pack_token(const DispatchGeom& g, const PackArgs& P, int64_t t,
                                           int lane, bool decide, int copy_wave) {
    const int64_t s = t / g.T_s;
    const int64_t pitch = pool_pitch(g.L);
    int64_t row = -1;
    int64_t brow = -1;   // bank row of a receiver-kept row: its expert row list position
    int e = 0;
    if (lane < g.k) {
        const int64_t a = t * g.k + lane;
        e = P.idx[a];
        row = P.send_row[a];
        if (g.ragged && row >= 0) row = P.blk_off[row >> 32] + (row & 0xffffffffll);
        if (row >= 0 && !moe_check(row < g.pool_rows, 1001)) row = -1;
        if (decide) {
            int32_t so = -1;
            uint8_t dr = 1;
            if (row >= 0 && e >= 0 && e < g.E) {
                const int r = P.base_se[s * g.E + e] + P.rloc[a];
                if (r < g.c_recv) {
                    const int64_t at = g.ragged ? static_cast<int64_t>(P.eoff[e]) + r
                                                : static_cast<int64_t>(e) * g.c_recv + r;
                    if (moe_check(at >= 0 && at < (g.ragged ? g.T * g.k
                                                            : static_cast<int64_t>(g.E) * g.c_recv),
                                  1002)) {
                        P.expert_rows[at] = static_cast<int32_t>(row);
                        if (P.bank) brow = at;
                    }
                    so = static_cast<int32_t>(row);
                    dr = 0;
                } else {
                    dr = 2;
                }
            }
            P.slot_of[a] = so;
            P.drop[a] = dr;
        }
        if (copy_wave < -1 ||
            (copy_wave >= 0 && row >= 0 && !(e >= 0 && e < g.E && (e % g.E_l) / g.E_w == copy_wave)))
            row = brow = -1;
    }
    if (!__any_sync(0xffffffffu, row >= 0)) return;
    const int nchunk = g.L / 8;
    const uint4* src = reinterpret_cast<const uint4*>(P.z + t * g.L);
    for (int cb = 0; cb < nchunk; cb += 32 * CH) {
        uint4 v[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const int ch = cb + lane + 32 * c;
            if (ch < nchunk) v[c] = STREAM ? __ldcs(src + ch) : __ldg(src + ch);
        }
        for (int j = 0; j < g.k; ++j) {
            const int64_t rj = __shfl_sync(0xffffffffu, row, j);
            if (rj < 0) continue;
            uint4* dst = reinterpret_cast<uint4*>(P.pool + rj * pitch);
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int ch = cb + lane + 32 * c;
                if (ch < nchunk) {
                    if (STREAM)
                        __stcs(dst + ch, v[c]);
                    else
                        dst[ch] = v[c];
                }
            }
            const int64_t bj = __shfl_sync(0xffffffffu, brow, j);
            if (bj < 0) continue;
            uint4* bdst = reinterpret_cast<uint4*>(P.bank + bj * g.L);
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int ch = cb + lane + 32 * c;
                if (ch < nchunk) {
                    if (STREAM)
                        __stcs(bdst + ch, v[c]);
                    else
                        bdst[ch] = v[c];
                }
            }
        }
    }
    if (lane < g.k && row >= 0)
        *reinterpret_cast<int4*>(P.pool + row * pitch + g.L) =
            make_int4(e, static_cast<int>(t), lane, 0);
}

}  // namespace moe
