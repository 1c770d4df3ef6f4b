// backward.cu -- gradients of the layer (the pages report a training-step
// throughput; this is the derivative of the forward, step by step in reverse):
//   out = c W_lu^T + sum_s a_s Wsd_s^T   -> dc, da, dW_lu, dWsd
//   a = silu(x Wsg^T) (x Wsu^T)          -> dgs, dus (g/u recomputed), dWsg, dWsu
//   c_t = sum_kept w_tj Y_row            -> dY_row = w dc_t, dw_tj = <dc_t, Y_row>
//   per expert: Y = h Wd^T, h = silu(g) u, g/u = X Wg^T / X Wu^T
//                                        -> dh, dg, du, dX, dWd, dWg, dWu
//   X_row = z_t                          -> dz_t = sum_kept dX_row (the return of the
//                                           exchange, in reverse)
//   z = x W_ld^T                         -> dW_ld
//   w = softmax(selected logits)         -> dlogits, dWr
//   x                                    -> dx
// Every product runs on the tcgen05 GEMM engine; products over the token or
// row axis read their operands MN-major.
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace moe {

// dY = bf16(w_tj dc_t) for kept (t, j), written to the assignment's row in
// the per-expert layout (rowinv of its pool slot); dw_tj = <dc_t, Y[slot]>
// (fp32).  One warp per token, each lane's 16-byte chunks ch = lane + 32 i
// taken in passes of CH, both rows' chunks of a pass loaded before any is
// used.  The grid holds only the blocks resident at once; each warp strides
// over the tokens.
template <int CH>
__global__ void __launch_bounds__(256) combine_bwd_kernel(const uint16_t* __restrict__ dc,
                                                          const uint16_t* __restrict__ ypool,
                                                          const int32_t* __restrict__ slot_of,
                                                          const int32_t* __restrict__ rowinv,
                                                          const float* __restrict__ w, int64_t T,
                                                          int k, int L, uint16_t* __restrict__ dy,
                                                          float* __restrict__ dw, int64_t rows,
                                                          int64_t dst_rows) {
    const int lane = threadIdx.x & 31;
    const int nchunk = L / 8;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         t < T; t += nwarps) {
        int32_t my_row = -1, my_dst = 0;
        float my_w = 0.0f;
        if (lane < k) {
            my_row = slot_of[t * k + lane];
            my_w = w[t * k + lane];
            if (my_row >= 0 && !moe_check(my_row < rows, 1007)) my_row = -1;
            if (my_row >= 0) my_dst = rowinv[my_row];
            if (my_row >= 0 && !moe_check(my_dst >= 0 && my_dst < dst_rows, 1008)) my_row = -1;
        }
        const uint4* crow = reinterpret_cast<const uint4*>(dc + t * L);
        float dot_mine = 0.0f;   // lane j keeps dw for assignment j
        for (int j = 0; j < k; ++j) {
            const int32_t r = __shfl_sync(0xffffffffu, my_row, j);
            const int32_t rd = __shfl_sync(0xffffffffu, my_dst, j);
            const float wj = __shfl_sync(0xffffffffu, my_w, j);
            float dot = 0.0f;
            if (r >= 0) {
                const uint4* yrow =
                    reinterpret_cast<const uint4*>(ypool + static_cast<int64_t>(r) * L);
                uint4* drow = reinterpret_cast<uint4*>(dy + static_cast<int64_t>(rd) * L);
                for (int cb = 0; cb < nchunk; cb += 32 * CH) {
                    uint4 cv[CH], yv[CH];
#pragma unroll
                    for (int q = 0; q < CH; ++q) {
                        const int ch = cb + lane + 32 * q;
                        if (ch < nchunk) {
                            cv[q] = __ldg(crow + ch);
                            yv[q] = __ldg(yrow + ch);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < CH; ++q) {
                        const int ch = cb + lane + 32 * q;
                        if (ch < nchunk) {
                            const uint32_t cu[4] = {cv[q].x, cv[q].y, cv[q].z, cv[q].w};
                            const uint32_t yu[4] = {yv[q].x, yv[q].y, yv[q].z, yv[q].w};
                            uint32_t o[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const float c0 = bf16_lo(cu[h]), c1 = bf16_hi(cu[h]);
                                dot = fmaf(c0, bf16_lo(yu[h]), dot);
                                dot = fmaf(c1, bf16_hi(yu[h]), dot);
                                o[h] = pack_bf16x2(wj * c0, wj * c1);
                            }
                            drow[ch] = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                }
            }
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            if (lane == j) dot_mine = r >= 0 ? dot : 0.0f;
        }
        if (lane < k) dw[t * k + lane] = dot_mine;
    }
}

// dlogits[t, e] = bf16(w_j (dw_j - sum_i w_i dw_i)) for e = idx[t, j], else 0.
__global__ void __launch_bounds__(256) router_bwd_kernel(const int32_t* __restrict__ idx,
                                                         const float* __restrict__ w,
                                                         const float* __restrict__ dw, int64_t T,
                                                         int k, int E,
                                                         uint16_t* __restrict__ dlogits) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_e = -1;
    float my_w = 0.0f, my_dw = 0.0f;
    if (lane < k) {
        my_e = idx[t * k + lane];
        my_w = w[t * k + lane];
        my_dw = dw[t * k + lane];
    }
    float s = my_w * my_dw;
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const float my_dl = my_w * (my_dw - s);
    uint16_t* row = dlogits + t * E;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        float v = 0.0f;
        for (int j = 0; j < k; ++j) {
            const int ej = __shfl_sync(0xffffffffu, my_e, j);
            const float dj = __shfl_sync(0xffffffffu, my_dl, j);
            if (ej == e) v = dj;
        }
        if (e < E) {
            const __nv_bfloat16 b = __float2bfloat16_rn(v);
            row[e] = *reinterpret_cast<const uint16_t*>(&b);
        }
    }
}

// rowinv[rows[e][r]] = e * c_recv + r for r < count[e]: where each kept pool
// row sits in the per-expert layout.
__global__ void __launch_bounds__(256) row_inverse_kernel(const int32_t* __restrict__ rows,
                                                          const int32_t* __restrict__ count, int E,
                                                          int c_recv, int32_t* __restrict__ rowinv) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(E) * c_recv) return;
    const int e = static_cast<int>(i / c_recv);
    const int r = static_cast<int>(i - static_cast<int64_t>(e) * c_recv);
    if (r < count[e]) rowinv[rows[i]] = static_cast<int32_t>(i);
}

// dst[e][r][0:L] = src[rows[e][r]][0:L] for r < count[e], zeros up to c_recv.
__global__ void __launch_bounds__(256) gather_expert_rows_kernel(
    const uint16_t* __restrict__ src, int64_t pitch, const int32_t* __restrict__ rows,
    const int32_t* __restrict__ count, int E, int c_recv, int L, uint16_t* __restrict__ dst) {
    const int lane = threadIdx.x & 31;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (wid >= static_cast<int64_t>(E) * c_recv) return;
    const int e = static_cast<int>(wid / c_recv);
    const int r = static_cast<int>(wid - static_cast<int64_t>(e) * c_recv);
    uint4* d = reinterpret_cast<uint4*>(dst + wid * L);
    const int nchunk = L / 8;
    if (r < count[e]) {
        const uint4* sp = reinterpret_cast<const uint4*>(
            src + static_cast<int64_t>(rows[static_cast<int64_t>(e) * c_recv + r]) * pitch);
        for (int ch = lane; ch < nchunk; ch += 32) d[ch] = __ldg(sp + ch);
    } else {
        for (int ch = lane; ch < nchunk; ch += 32) d[ch] = make_uint4(0, 0, 0, 0);
    }
}

// Rows r >= count[e] of a [E, c_recv, W] buffer set to zero.
__global__ void __launch_bounds__(256) zero_pad_rows_kernel(uint16_t* __restrict__ buf,
                                                            const int32_t* __restrict__ count,
                                                            int E, int c_recv, int W) {
    const int lane = threadIdx.x & 31;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (wid >= static_cast<int64_t>(E) * c_recv) return;
    const int e = static_cast<int>(wid / c_recv);
    const int r = static_cast<int>(wid - static_cast<int64_t>(e) * c_recv);
    if (r < count[e]) return;
    uint4* d = reinterpret_cast<uint4*>(buf + wid * W);
    for (int ch = lane; ch < W / 8; ch += 32) d[ch] = make_uint4(0, 0, 0, 0);
}

// ---- dropless (ragged) layout: expert e's rows padded to a multiple of 64 at
// poff[e], so that the weight gradients contract over whole 64-row blocks of
// zero-padded operands.

// poff[e] = sum over e' < e of count[e'] rounded up to 64; poff[E] = total.
// One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) padded_offsets_kernel(const int32_t* __restrict__ count,
                                                              int E, int32_t* __restrict__ poff) {
    __shared__ int warp_sum[32];
    __shared__ int carry;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const int v = e < E ? (count[e] + 63) & ~63 : 0;
        int incl = v;
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_sum[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            int ws = warp_sum[lane];
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, ws, off);
                if (lane >= off) ws += y;
            }
            warp_sum[lane] = ws;
        }
        __syncthreads();
        const int excl = carry + (wid ? warp_sum[wid - 1] : 0) + incl - v;
        if (e < E) poff[e] = excl;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = excl + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) poff[E] = carry;
}

// rowinv[rows[eoff[e] + r]] = poff[e] + r for r < count[e].  One CTA per expert.
__global__ void __launch_bounds__(256) row_inverse_ragged_kernel(
    const int32_t* __restrict__ rows, const int32_t* __restrict__ eoff,
    const int32_t* __restrict__ count, const int32_t* __restrict__ poff,
    int32_t* __restrict__ rowinv) {
    const int e = blockIdx.x;
    for (int r = threadIdx.x; r < count[e]; r += blockDim.x) rowinv[rows[eoff[e] + r]] = poff[e] + r;
}

// Rows poff[e] + count[e] .. poff[e+1] - 1 of a [*, W] buffer set to zero.
__global__ void __launch_bounds__(256) zero_pad_ragged_kernel(uint16_t* __restrict__ buf,
                                                              const int32_t* __restrict__ count,
                                                              const int32_t* __restrict__ poff,
                                                              int W) {
    const int e = blockIdx.x;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int first = poff[e] + count[e];
    for (int r = first + wid; r < poff[e + 1]; r += blockDim.x >> 5) {
        uint4* d = reinterpret_cast<uint4*>(buf + static_cast<int64_t>(r) * W);
        for (int ch = lane; ch < W / 8; ch += 32) d[ch] = make_uint4(0, 0, 0, 0);
    }
}

// dst[poff[e] + r][0:W] = src[row r of expert e][0:W] for r < count[e], zeros
// up to poff[e+1]; the source row is rows[eoff[e] + r] (a row map) or, with
// rows null, eoff[e] + r.  One CTA per expert, a warp per row.
__global__ void __launch_bounds__(256) gather_ragged_kernel(
    const uint16_t* __restrict__ src, int64_t pitch, const int32_t* __restrict__ rows,
    const int32_t* __restrict__ eoff, const int32_t* __restrict__ count,
    const int32_t* __restrict__ poff, int W, uint16_t* __restrict__ dst) {
    const int e = blockIdx.x;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int cnt = count[e], p0 = poff[e], n = poff[e + 1] - p0;
    for (int r = wid; r < n; r += blockDim.x >> 5) {
        uint4* d = reinterpret_cast<uint4*>(dst + static_cast<int64_t>(p0 + r) * W);
        if (r < cnt) {
            const int64_t sr = rows ? rows[eoff[e] + r] : static_cast<int64_t>(eoff[e]) + r;
            const uint4* sp = reinterpret_cast<const uint4*>(src + sr * pitch);
            for (int ch = lane; ch < W / 8; ch += 32) d[ch] = __ldg(sp + ch);
        } else {
            for (int ch = lane; ch < W / 8; ch += 32) d[ch] = make_uint4(0, 0, 0, 0);
        }
    }
}

static size_t al(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

int check_status_backward() { return moe_check_read_reset(); }

// Rows of the per-expert layout: [E, c_recv] (capped) or the padded ragged
// bound T*k + 64 E.
static int64_t expert_layout_rows(const DispatchGeom& g) {
    return g.ragged ? g.T * g.k + 64ll * g.E : static_cast<int64_t>(g.E) * g.c_recv;
}

BackwardWs backward_ws_layout(const DispatchGeom& g, int d, int H, int Hs, int ns) {
    BackwardWs w;
    std::memset(&w, 0, sizeof(w));
    size_t o = 0;
    const size_t T = static_cast<size_t>(g.T), L = g.L, E = g.E;
    const size_t P = static_cast<size_t>(g.pool_rows), HS = static_cast<size_t>(ns) * Hs;
    const size_t PE = static_cast<size_t>(expert_layout_rows(g));   // per-expert rows
    w.dc = o;       o = al(o + T * L * 2);
    w.da = o;       o = al(o + T * HS * 2);
    w.dgs = o;      o = al(o + T * HS * 2);
    w.dus = o;      o = al(o + T * HS * 2);
    w.dw = o;       o = al(o + T * g.k * 4);
    w.rowinv = o;   o = al(o + P * 4);
    w.dxpool = o;   o = al(o + P * L * 2);
    w.dh = o;       o = al(o + PE * H * 2);
    w.dg = o;       o = al(o + PE * H * 2);
    w.du = o;       o = al(o + PE * H * 2);
    w.xe = o;       o = al(o + PE * L * 2);
    w.dye = o;      o = al(o + PE * L * 2);
    w.dz = o;       o = al(o + T * L * 2);
    w.dlogits = o;  o = al(o + T * E * 2);
    const size_t max_mt = g.ragged ? P / 128 + E : E * ((static_cast<size_t>(g.c_recv) + 127) / 128);
    w.tiles = o;    o = al(o + max_mt * 8 + 16);
    if (g.ragged) {   // padded copy of h, padded row offsets
        w.hp = o;   o = al(o + PE * H * 2);
        w.poff = o; o = al(o + (E + 1) * 4);
    }
    w.total = o;
    (void)d;
    return w;
}

int launch_backward(const DispatchGeom& g, int d, int H, int Hs, int ns,
                    const moe_backward_args_t& a, cudaStream_t st) {
    const BackwardWs L_ = backward_ws_layout(g, d, H, Hs, ns);
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    auto bf = [&](size_t off) { return reinterpret_cast<uint16_t*>(ws + off); };
    uint16_t *dc = bf(L_.dc), *da = bf(L_.da), *dgs = bf(L_.dgs), *dus = bf(L_.dus);
    int32_t* rowinv = reinterpret_cast<int32_t*>(ws + L_.rowinv);
    uint16_t *dxp = bf(L_.dxpool), *dh = bf(L_.dh), *dg = bf(L_.dg),
             *du = bf(L_.du), *xe = bf(L_.xe), *dye = bf(L_.dye), *dz = bf(L_.dz),
             *dl = bf(L_.dlogits);
    float* dw = reinterpret_cast<float*>(ws + L_.dw);
    int32_t* tiles = reinterpret_cast<int32_t*>(ws + L_.tiles);
    const int64_t T = g.T;
    const int L = g.L, E = g.E, k = g.k, cr = g.ragged ? 0 : g.c_recv;
    // ragged layout: expert e's rows at a.expert_offsets[e] in the flat row map
    // and h; padded to 64-row blocks at poff[e] in the per-expert buffers
    const bool rag = g.ragged != 0;
    const int32_t* eoff = a.expert_offsets;
    int32_t* poff = rag ? reinterpret_cast<int32_t*>(ws + L_.poff) : nullptr;
    uint16_t* hp = rag ? bf(L_.hp) : nullptr;
    const int64_t PE = expert_layout_rows(g);
    const int HS = ns * Hs;
    int rc;
    auto mm = [&](GemmDesc& q, const char* name) {
        q.status = a.status;
        q.name = name;
        return gemm_launch(q, st);
    };
    GemmDesc q;
    // ---- output layer: dc = dout W_lu, da_s = dout Wsd_s
    std::memset(&q, 0, sizeof(q));
    q.a_mode = A_DENSE; q.epi = EPI_BF16; q.bn = 256; q.b_mn = 1;
    q.M = T; q.N = L; q.nseg = 1; q.seg[0] = GemmSeg{a.dout, d, a.W_lu, L, d}; q.b_rows = L;
    q.out = dc; q.ldo = L;
    if ((rc = mm(q, "bwd_gemm_dc"))) return rc;
    for (int s = 0; s < ns; ++s) {
        std::memset(&q, 0, sizeof(q));
        q.a_mode = A_DENSE; q.epi = EPI_BF16; q.bn = 256; q.b_mn = 1;
        q.M = T; q.N = Hs; q.nseg = 1;
        q.seg[0] = GemmSeg{a.dout, d, a.Wsd + static_cast<size_t>(s) * d * Hs, Hs, d};
        q.b_rows = Hs; q.out = da + static_cast<size_t>(s) * Hs; q.ldo = HS;
        if ((rc = mm(q, "bwd_gemm_da"))) return rc;
    }
    // ---- weight gradients of the output layer (products over tokens)
    std::memset(&q, 0, sizeof(q));
    q.a_mode = A_DENSE; q.epi = EPI_F32; q.bn = 256; q.a_mn = 1; q.b_mn = 1;
    q.M = d; q.N = L; q.nseg = 1; q.seg[0] = GemmSeg{a.dout, d, a.c, L, static_cast<int>(T)};
    q.b_rows = L; q.out = a.dW_lu; q.ldo = L;
    if ((rc = mm(q, "bwd_gemm_dW_lu"))) return rc;
    for (int s = 0; s < ns; ++s) {
        std::memset(&q, 0, sizeof(q));
        q.a_mode = A_DENSE; q.epi = EPI_F32; q.bn = 256; q.a_mn = 1; q.b_mn = 1;
        q.M = d; q.N = Hs; q.nseg = 1;
        q.seg[0] = GemmSeg{a.dout, d, a.a + static_cast<size_t>(s) * Hs, HS, static_cast<int>(T)};
        q.b_rows = Hs; q.out = a.dWsd + static_cast<size_t>(s) * d * Hs; q.ldo = Hs;
        if ((rc = mm(q, "bwd_gemm_dWsd"))) return rc;
    }
    // ---- shared experts: recompute g/u, SwiGLU backward, weight gradients
    if (ns > 0) {
        std::memset(&q, 0, sizeof(q));
        q.a_mode = A_DENSE; q.epi = EPI_SWIGLU_BWD; q.bn = 256;
        q.M = T; q.N = HS; q.nseg = 1; q.seg[0] = GemmSeg{a.x, d, a.Wsg, d, d};
        q.B_up = a.Wsu; q.b_rows = HS; q.aux = da; q.out = dgs; q.out2 = dus; q.ldo = HS;
        if ((rc = mm(q, "bwd_gemm_shared_swiglu"))) return rc;
        for (int which = 0; which < 2; ++which) {
            std::memset(&q, 0, sizeof(q));
            q.a_mode = A_DENSE; q.epi = EPI_F32; q.bn = 256; q.a_mn = 1; q.b_mn = 1;
            q.M = HS; q.N = d; q.nseg = 1;
            q.seg[0] = GemmSeg{which ? dus : dgs, HS, a.x, d, static_cast<int>(T)};
            q.b_rows = d; q.out = which ? a.dWsu : a.dWsg; q.ldo = d;
            if ((rc = mm(q, "bwd_gemm_dWshared"))) return rc;
        }
    }
    // ---- combine backward (the return path in reverse): dY straight into the
    // per-expert layout, whose rows past each expert's count are zero
    {
        if (rag) {
            padded_offsets_kernel<<<1, 1024, 0, st>>>(a.expert_count, E, poff);
            row_inverse_ragged_kernel<<<E, 256, 0, st>>>(a.expert_rows, eoff, a.expert_count, poff,
                                                         rowinv);
            zero_pad_ragged_kernel<<<E, 256, 0, st>>>(dye, a.expert_count, poff, L);
        } else {
            const int64_t nw = static_cast<int64_t>(E) * cr;
            const unsigned g_inv = static_cast<unsigned>((nw + 255) / 256);
            const unsigned g_pad = static_cast<unsigned>((nw + 7) / 8);
            row_inverse_kernel<<<g_inv, 256, 0, st>>>(a.expert_rows, a.expert_count, E, cr, rowinv);
            zero_pad_rows_kernel<<<g_pad, 256, 0, st>>>(dye, a.expert_count, E, cr, L);
        }
        // resident blocks of each instance, queried once (no runtime call
        // inside a stream capture after the first launch)
        static int per_sm[2] = {0, 0};
        const bool wide = L / 8 > 32 * 4;
        if (!per_sm[wide]) {
            int nb = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    &nb, wide ? combine_bwd_kernel<12> : combine_bwd_kernel<4>, 256, 0) !=
                cudaSuccess)
                return MOE_ECUDA;
            per_sm[wide] = nb > 0 ? nb : 1;
        }
        int dev, sms;
        if ((rc = current_device(&dev, &sms))) return rc;
        const int64_t need = (T + 7) / 8, most = static_cast<int64_t>(sms) * per_sm[wide];
        const unsigned grid = static_cast<unsigned>(need < most ? need : most);
        if (wide)
            combine_bwd_kernel<12><<<grid, 256, 0, st>>>(dc, a.ypool, a.slot_of, rowinv, a.w, T, k,
                                                          L, dye, dw, g.pool_rows, PE);
        else
            combine_bwd_kernel<4><<<grid, 256, 0, st>>>(dc, a.ypool, a.slot_of, rowinv, a.w, T, k,
                                                         L, dye, dw, g.pool_rows, PE);
        if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
        trace_after(st, "bwd_combine");
    }
    // ---- experts
    const int max_mt = rag ? static_cast<int>(g.pool_rows / 128 + E) : E * ((cr + 127) / 128);
    int32_t* tile_count = tiles + 2 * max_mt;
    if ((rc = launch_build_tiles(a.expert_count, E, 128, tiles, tile_count, st))) return rc;
    // Capped layout, widths in whole blocks: the three expert products on CTA
    // pairs over row groups, whose list sits at the start of dz (written only
    // by the return of dX below); each falls back to the grouped GEMM where
    // its path is not open.
    ExpertGroups gl{};
    bool groups = false;
    const size_t list_bytes = rag ? expert_pair_lists_bytes_ragged(E, g.pool_rows)
                                  : expert_pair_chunks_bytes(E, cr);
    if (static_cast<size_t>(T) * L * 2 >= list_bytes) {
        rc = rag ? expert_group_list_ragged(E, g.pool_rows, a.expert_count, dz, &gl, st)
                 : expert_group_list(E, cr, a.expert_count, dz, &gl, st);
        if (rc == MOE_OK)
            groups = true;
        else if (rc != MOE_EINVAL)
            return rc;
    }
    // dropless: the per-expert buffers' rows at the padded offsets poff
    const int32_t* roff = rag ? poff : nullptr;
    rc = groups ? expert_dh_group(E, cr, L, H, dye, a.Wd, gl, dh, a.status, st, roff, PE)
                : MOE_EINVAL;
    if (rc == MOE_EINVAL) {
        std::memset(&q, 0, sizeof(q));   // dh = dY_e Wd_e (per-expert rows by TMA)
        q.a_mode = A_GROUPED; q.epi = EPI_BF16; q.bn = 256; q.b_mn = 1;
        q.N = H; q.nseg = 1; q.seg[0] = GemmSeg{dye, L, a.Wd, H, L};
        q.groups = E; q.rows_per_group = rag ? static_cast<int>(PE) : cr;
        q.a_gstride = static_cast<int64_t>(cr) * L;
        q.b_rows = H; q.b_gstride = static_cast<int64_t>(L) * H;
        q.tile_list = tiles; q.tile_count = tile_count; q.max_tiles = max_mt;
        q.rowmap = a.expert_rows; q.counts = a.expert_count; q.rowmap_ld = cr;
        q.goff = poff;   // ragged: the padded per-expert rows (A and out)
        q.out = dh; q.ldo = H; q.out_gstride = static_cast<int64_t>(cr) * H;
        if ((rc = mm(q, "bwd_gemm_dh"))) return rc;
    } else if (rc) {
        return rc;
    }
    // Capped layout: X in per-expert contiguous rows with zero padding (which
    // the weight gradients contract over) and h's unwritten rows zeroed, made
    // first, so that the SwiGLU backward can read X as whole TMA tiles.  X
    // is the forward's bank when the caller passes it (its kept rows are the
    // pool rows' payloads; only its padding rows need zeroing), else a copy
    // gathered from the pool rows.
    bool grouped = false;
    if (!rag) {
        const int64_t nw = static_cast<int64_t>(E) * cr;
        const unsigned grid = static_cast<unsigned>((nw + 7) / 8);
        if (a.bank) {
            xe = a.bank;
            zero_pad_rows_kernel<<<grid, 256, 0, st>>>(xe, a.expert_count, E, cr, L);
        } else {
            gather_expert_rows_kernel<<<grid, 256, 0, st>>>(a.pool, pool_pitch(L), a.expert_rows,
                                                            a.expert_count, E, cr, L, xe);
        }
        zero_pad_rows_kernel<<<grid, 256, 0, st>>>(a.h, a.expert_count, E, cr, H);
        if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
        trace_after(st, "bwd_gather_rows");
        // recompute g/u and the SwiGLU backward over row groups
        rc = groups ? expert_swiglu_bwd_group(E, cr, L, H, xe, a.Wg, a.Wu, dh, gl, dg, du, a.status,
                                              st)
                    : MOE_EINVAL;
        if (rc == MOE_OK) {
            grouped = true;
            // rows past each expert's count: zeros, which the weight
            // gradients contract over
            zero_pad_rows_kernel<<<grid, 256, 0, st>>>(dg, a.expert_count, E, cr, H);
            zero_pad_rows_kernel<<<grid, 256, 0, st>>>(du, a.expert_count, E, cr, H);
            if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
            trace_after(st, "bwd_zero_pad");
        } else if (rc != MOE_EINVAL) {
            return rc;
        }
    } else {
        // dropless: padded per-expert copies of X and of h (zero padding),
        // then the SwiGLU backward over row groups from X
        gather_ragged_kernel<<<E, 256, 0, st>>>(a.pool, pool_pitch(L), a.expert_rows, eoff,
                                                a.expert_count, poff, L, xe);
        gather_ragged_kernel<<<E, 256, 0, st>>>(a.h, H, nullptr, eoff, a.expert_count, poff, H,
                                                hp);
        if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
        trace_after(st, "bwd_gather_rows");
        rc = groups ? expert_swiglu_bwd_group(E, cr, L, H, xe, a.Wg, a.Wu, dh, gl, dg, du,
                                              a.status, st, roff, PE)
                    : MOE_EINVAL;
        if (rc == MOE_OK) {
            grouped = true;
            zero_pad_ragged_kernel<<<E, 256, 0, st>>>(dg, a.expert_count, poff, H);
            zero_pad_ragged_kernel<<<E, 256, 0, st>>>(du, a.expert_count, poff, H);
            if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
            trace_after(st, "bwd_zero_pad");
        } else if (rc != MOE_EINVAL) {
            return rc;
        }
    }
    if (!grouped) {
        std::memset(&q, 0, sizeof(q));   // recompute g/u of the received rows, SwiGLU backward
        // (its epilogue also zeroes each expert's padding rows of dg and du)
        q.a_mode = A_GATHER; q.epi = EPI_SWIGLU_BWD; q.bn = 256;
        q.N = H; q.nseg = 1; q.seg[0] = GemmSeg{nullptr, 0, a.Wg, L, L};
        q.B_up = a.Wu; q.groups = E; q.rows_per_group = cr; q.b_rows = H;
        q.b_gstride = static_cast<int64_t>(H) * L;
        q.tile_list = tiles; q.tile_count = tile_count; q.max_tiles = max_mt;
        q.rowmap = a.expert_rows; q.counts = a.expert_count; q.rowmap_ld = cr;
        q.goff = poff; q.rmoff = eoff;   // ragged: outputs padded, rows from the flat map
        q.gather_src = a.pool; q.gather_pitch = pool_pitch(L); q.gather_rows = g.pool_rows;
        q.aux = dh; q.out = dg; q.out2 = du; q.ldo = H; q.out_gstride = static_cast<int64_t>(cr) * H;
        if ((rc = mm(q, "bwd_gemm_expert_swiglu"))) return rc;
    }
    rc = groups ? expert_dx_group(E, cr, L, H, dg, du, a.Wg, a.Wu, gl, a.expert_rows, dxp,
                                  g.pool_rows, a.status, st, roff, PE, rag ? eoff : nullptr)
                : MOE_EINVAL;
    if (rc == MOE_EINVAL) {
        std::memset(&q, 0, sizeof(q));   // dX = dg Wg_e + du Wu_e, back to the pool rows
        q.a_mode = A_GROUPED; q.epi = EPI_SCATTER; q.bn = 256; q.b_mn = 1;
        q.N = L; q.nseg = 2;
        q.seg[0] = GemmSeg{dg, H, a.Wg, L, H};
        q.seg[1] = GemmSeg{du, H, a.Wu, L, H};
        q.groups = E; q.rows_per_group = rag ? static_cast<int>(PE) : cr;
        q.a_gstride = static_cast<int64_t>(cr) * H;
        q.b_rows = L; q.b_gstride = static_cast<int64_t>(H) * L;
        q.tile_list = tiles; q.tile_count = tile_count; q.max_tiles = max_mt;
        q.rowmap = a.expert_rows; q.counts = a.expert_count; q.rowmap_ld = cr;
        q.goff = poff; q.rmoff = eoff;
        q.out = dxp; q.ldo = L; q.gather_rows = g.pool_rows;
        if ((rc = mm(q, "bwd_gemm_dX"))) return rc;
    } else if (rc) {
        return rc;
    }
    auto wgrad = [&](const uint16_t* A, int M, const uint16_t* B, int N, float* out, const char* nm) {
        std::memset(&q, 0, sizeof(q));   // out_e[M, N] = A_e^T B_e over the expert's rows
        q.a_mode = A_GROUPED; q.epi = EPI_F32; q.bn = 256; q.a_mn = 1; q.b_mn = 1;
        q.M = M; q.N = N; q.nseg = 1;
        q.seg[0] = GemmSeg{A, M, B, N, rag ? static_cast<int>(PE) : cr};
        q.groups = E; q.uniform_groups = E;
        q.a_gstride = static_cast<int64_t>(cr) * M; q.b_rows = N;
        q.b_gstride = static_cast<int64_t>(cr) * N;
        q.kgoff = poff; q.k_rows = PE;   // ragged: each expert's padded row range
        if (!rag) q.kcount = a.expert_count;   // capped: only the blocks holding its rows
        q.out = out; q.ldo = N; q.out_gstride = static_cast<int64_t>(M) * N;
        return mm(q, nm);
    };
    if ((rc = wgrad(dye, L, rag ? hp : a.h, H, a.dWd, "bwd_gemm_dWd"))) return rc;
    if ((rc = wgrad(dg, H, xe, L, a.dWg, "bwd_gemm_dWg"))) return rc;
    if ((rc = wgrad(du, H, xe, L, a.dWu, "bwd_gemm_dWu"))) return rc;
    // ---- return of the gradients to the tokens, latent projection
    if ((rc = launch_combine(dxp, a.slot_of, nullptr, T, k, L, dz, g.pool_rows, st))) return rc;
    std::memset(&q, 0, sizeof(q));
    q.a_mode = A_DENSE; q.epi = EPI_F32; q.bn = 256; q.a_mn = 1; q.b_mn = 1;
    q.M = L; q.N = d; q.nseg = 1; q.seg[0] = GemmSeg{dz, L, a.x, d, static_cast<int>(T)};
    q.b_rows = d; q.out = a.dW_ld; q.ldo = d;
    if ((rc = mm(q, "bwd_gemm_dW_ld"))) return rc;
    // ---- router
    {
        const unsigned grid = static_cast<unsigned>((T + 7) / 8);
        router_bwd_kernel<<<grid, 256, 0, st>>>(a.idx, a.w, dw, T, k, E, dl);
        if (cudaPeekAtLastError() != cudaSuccess) return MOE_ECUDA;
        trace_after(st, "bwd_router");
    }
    std::memset(&q, 0, sizeof(q));
    q.a_mode = A_DENSE; q.epi = EPI_F32; q.bn = 256; q.a_mn = 1; q.b_mn = 1;
    q.M = E; q.N = d; q.nseg = 1; q.seg[0] = GemmSeg{dl, E, a.x, d, static_cast<int>(T)};
    q.b_rows = d; q.out = a.dWr; q.ldo = d;
    if ((rc = mm(q, "bwd_gemm_dWr"))) return rc;
    // ---- dx = dz W_ld + dlogits Wr + dgs Wsg + dus Wsu (one product, four K segments)
    std::memset(&q, 0, sizeof(q));
    q.a_mode = A_DENSE; q.epi = EPI_BF16; q.bn = 256; q.b_mn = 1;
    q.M = T; q.N = d; q.nseg = ns > 0 ? 4 : 2;
    q.seg[0] = GemmSeg{dz, L, a.W_ld, d, L};
    q.seg[1] = GemmSeg{dl, E, a.Wr, d, E};
    if (ns > 0) {
        q.seg[2] = GemmSeg{dgs, HS, a.Wsg, d, HS};
        q.seg[3] = GemmSeg{dus, HS, a.Wsu, d, HS};
    }
    q.b_rows = d; q.out = a.dx; q.ldo = d;
    return mm(q, "bwd_gemm_dx");
}

}  // namespace moe
