/*
 * moe_pooled_wave.h -- C ABI of the GB300 (sm_103a) pooled-wave MoE layer.
 *
 * One MoE branch forward as the Marin 535B-A23B pages state it (lamjinlab,
 * "Marin 開始公開訓練 535B 參數 MoE 模型", section 二 "稀疏模型的組織方式", and
 * its Japanese edition, section 二): a router picks k of E routed experts per
 * token; a latent projection compresses the routed activations (6144 -> 3072)
 * before the exchange; each source keeps one fixed pool per destination rank,
 * sent in W same-shape waves with the expert id packed into the payload row;
 * a sender capacity factor bounds one source -> one destination, a receiver
 * capacity factor bounds the rows of one local expert, and any assignment
 * that overflows either buffer is dropped and counted; each destination runs
 * its local experts on what it received; the outputs return, are combined,
 * projected back to model width and added to the shared experts, which see
 * every token.
 *
 * On one GPU the S source ranks and D = S destination ranks are regions of
 * device memory: the pool is laid out destination-major, so the sender's pool
 * *is* the receiver's buffer and the exchange is the pack scatter (and the
 * return path the combine gather).
 *
 * Conventions for every entry point
 *  - All tensor arguments are DEVICE pointers owned by the caller, row-major,
 *    16-byte aligned, non-overlapping unless stated.  bf16 tensors are passed
 *    as uint16_t (IEEE bfloat16 bit patterns).  Weights are stored
 *    out-features-major ([out, in], as torch.nn.Linear does).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *    only enqueues work: it never synchronises the host and never allocates
 *    or frees memory.  Scratch space is caller-provided (sizes from moe_plan).
 *  - Return value: MOE_OK (0) or a negative MOE_E* code.  Host-side argument
 *    checks run before anything is enqueued; on error nothing is enqueued.
 *    With T = 0 (an empty batch) every call returns MOE_OK without touching
 *    its tensor pointers, which may then be NULL (moe_dispatch_pooled still
 *    writes expert_count and stats).
 *  - `status` is a caller-owned device int32.  A kernel whose bounded wait on
 *    an on-chip barrier runs out writes MOE_ETIMEOUT there (first error wins)
 *    and returns early; its outputs are then undefined.  The library never
 *    clears it: zero it once and read it when convenient.
 *  - Results are deterministic: identical inputs give identical bits,
 *    including pool slots and drop decisions.
 */
#ifndef MOE_POOLED_WAVE_H
#define MOE_POOLED_WAVE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK        0
#define MOE_EINVAL   -1   /* bad sizes, divisibility, alignment or null pointer      */
#define MOE_ENOSPC   -2   /* caller-provided scratch smaller than moe_plan asks for   */
#define MOE_ECUDA    -3   /* a CUDA runtime/driver call failed (launch, tensor map)   */
#define MOE_ETIMEOUT -4   /* a device-side bounded wait ran out (written to status)   */
#define MOE_ENODEV   -5   /* the current device is not sm_103 (GB300)                 */

/* Layer sizes.  S = D = n_ranks logical ranks; T must divide by n_ranks,
 * n_experts by n_ranks, and (n_experts / n_ranks) by n_waves.  d_model,
 * d_latent, h_expert and h_shared must be multiples of 8 (16-byte rows).
 * Capacity factors are read to six decimals; a factor >= 1e6 or an infinity
 * means "no cap". */
typedef struct moe_config {
    int64_t T;            /* tokens in the batch (may be 0)                          */
    int32_t d_model;      /* d: token state width (6144 in the pages)                */
    int32_t d_latent;     /* L: latent width crossing the exchange (3072)            */
    int32_t n_experts;    /* E: routed experts (384)                                 */
    int32_t n_ranks;      /* S = D: logical expert-parallel ranks (64)               */
    int32_t top_k;        /* k: experts per token (8)                                */
    int32_t n_waves;      /* W: same-shape waves (3)                                 */
    int32_t n_shared;     /* n_s: shared experts (2); 0 allowed                      */
    int32_t h_expert;     /* H: routed SwiGLU hidden size                            */
    int32_t h_shared;     /* Hs: shared SwiGLU hidden size per shared expert         */
    int32_t reserved;     /* must be 0                                               */
    double  cf_send;      /* sender capacity factor (1.10)                           */
    double  cf_recv;      /* receiver capacity factor (1.15)                         */
} moe_config_t;

/* Derived sizes (host-only computation).
 * c_send = ceil(cf_send * (T/S) * k / (D * W)): rows of one (source,
 *   destination, wave) slice -- the uniform expected load of that slice times
 *   the factor.  c_recv = ceil(cf_recv * T * k / E): rows of one expert.
 *   Both are clamped to the most rows that can ever arrive
 *   ((T/S) * min(k, E/D/W) and T).
 * Pool row of (dst, wave, src, slot) = ((dst*W + wave)*S + src)*c_send + slot;
 *   wave w of a destination carries its local experts [w*E_w, (w+1)*E_w),
 *   E_w = E/D/W. */
typedef struct moe_plan {
    int64_t tokens_per_rank;     /* T_s = T / S                                      */
    int32_t experts_per_rank;    /* E_l = E / D                                      */
    int32_t experts_per_wave;    /* E_w = E_l / W                                    */
    int32_t c_send;              /* rows per (src, dst, wave) slice                  */
    int32_t c_recv;              /* rows per expert                                  */
    int64_t pool_rows;           /* D * W * S * c_send                               */
    int64_t pool_row_bytes;      /* 2*L + 16 rounded up to a multiple of 128: L bf16 */
                                 /* payload, 16-byte tag, padding (never written)    */
    int64_t ws_dispatch_bytes;   /* scratch for moe_dispatch_pooled (and the         */
                                 /* overlapped dispatch calls)                       */
    int64_t ws_ffn_bytes;        /* scratch for moe_expert_ffn_grouped (incl. h)     */
    int64_t h_offset_bytes;      /* where h [E, c_recv, H] bf16 sits in ws_ffn       */
} moe_plan_t;

/* Pool row tag (the 16 bytes after the L payload values of every pool row).
 * Filled slot: {expert, token, top-k rank, 0}.  Empty slot: {-1, -1, -1, 0}. */
typedef struct moe_row_tag {
    int32_t expert;
    int32_t token;
    int32_t rank;
    int32_t reserved;
} moe_row_tag_t;

/* Drop accounting, written by moe_dispatch_pooled (device memory). */
typedef struct moe_drop_stats {
    int64_t assignments;    /* T * k                                                 */
    int64_t kept;           /* assignments that reach an expert                      */
    int64_t dropped_send;   /* over the (src, dst, wave) slice capacity              */
    int64_t dropped_recv;   /* sender-kept but over the expert's capacity            */
    int32_t max_send_fill;  /* fullest (src, dst, wave) slice, rows                  */
    int32_t max_expert_rows;/* fullest expert, rows                                  */
    int32_t status;         /* MOE_OK or a device-side error code                    */
    int32_t reserved;
} moe_drop_stats_t;

/* Sizes and scratch requirements; checks the config.  Host only. */
int moe_plan(const moe_config_t* cfg, moe_plan_t* plan);

/* Router: logits = x Wr^T (+ bias), then per token the k largest logits
 * (descending; equal logits -> lower expert id first), gate weights = softmax
 * over the k selected logits, and a near-tie flag.
 *   x      [T, d] bf16        Wr [E, d] bf16        bias [E] fp32 or NULL
 *   logits [T, E] fp32 (out)  idx [T, k] int32 (out)  w [T, k] fp32 (out)
 *   tie    [T] uint8 (out): bit 0 = k-th and (k+1)-th logits closer than
 *          float(1e-4); bit 1 = two adjacent selected logits closer than that.
 * Source: lamjinlab zh-HK section 二 (eight experts per token); the bias is
 * the quantile-balancing bias added to the router logits (devpress.csdn.net,
 * appendix A.2).  Tensor cores: tcgen05 GEMM (one 128 x 384 tile per 128
 * tokens when E <= 384); top-k: one warp per token (k <= 32). */
int moe_router_topk(const moe_config_t* cfg, const uint16_t* x, const uint16_t* Wr,
                    const float* bias, float* logits, int32_t* idx, float* w,
                    uint8_t* tie, int32_t* status, void* stream);

/* Dense projection out[M, N] = bf16(in[M, K] W[N, K]^T), fp32 accumulation.
 * Used for the latent down-projection z = x W_ld^T (lamjinlab zh-HK section
 * 二: 6144 -> 3072 before the exchange).  K and N multiples of 8. */
int moe_latent_proj(const uint16_t* in, const uint16_t* W, int64_t M, int32_t K, int32_t N,
                    uint16_t* out, int32_t* status, void* stream);

/* General bf16 product on the tensor cores with fp32 accumulation (the
 * building block of the layer's backward pass, whose products over the token
 * axis read their operands MN-major):
 *   out[m, n] = sum_k A(m, k) * B(n, k),  m < M, n < N, k < K
 *   A(m, k) = A[m*lda + k] if a_mn == 0 (A stored [M, K]),
 *             A[k*lda + m] if a_mn == 1 (A stored [K, M]);
 *   B(n, k) = B[n*ldb + k] if b_mn == 0, B[k*ldb + n] if b_mn == 1;
 *   out [M, N] row-major with leading dimension ldo, bf16 (out_f32 = 0,
 *   N % 8 == 0) or fp32 (out_f32 = 1).
 * K, lda, ldb multiples of 8; pointers 16-byte aligned. */
int moe_matmul(const uint16_t* A, int a_mn, int64_t lda, const uint16_t* B, int b_mn,
               int64_t ldb, int64_t M, int32_t N, int32_t K, void* out, int out_f32, int64_t ldo,
               int32_t* status, void* stream);

/* moe_router_topk and moe_latent_proj(x, W_ld) in one pass over x: both read
 * the token states (lamjinlab zh-HK section 二: the router picks the experts,
 * the latent projection compresses the routed activations), so one GEMM
 * computes [z | logits] = x [W_ld | Wr]^T, its column tiles writing z (bf16)
 * or logits (fp32 + bias), followed by the top-k kernel.  Same outputs, with
 * the same layouts and the same bits, as the two calls; z [T, L] bf16 is the
 * extra output.  When L is not a multiple of 256 it runs the two calls. */
int moe_route_project(const moe_config_t* cfg, const uint16_t* x, const uint16_t* Wr,
                      const float* bias, const uint16_t* W_ld, float* logits, int32_t* idx,
                      float* w, uint8_t* tie, uint16_t* z, int32_t* status, void* stream);

/* Fixed pooled-wave dispatch (lamjinlab zh-HK section 二: one fixed pool per
 * destination, W same-shape waves, expert id in the payload row, the two
 * capacity factors, drops counted separately).  Priority: token ascending,
 * then top-k rank ascending.  Sender stage per (src, dst, wave) slice, then
 * receiver stage per expert over the sender-kept rows in the same order.
 *   z           [T, L] bf16      idx [T, k] int32 (each row: distinct experts)
 *   ws          scratch, >= plan.ws_dispatch_bytes
 *   pool        [pool_rows, plan.pool_row_bytes / 2] uint16: payload z[t]
 *               (elements 0..L-1) for every sender-kept assignment, tag
 *               (moe_row_tag_t, elements L..L+7) on every row; each row
 *               starts on a 128-byte boundary
 *   slot_of     [T, k] int32: pool row of a kept assignment, else -1
 *   drop        [T, k] uint8: 0 kept, 1 dropped by the sender cap,
 *               2 dropped by the receiver cap
 *   expert_rows [E, c_recv] int32: pool rows of expert e in arrival order,
 *               -1 after expert_count[e]
 *   expert_count[E] int32        stats: moe_drop_stats_t (device)
 *   bank        optional (NULL: not written) [E, c_recv, L] bf16, 16-byte
 *               aligned: the receiver's rows grouped by local expert, i.e.
 *               bank[e][r] = z[t] for the assignment in expert_rows[e][r];
 *               rows r >= expert_count[e] are left as they were.  On one GPU
 *               the receiver side of the exchange lives in the same memory,
 *               so the pack writes this arrangement directly; it lets
 *               moe_expert_ffn_grouped load each expert's rows as whole tiles.
 * Out-of-range expert ids in idx give MOE_EINVAL in stats->status and leave
 * the outputs undefined. */
int moe_dispatch_pooled(const moe_config_t* cfg, const uint16_t* z, const int32_t* idx,
                        void* ws, size_t ws_bytes, uint16_t* pool, int32_t* slot_of,
                        uint8_t* drop, int32_t* expert_rows, int32_t* expert_count,
                        moe_drop_stats_t* stats, uint16_t* bank, void* stream);

/* moe_dispatch_pooled for callers that cannot allocate device memory.  The
 * paper has no counterpart: it is a way of calling the dispatch above.
 * Some callers cannot cudaMalloc: a host application that reserves the
 * device's memory up front and forbids later allocations, code on a
 * latency-critical path where an allocation's implicit device
 * synchronisation is not acceptable, or a plug-in that is handed tensors but
 * no allocator.  This entry point takes the same arguments as
 * moe_dispatch_pooled minus the scratch, and uses instead a fixed array of
 * MOE_DISPATCH_NOALLOC_SCRATCH_BYTES in device memory that the library
 * defines (every GPU that loads the library holds it until the process
 * exits).  It allocates nothing and calls no allocating routine.
 *  - Limit: a configuration whose plan.ws_dispatch_bytes exceeds the array
 *    is rejected with MOE_ENOSPC before anything is enqueued (8 MiB covers
 *    T*k up to about 678,000 assignments at E=384, 64 ranks, 3 waves).
 *  - Set-up: the first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress, with that device current) and caches
 *    it together with the id of the device's CUDA context; make that first
 *    call before any stream capture.  After cudaDeviceReset the device's
 *    next context has another id, so the next call looks the address up
 *    again (and should also come before any capture).
 *  - Sharing: every call on a device uses the same array, which keeps the
 *    last call's contents.  Nothing in it needs to start at zero (each call
 *    writes every word before reading it), but calls whose work overlaps on
 *    the GPU (different streams without ordering between them) race on it.
 * Outputs and errors are those of moe_dispatch_pooled. */
#define MOE_DISPATCH_NOALLOC_SCRATCH_BYTES (8u << 20)
int moe_dispatch_pooled_noalloc(const moe_config_t* cfg, const uint16_t* z, const int32_t* idx,
                                uint16_t* pool, int32_t* slot_of, uint8_t* drop,
                                int32_t* expert_rows, int32_t* expert_count,
                                moe_drop_stats_t* stats, void* stream);

/* Dropless ragged variant: the pages' fallback should drops stay too high
 * (lamjinlab zh-HK section 四, "a ragged all-to-all without drops").  No
 * capacity factor applies; every assignment is kept.  The pool keeps the
 * destination-major order (destination, wave, source, priority), but each
 * (source, destination, wave) block holds exactly the rows routed there, so
 * the pool has T*k rows and no empty slot.
 * moe_plan_ragged: as moe_plan with pool_rows = T*k, c_send = c_recv = 0
 *   (no caps) and the ragged scratch sizes.
 * moe_dispatch_ragged: outputs as moe_dispatch_pooled, except
 *   expert_offsets [E+1] int32: expert e's rows are
 *   expert_rows[expert_offsets[e] .. expert_offsets[e+1]) (flat [T*k] int32,
 *   priority order); expert_count [E] = the differences; drop is all 0 and
 *   slot_of >= 0 everywhere.  bank: optional (NULL: not written) [T*k, L]
 *   bf16, 16-byte aligned, L a multiple of 8: bank[i] = z[t] for the
 *   assignment in expert_rows[i], i.e. every expert's rows contiguous from
 *   row expert_offsets[e], in the row list's order.
 * moe_expert_ffn_ragged: moe_expert_ffn_grouped over those row lists; h
 *   [T*k, H] sits at plan.h_offset_bytes of ws with expert e's rows from
 *   expert_offsets[e].  ypool [T*k, L].  moe_combine applies unchanged.
 *   bank: optional, the one moe_dispatch_ragged wrote (16-byte aligned); with
 *   L a multiple of 256 and H of 128 the products then load each expert's
 *   rows from it as whole tiles (same h and ypool, bit for bit, as without
 *   it); otherwise it is not read. */
int moe_plan_ragged(const moe_config_t* cfg, moe_plan_t* plan);
int moe_dispatch_ragged(const moe_config_t* cfg, const uint16_t* z, const int32_t* idx,
                        void* ws, size_t ws_bytes, uint16_t* pool, int32_t* slot_of,
                        uint8_t* drop, int32_t* expert_offsets, int32_t* expert_rows,
                        int32_t* expert_count, moe_drop_stats_t* stats, uint16_t* bank,
                        void* stream);
/* moe_dispatch_ragged overlapped with the shared experts, as
 * moe_dispatch_shared_overlap does for the capped layout: the same outputs,
 * bit for bit, as moe_dispatch_ragged (the optional bank included) followed
 * by moe_combine's shared step, which writes a [T, n_s*Hs]; the sender
 * stage, the receiver counts and the ragged offsets run as kernels of their
 * own, the final decisions, row lists, payload rows and tags (and the
 * bank's rows) in four extra warps per CTA of the shared gate/up launch.
 * Pass Wsg = Wsu = NULL to moe_combine afterwards.  With n_s = 0 or no
 * tokens it is moe_dispatch_ragged. */
int moe_dispatch_ragged_shared_overlap(const moe_config_t* cfg, const uint16_t* z,
                                       const int32_t* idx, void* ws, size_t ws_bytes,
                                       uint16_t* pool, int32_t* slot_of, uint8_t* drop,
                                       int32_t* expert_offsets, int32_t* expert_rows,
                                       int32_t* expert_count, moe_drop_stats_t* stats,
                                       uint16_t* bank, const uint16_t* x, const uint16_t* Wsg,
                                       const uint16_t* Wsu, uint16_t* a, int32_t* status,
                                       void* stream);
int moe_expert_ffn_ragged(const moe_config_t* cfg, const uint16_t* pool, const uint16_t* bank,
                          const int32_t* expert_offsets, const int32_t* expert_rows,
                          const int32_t* expert_count, const uint16_t* Wg, const uint16_t* Wu,
                          const uint16_t* Wd, void* ws, size_t ws_bytes, uint16_t* ypool,
                          int32_t* status, void* stream);

/* Grouped SwiGLU experts on the received rows: for expert e and r <
 * expert_count[e], with X = payload of pool row expert_rows[e][r]:
 *   h = bf16(silu(X Wg_e^T) * (X Wu_e^T)),  Y = bf16(h Wd_e^T)
 * and Y is written to ypool at that same pool row (the return path keeps the
 * slot).  Rows of ypool that no expert computes are left untouched.
 *   Wg, Wu [E, H, L] bf16     Wd [E, L, H] bf16     ypool [pool_rows, L] bf16
 *   ws     scratch, >= plan.ws_ffn_bytes (holds h [E, c_recv, H] at
 *          plan.h_offset_bytes; rows r < expert_count[e] written)
 *   bank   optional: the per-expert rows written by the dispatch (see
 *          moe_dispatch_pooled); NULL: the rows are gathered from the pool.
 *          With a bank, L a multiple of 256 and H of 128, the products run
 *          on CTA pairs with each expert's rows on the MMA's N axis, in
 *          chunks of at most 256 rows (less padding than 128-row tiles);
 *          otherwise as without it.
 * The pages give each receiver its local experts (section 二) but no
 * activation; the SwiGLU form and the hidden size are the workload's. */
int moe_expert_ffn_grouped(const moe_config_t* cfg, const uint16_t* pool, const uint16_t* bank,
                           const int32_t* expert_rows, const int32_t* expert_count,
                           const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                           void* ws, size_t ws_bytes, uint16_t* ypool, int32_t* status,
                           void* stream);

/* Wave-pipelined dispatch and experts (lamjinlab zh-HK section 二: the
 * waves let the exchange of one wave overlap the computation of another).
 * Same arguments, outputs and errors as moe_dispatch_pooled(cfg, z, idx, ws,
 * ws_bytes, pool, slot_of, drop, expert_rows, expert_count, stats, NULL,
 * stream) followed by moe_expert_ffn_grouped(cfg, pool, NULL, expert_rows,
 * expert_count, Wg, Wu, Wd, ffn_ws, ffn_ws_bytes, ypool, status, stream), and the same
 * results bit for bit.  The dispatch makes every sender and receiver
 * decision but writes only wave 0's payload rows; the gate/up launch, one
 * CTA per SM launched cooperatively, copies the rows of waves 1..W-1 into
 * the pool with four extra warps per CTA while its tensor cores work
 * through wave 0's experts, and a later wave's expert tiles start once
 * every CTA has copied that wave (per-wave counters in ws; the wait is
 * bounded, and on expiry status receives MOE_ETIMEOUT).  With W = 1, no
 * tokens or c_recv = 0 it is exactly the two calls.  ws must not be shared
 * with other work in flight. */
int moe_dispatch_expert_waves(const moe_config_t* cfg, const uint16_t* z, const int32_t* idx,
                              void* ws, size_t ws_bytes, uint16_t* pool, int32_t* slot_of,
                              uint8_t* drop, int32_t* expert_rows, int32_t* expert_count,
                              moe_drop_stats_t* stats, const uint16_t* Wg, const uint16_t* Wu,
                              const uint16_t* Wd, void* ffn_ws, size_t ffn_ws_bytes,
                              uint16_t* ypool, int32_t* status, void* stream);

/* Dispatch overlapped with the shared experts.  The shared experts see every
 * token and do not depend on the routing (lamjinlab zh-HK section 四: a dense
 * backbone beside the routed experts), so the exchange can proceed while
 * they compute.  Same arguments, outputs and errors as moe_dispatch_pooled
 * (the optional bank included), plus the shared experts' activations
 *   a = bf16(silu(x Wsg_s^T) * (x Wsu_s^T)), [T, n_s*Hs] (as moe_combine)
 *   x [T, d]  Wsg, Wsu [n_s, Hs, d]  status: device status word
 * and the same results bit for bit as moe_dispatch_pooled followed by
 * moe_combine's shared step.  The sender stage and the receiver counts run
 * as kernels of their own; the final decisions (slot_of, drop codes, the
 * expert row lists) and the pool's payload rows and tags (and the bank's
 * rows) are written by four extra warps per CTA of the shared gate/up
 * launch.  Pass
 * Wsg = Wsu = NULL to moe_combine afterwards so that it uses this a.  With
 * n_s = 0 or no tokens it is moe_dispatch_pooled. */
int moe_dispatch_shared_overlap(const moe_config_t* cfg, const uint16_t* z, const int32_t* idx,
                                void* ws, size_t ws_bytes, uint16_t* pool, int32_t* slot_of,
                                uint8_t* drop, int32_t* expert_rows, int32_t* expert_count,
                                moe_drop_stats_t* stats, uint16_t* bank, const uint16_t* x,
                                const uint16_t* Wsg, const uint16_t* Wsu, uint16_t* a,
                                int32_t* status, void* stream);

/* Return path, weighted combine, up-projection and shared experts:
 *   c[t]   = bf16(sum over kept j, in j order, of w[t,j] * ypool[slot_of[t,j]])
 *   a      = bf16(silu(x Wsg_s^T) * (x Wsu_s^T)) for each shared expert s,
 *            concatenated along the hidden axis: [T, n_s*Hs]
 *   out    = bf16(c W_lu^T + sum_s a_s Wsd_s^T)     (fp32 accumulation)
 * Dropped assignments contribute nothing and weights are not renormalised;
 * the shared experts see every token (lamjinlab zh-HK sections 二 and 四).
 *   ypool [pool_rows, L]  slot_of [T, k]  w [T, k] fp32  W_lu [d, L]  x [T, d]
 *   Wsg, Wsu [n_s, Hs, d]  Wsd [n_s, d, Hs]
 *   c [T, L] bf16 (out)  a [T, n_s*Hs] bf16 (out)  out [T, d] bf16 (out)
 * Wsg = Wsu = NULL (n_s > 0): a is an input holding the shared activations
 * (from moe_dispatch_shared_overlap) and x may be NULL. */
int moe_combine(const moe_config_t* cfg, const uint16_t* ypool, const int32_t* slot_of,
                const float* w, const uint16_t* W_lu, const uint16_t* x,
                const uint16_t* Wsg, const uint16_t* Wsu, const uint16_t* Wsd,
                uint16_t* c, uint16_t* a, uint16_t* out, int32_t* status, void* stream);

/* The whole layer forward in one call, and a pipeline that feeds it from
 * host memory.  These compose the calls above; the pages describe the layer
 * (lamjinlab zh-HK section 二), not this packaging of it.
 *
 * moe_layer_buffers_t: every device buffer of one layer instance (caller-
 * owned; sizes as for the individual calls: logits [T, E] fp32, idx, w
 * [T, k], tie [T], z [T, L], ws_dispatch >= plan.ws_dispatch_bytes, pool,
 * slot_of, drop, expert_rows, expert_count, stats, bank (optional, NULL:
 * no bank), ws_ffn >= plan.ws_ffn_bytes, ypool [pool_rows, L], c [T, L],
 * a [T, n_s*Hs] (NULL when n_s = 0), status), plus the weights (bias
 * optional).
 *
 * moe_layer_forward: out = layer(x) for device x [T, d] and out [T, d]
 * bf16, enqueued on `stream`: moe_route_project; with shared experts
 * moe_dispatch_shared_overlap (the pool fill inside their gate/up launch),
 * else moe_dispatch_pooled; moe_expert_ffn_grouped; moe_combine.  Results as
 * those calls in that order; errors as theirs (the first one returned). */
typedef struct moe_layer_buffers {
    const uint16_t* Wr;
    const float* bias;
    const uint16_t* W_ld;
    const uint16_t* Wg;
    const uint16_t* Wu;
    const uint16_t* Wd;
    const uint16_t* W_lu;
    const uint16_t* Wsg;
    const uint16_t* Wsu;
    const uint16_t* Wsd;
    float* logits;
    int32_t* idx;
    float* w;
    uint8_t* tie;
    uint16_t* z;
    void* ws_dispatch;
    size_t ws_dispatch_bytes;
    uint16_t* pool;
    int32_t* slot_of;
    uint8_t* drop;
    int32_t* expert_rows;
    int32_t* expert_count;
    moe_drop_stats_t* stats;
    uint16_t* bank;
    void* ws_ffn;
    size_t ws_ffn_bytes;
    uint16_t* ypool;
    uint16_t* c;
    uint16_t* a;
    int32_t* status;
} moe_layer_buffers_t;

int moe_layer_forward(const moe_config_t* cfg, const moe_layer_buffers_t* buffers,
                      const uint16_t* x, uint16_t* out, void* stream);

/* Host-memory pipeline over moe_layer_forward, as a serving loop runs it:
 * batch i's x is copied host -> device on the pipeline's own stream while
 * batch i-1 computes on the caller's stream and batch i-2's output (and
 * drop statistics) copy back on a second stream of its own; events order
 * the three over a ring of `depth` device staging buffers.
 *   create:  x_dev[depth], out_dev[depth] [T, d] bf16 and stats_dev[depth]
 *            (device, caller-owned, 16- and 8-byte aligned) form the ring;
 *            the pipeline creates its two streams and 3*depth events on the
 *            current device (no device memory).  MOE_EINVAL on bad
 *            arguments, MOE_ECUDA if a stream or event cannot be created.
 *   submit:  enqueue one batch: x_host [T, d] -> the layer (buffers, on
 *            `stream`) -> out_host [T, d] and, if not NULL, stats_host.  All
 *            asynchronous; host buffers should be pinned for the copies to
 *            overlap.  Call with the pipeline's device current.  After an
 *            error the pipeline's state is undefined: destroy it.
 *   sync:    wait until every submitted batch's copies back have landed.
 *   destroy: sync, then release the streams and events. */
typedef struct moe_host_pipe moe_host_pipe_t;
int moe_host_pipe_create(const moe_config_t* cfg, int depth, uint16_t* const* x_dev,
                         uint16_t* const* out_dev, moe_drop_stats_t* const* stats_dev,
                         moe_host_pipe_t** pipe);
int moe_host_pipe_submit(moe_host_pipe_t* pipe, const moe_layer_buffers_t* buffers,
                         const uint16_t* x_host, uint16_t* out_host,
                         moe_drop_stats_t* stats_host, void* stream);
int moe_host_pipe_sync(moe_host_pipe_t* pipe);
int moe_host_pipe_destroy(moe_host_pipe_t* pipe);

/* Backward pass of the layer (capped layout).  The pages give the forward
 * only; the throughput they quote is a training step, so this is the
 * forward's derivative, step by step in reverse: output layer, shared
 * experts (their gate/up recomputed), combine (dY = w dc, dw = <dc, Y>),
 * routed experts (gate/up recomputed; dh, dg, du, dX, weight gradients), the
 * return of dX to the tokens (dz), the latent projection, the router
 * (softmax over the selected logits; the balancing bias is stop-gradient)
 * and dx.  Storage precision: activation gradients bf16 (dc, da, dY, dh, dg,
 * du, dX, dz, dlogits, dx), weight gradients fp32, all products accumulate
 * in fp32.
 * moe_backward_plan: byte offsets of the intermediates inside the scratch
 *   and its total size (layout->total).  Among them: dY and X of the routed
 *   experts in per-expert row order ([E, c_recv, L], dye and xe), rowinv
 *   (int32 per pool row: e * c_recv + r for the r-th row of expert e), dX in
 *   pool row order (dxpool) and dh, dg, du ([E, c_recv, H]).
 * moe_layer_backward: inputs are the forward's inputs and the tensors its
 *   calls produced (idx, w, pool, slot_of, expert_rows, expert_count, h =
 *   ws_ffn + plan.h_offset_bytes, ypool, c, a), plus dout [T, d] bf16.
 *   Weight gradients are written (not accumulated) in the weights' own
 *   layouts: dWr [E, d], dW_ld [L, d], dWg, dWu [E, H, L], dWd [E, L, H],
 *   dW_lu [d, L], dWsg, dWsu [n_s, Hs, d], dWsd [n_s, d, Hs], all fp32;
 *   dx [T, d] bf16.  The rows of h past each expert's count are set to zero
 *   (they were never written by the forward).  All device pointers,
 *   16-byte aligned; scratch ws of at least layout.total bytes. */
typedef struct moe_backward_ws {
    int64_t dc, da, dgs, dus, dw, rowinv, dxpool, dh, dg, du, xe, dye, dz, dlogits, tiles;
    int64_t hp, poff;   /* dropless layout only (else 0): padded copy of h, row offsets */
    int64_t total;
} moe_backward_ws_t;

typedef struct moe_backward_args {
    const uint16_t *x, *Wr, *W_ld, *Wg, *Wu, *Wd, *W_lu, *Wsg, *Wsu, *Wsd;
    const int32_t* idx;
    const float* w;
    const uint16_t* pool;
    const int32_t *slot_of, *expert_rows, *expert_count;
    uint16_t* h;
    const uint16_t *ypool, *c, *a;
    const uint16_t* dout;
    uint16_t* dx;
    float *dWr, *dW_ld, *dWg, *dWu, *dWd, *dW_lu, *dWsg, *dWsu, *dWsd;
    void* ws;
    size_t ws_bytes;
    int32_t* status;
    const int32_t* expert_offsets;   /* dropless layout: [E + 1], from moe_dispatch_ragged;
                                        NULL for the capped layout */
    uint16_t* bank;                  /* capped layout, optional (NULL: not used): the
                                        forward dispatch's per-expert bank [E, c_recv, L];
                                        X is then read from it instead of copied out of
                                        the pool rows (the same values), and its rows past
                                        each expert's count are set to zero.  Ignored by
                                        the dropless backward. */
} moe_backward_args_t;

int moe_backward_plan(const moe_config_t* cfg, moe_backward_ws_t* layout);
int moe_layer_backward(const moe_config_t* cfg, const moe_backward_args_t* args, void* stream);

/* The backward pass of the dropless ragged layer (the forward of
 * moe_dispatch_ragged + moe_expert_ffn_ragged + moe_combine): the same
 * derivative, every assignment kept.  args as for moe_layer_backward, with
 * expert_rows / expert_offsets / expert_count of the ragged dispatch and h
 * the flat [T*k, H] of moe_expert_ffn_ragged (left unchanged).  In the
 * scratch, expert e's rows are padded to a multiple of 64 at poff[e]
 * (int32 [E+1] at layout.poff) in dye, xe, dh, dg, du and a padded copy of h
 * (layout.hp), so that each expert's weight gradient contracts over whole
 * 64-row blocks; rowinv maps pool rows to those positions. */
int moe_backward_plan_ragged(const moe_config_t* cfg, moe_backward_ws_t* layout);
int moe_layer_backward_ragged(const moe_config_t* cfg, const moe_backward_args_t* args,
                              void* stream);

/* Quantile-balancing bias update (devpress.csdn.net, section 四 and appendix
 * A.2): a global histogram H counts how often each expert was selected;
 * f_e = H[e] / sum(H); b_e = -alpha * (f_e - 1/E); the bias is added to the
 * router logits from the next batch on, without gradient.
 *   idx   [T, k] int32: this batch's top-k selections (before capacity drops)
 *   hist  [E] int64 (in/out): the histogram; this batch's counts are added.
 *         It accumulates over every call since the caller last zeroed it, so
 *         the caller chooses the window of batches.
 *   bias  [E] fp32 (out): the new bias; 0 everywhere while H is empty.  It
 *         may be the buffer moe_router_topk reads: calls on the same stream
 *         then route the next batch with it.
 * For an exact window of the past N batches see moe_balance_update_window. */
int moe_balance_update(const moe_config_t* cfg, const int32_t* idx, int64_t* hist, float alpha,
                       float* bias, void* stream);

/* The same bias with H over exactly the past `window` batches (appendix
 * A.2: "the past N batches"; section 四's "10,000 bins" read as that window
 * length, the caller's choice).  Each call counts this batch's selections,
 * takes the counts of the batch leaving the window out of H and puts this
 * batch's in, then writes the bias as moe_balance_update does.
 *   hist   [E] int64 (in/out): H, zero before the first call
 *   ring   [window, E] int64 (in/out): per-batch counts, batch b in row
 *          b % window; zero before the first call
 *   step   [1] int64 (in/out, device): batches seen so far, zero before the
 *          first call (kept on the device: the update needs no host state
 *          and can be captured in a CUDA graph)
 *   window >= 1, else MOE_EINVAL. */
int moe_balance_update_window(const moe_config_t* cfg, const int32_t* idx, int64_t* hist,
                              int64_t* ring, int32_t window, int64_t* step, float alpha,
                              float* bias, void* stream);

/* Index checks of a checked build (compiled with -DMOE_CHECK=1; the pages
 * define no such operation): every row, slot, expert and tile index the
 * kernels compute is checked before use; a failed check skips the access
 * and records a site code (1001.. by kernel) in a device word.  Returns the
 * first recorded code since the last call (0: none) and resets it; a normal
 * build always returns 0.  Synchronous: call after the work has finished. */
int moe_check_status(void);

/* Checked builds only (libmoe_pooled_wave_check.so; a normal build does not
 * export it; the pages define no such operation): sets the limit, in ns of
 * the GPU's global timer, of the wave pipeline's wait for every CTA's count
 * of a wave (moe_dispatch_expert_waves; default 4e9 = 4 s).  A test sets it
 * near 0 so that the wait runs out on legitimate work: the waiting threads
 * record MOE_ETIMEOUT in the status word, raise their CTA's abort flag and
 * the CTA unwinds (armed copies land, issued MMAs finish, TMEM is freed)
 * and returns.  The waits that drain copies and MMAs keep their own limits.
 * Affects launches enqueued after it returns, on the current device.
 * Returns MOE_OK, or MOE_ECUDA if the device symbol cannot be written. */
int moe_check_set_wave_wait_limit_ns(unsigned long long ns);

/* Kernel timing trace (instrumentation; the pages define no such operation).
 * moe_trace_begin(n) creates n CUDA events (timing enabled) owned by the
 *   library and turns tracing on; from then on every kernel the library
 *   launches is followed by a cudaEventRecord of the next event on the same
 *   stream, until n events are used.  n = 0 frees the events.  Host only,
 *   process-wide; do not trace while capturing a CUDA graph.
 * moe_trace_mark(stream) records the next event with the name "mark".
 * moe_trace_end() turns tracing off and returns the number of events used.
 * moe_trace_event(i, &name, &ms) waits for event i and returns the name of
 *   the kernel it follows and the milliseconds since event i-1 (0 for i=0).
 *   name points to a static string. */
int moe_trace_begin(int n);
int moe_trace_mark(void* stream);
int moe_trace_end(void);
int moe_trace_event(int i, const char** name, float* ms_since_prev);

/* Human-readable name of a MOE_* code (static string). */
const char* moe_strerror(int code);

/* ABI version: 6 (2: the optional per-expert bank of the dispatch and the
 * expert FFN; 3: the whole-layer forward and the host-memory pipeline; 4: the
 * optional bank of the dropless dispatch and expert FFN; 5: the optional bank
 * as the backward's source of X; 6: the dropless dispatch overlapped with the
 * shared experts). */
int moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_POOLED_WAVE_H */
