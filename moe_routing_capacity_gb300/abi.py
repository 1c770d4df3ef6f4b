"""ctypes binding of ``libmoe_pooled_wave.so`` (the C ABI in
``include/moe_pooled_wave.h``).

Argument marshalling only: each function takes torch tensors, checks dtype,
device and contiguity, and passes raw pointers, sizes and the current CUDA
stream to the C entry point of the same name.  Every step of the layer runs
in the library's kernels; if the library is missing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_pooled_wave.so")

MOE_OK, MOE_EINVAL, MOE_ENOSPC, MOE_ECUDA, MOE_ETIMEOUT, MOE_ENODEV = 0, -1, -2, -3, -4, -5

# Every entry point the header declares (checked by the tests).
EXPORTS = ("moe_plan", "moe_router_topk", "moe_latent_proj", "moe_route_project", "moe_matmul",
           "moe_dispatch_pooled",
           "moe_dispatch_pooled_noalloc", "moe_expert_ffn_grouped", "moe_dispatch_expert_waves",
           "moe_dispatch_shared_overlap", "moe_balance_update", "moe_balance_update_window",
           "moe_plan_ragged", "moe_dispatch_ragged", "moe_dispatch_ragged_shared_overlap",
           "moe_expert_ffn_ragged",
           "moe_backward_plan", "moe_layer_backward", "moe_backward_plan_ragged",
           "moe_layer_backward_ragged", "moe_combine", "moe_trace_begin", "moe_trace_mark",
           "moe_trace_end", "moe_trace_event", "moe_check_status", "moe_strerror",
           "moe_abi_version", "moe_layer_forward", "moe_host_pipe_create", "moe_host_pipe_submit",
           "moe_host_pipe_sync", "moe_host_pipe_destroy")
# Declared in the header too, but exported by the checked build only.
CHECKED_ONLY = ("moe_check_set_wave_wait_limit_ns",)


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d_model", ctypes.c_int32), ("d_latent", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("n_ranks", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_waves", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("h_expert", ctypes.c_int32),
                ("h_shared", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("cf_send", ctypes.c_double), ("cf_recv", ctypes.c_double)]


class Plan(ctypes.Structure):
    _fields_ = [("tokens_per_rank", ctypes.c_int64), ("experts_per_rank", ctypes.c_int32),
                ("experts_per_wave", ctypes.c_int32), ("c_send", ctypes.c_int32),
                ("c_recv", ctypes.c_int32), ("pool_rows", ctypes.c_int64),
                ("pool_row_bytes", ctypes.c_int64), ("ws_dispatch_bytes", ctypes.c_int64),
                ("ws_ffn_bytes", ctypes.c_int64), ("h_offset_bytes", ctypes.c_int64)]


class DropStats(ctypes.Structure):
    _fields_ = [("assignments", ctypes.c_int64), ("kept", ctypes.c_int64),
                ("dropped_send", ctypes.c_int64), ("dropped_recv", ctypes.c_int64),
                ("max_send_fill", ctypes.c_int32), ("max_expert_rows", ctypes.c_int32),
                ("status", ctypes.c_int32), ("reserved", ctypes.c_int32)]


STATS_WORDS = ctypes.sizeof(DropStats) // 8    # int64 words of a stats record

BWD_WS_FIELDS = ("dc", "da", "dgs", "dus", "dw", "rowinv", "dxpool", "dh", "dg", "du", "xe", "dye",
                 "dz", "dlogits", "tiles", "hp", "poff", "total")


class BackwardWs(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int64) for f in BWD_WS_FIELDS]


BWD_ARG_FIELDS = ("x", "Wr", "W_ld", "Wg", "Wu", "Wd", "W_lu", "Wsg", "Wsu", "Wsd", "idx", "w",
                  "pool", "slot_of", "expert_rows", "expert_count", "h", "ypool", "c", "a",
                  "dout", "dx", "dWr", "dW_ld", "dWg", "dWu", "dWd", "dW_lu", "dWsg", "dWsu",
                  "dWsd", "ws")


class BackwardArgs(ctypes.Structure):
    _fields_ = ([(f, ctypes.c_void_p) for f in BWD_ARG_FIELDS] +
                [("ws_bytes", ctypes.c_size_t), ("status", ctypes.c_void_p),
                 ("expert_offsets", ctypes.c_void_p), ("bank", ctypes.c_void_p)])

LAYER_BUFFER_FIELDS = ("Wr", "bias", "W_ld", "Wg", "Wu", "Wd", "W_lu", "Wsg", "Wsu", "Wsd",
                       "logits", "idx", "w", "tie", "z", "ws_dispatch", "ws_dispatch_bytes",
                       "pool", "slot_of", "drop", "expert_rows", "expert_count", "stats", "bank",
                       "ws_ffn", "ws_ffn_bytes", "ypool", "c", "a", "status")


class LayerBuffers(ctypes.Structure):
    _fields_ = [(f, ctypes.c_size_t if f.endswith("_bytes") else ctypes.c_void_p)
                for f in LAYER_BUFFER_FIELDS]

_lib = None


def lib() -> ctypes.CDLL:
    """Load the library once; raise if it has not been built."""
    global _lib
    if _lib is None:
        _lib = load_library(LIB_PATH)
    return _lib


def load_library(path: str) -> ctypes.CDLL:
    """Load one build of the library (e.g. the checked one) with its
    signatures declared; ``lib()`` serves the package's own build."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m moe_routing_capacity_gb300.build`")
    L = ctypes.CDLL(path)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    pc = ctypes.POINTER(Config)
    L.moe_plan.argtypes = [pc, ctypes.POINTER(Plan)]
    L.moe_router_topk.argtypes = [pc, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_latent_proj.argtypes = [vp, vp, i64, i32, i32, vp, vp, vp]
    L.moe_route_project.argtypes = [pc, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_matmul.argtypes = [vp, ctypes.c_int, i64, vp, ctypes.c_int, i64, i64, i32, i32, vp,
                             ctypes.c_int, i64, vp, vp]
    L.moe_dispatch_pooled.argtypes = [pc, vp, vp, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_dispatch_pooled_noalloc.argtypes = [pc, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_expert_ffn_grouped.argtypes = [pc, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    L.moe_combine.argtypes = [pc, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_dispatch_expert_waves.argtypes = [pc, vp, vp, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp,
                                            vp, vp, sz, vp, vp, vp]
    L.moe_dispatch_shared_overlap.argtypes = [pc, vp, vp, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp,
                                              vp, vp, vp, vp, vp]
    L.moe_balance_update.argtypes = [pc, vp, vp, ctypes.c_float, vp, vp]
    L.moe_balance_update_window.argtypes = [pc, vp, vp, vp, i32, vp, ctypes.c_float, vp, vp]
    L.moe_plan_ragged.argtypes = [pc, ctypes.POINTER(Plan)]
    L.moe_dispatch_ragged.argtypes = [pc, vp, vp, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_dispatch_ragged_shared_overlap.argtypes = [pc, vp, vp, vp, sz, vp, vp, vp, vp, vp, vp,
                                                     vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_expert_ffn_ragged.argtypes = [pc, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    L.moe_backward_plan.argtypes = [pc, ctypes.POINTER(BackwardWs)]
    L.moe_layer_backward.argtypes = [pc, ctypes.POINTER(BackwardArgs), vp]
    L.moe_backward_plan_ragged.argtypes = [pc, ctypes.POINTER(BackwardWs)]
    L.moe_layer_backward_ragged.argtypes = [pc, ctypes.POINTER(BackwardArgs), vp]
    L.moe_strerror.argtypes = [ctypes.c_int]
    L.moe_strerror.restype = ctypes.c_char_p
    L.moe_abi_version.argtypes = []
    L.moe_check_status.argtypes = []
    L.moe_trace_begin.argtypes = [ctypes.c_int]
    L.moe_trace_mark.argtypes = [vp]
    L.moe_trace_end.argtypes = []
    L.moe_trace_event.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                                  ctypes.POINTER(ctypes.c_float)]
    for n in EXPORTS:
        if n != "moe_strerror":
            getattr(L, n).restype = ctypes.c_int
    pb = ctypes.POINTER(LayerBuffers)
    L.moe_layer_forward.argtypes = [pc, pb, vp, vp, vp]
    L.moe_host_pipe_create.argtypes = [pc, ctypes.c_int, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                       ctypes.POINTER(vp), ctypes.POINTER(vp)]
    L.moe_host_pipe_submit.argtypes = [vp, pb, vp, vp, vp, vp]
    L.moe_host_pipe_sync.argtypes = [vp]
    L.moe_host_pipe_destroy.argtypes = [vp]
    if hasattr(L, "moe_check_set_wave_wait_limit_ns"):
        L.moe_check_set_wave_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        L.moe_check_set_wave_wait_limit_ns.restype = ctypes.c_int
    return L


def strerror(code: int) -> str:
    return lib().moe_strerror(code).decode()


def make_config(cfg) -> Config:
    """C config from any object with the layer-size attributes."""
    return Config(cfg.T, cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.n_ranks, cfg.top_k,
                  cfg.n_waves, cfg.n_shared, cfg.h_expert, cfg.h_shared, 0,
                  float(cfg.cf_send), float(cfg.cf_recv))


def plan(cfg) -> Plan:
    p = Plan()
    rc = lib().moe_plan(ctypes.byref(make_config(cfg)), ctypes.byref(p))
    if rc:
        raise MoeError("moe_plan", rc)
    return p


def plan_ragged(cfg) -> Plan:
    p = Plan()
    rc = lib().moe_plan_ragged(ctypes.byref(make_config(cfg)), ctypes.byref(p))
    if rc:
        raise MoeError("moe_plan_ragged", rc)
    return p


def _ptr(t, dtype=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError("tensor required")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError("tensors must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, rc):
    if rc:
        raise MoeError(fn, rc)


bf16, f32, i32, u8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8


def router_topk(cfg, x, Wr, bias, logits, idx, w, tie, status, stream=None):
    _check("moe_router_topk", lib().moe_router_topk(
        ctypes.byref(make_config(cfg)), _ptr(x, bf16), _ptr(Wr, bf16),
        _ptr(bias, f32, allow_none=True), _ptr(logits, f32), _ptr(idx, i32), _ptr(w, f32),
        _ptr(tie, u8), _ptr(status, i32), _stream(stream)))


def latent_proj(inp, W, out, status, stream=None):
    M, K = inp.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(out.shape) != (M, N):
        raise ValueError("shape mismatch")
    _check("moe_latent_proj", lib().moe_latent_proj(
        _ptr(inp, bf16), _ptr(W, bf16), M, K, N, _ptr(out, bf16), _ptr(status, i32),
        _stream(stream)))


def matmul(A, B, M, N, K, out, status, a_mn=False, b_mn=False, stream=None):
    """out[M, N] = sum_k A(m, k) B(n, k); A stored [M, K] (or [K, M] if a_mn),
    B stored [N, K] (or [K, N] if b_mn); out bf16 or fp32, row-major."""
    lda, ldb = A.shape[1], B.shape[1]
    _check("moe_matmul", lib().moe_matmul(
        _ptr(A, bf16), int(bool(a_mn)), lda, _ptr(B, bf16), int(bool(b_mn)), ldb, M, N, K,
        _ptr(out), int(out.dtype == torch.float32), out.shape[1], _ptr(status, i32),
        _stream(stream)))


def route_project(cfg, x, Wr, bias, W_ld, logits, idx, w, tie, z, status, stream=None):
    _check("moe_route_project", lib().moe_route_project(
        ctypes.byref(make_config(cfg)), _ptr(x, bf16), _ptr(Wr, bf16),
        _ptr(bias, f32, allow_none=True), _ptr(W_ld, bf16), _ptr(logits, f32), _ptr(idx, i32),
        _ptr(w, f32), _ptr(tie, u8), _ptr(z, bf16), _ptr(status, i32), _stream(stream)))


def dispatch_pooled(cfg, z, idx, ws, pool, slot_of, drop, expert_rows, expert_count, stats,
                    stream=None, bank=None):
    """bank (optional, [E, c_recv, L] bf16): also receives each receiver-kept
    row at its expert's receiver rank."""
    _check("moe_dispatch_pooled", lib().moe_dispatch_pooled(
        ctypes.byref(make_config(cfg)), _ptr(z, bf16), _ptr(idx, i32), _ptr(ws, u8),
        ws.numel(), _ptr(pool, torch.int16), _ptr(slot_of, i32), _ptr(drop, u8),
        _ptr(expert_rows, i32), _ptr(expert_count, i32), _ptr(stats, torch.int64),
        _ptr(bank, bf16, allow_none=True), _stream(stream)))


# MOE_DISPATCH_NOALLOC_SCRATCH_BYTES of the header (a host test checks that
# the two agree)
NOALLOC_SCRATCH_BYTES = 8 << 20


def dispatch_pooled_noalloc(cfg, z, idx, pool, slot_of, drop, expert_rows, expert_count, stats,
                            stream=None):
    """moe_dispatch_pooled with the library's fixed scratch array instead of a
    caller-provided one (for callers that cannot allocate device memory)."""
    _check("moe_dispatch_pooled_noalloc", lib().moe_dispatch_pooled_noalloc(
        ctypes.byref(make_config(cfg)), _ptr(z, bf16), _ptr(idx, i32),
        _ptr(pool, torch.int16), _ptr(slot_of, i32), _ptr(drop, u8), _ptr(expert_rows, i32),
        _ptr(expert_count, i32), _ptr(stats, torch.int64), _stream(stream)))


def expert_ffn_grouped(cfg, pool, expert_rows, expert_count, Wg, Wu, Wd, ws, ypool, status,
                       stream=None, bank=None):
    """bank (optional): the per-expert rows the dispatch wrote; None gathers
    the rows from the pool."""
    _check("moe_expert_ffn_grouped", lib().moe_expert_ffn_grouped(
        ctypes.byref(make_config(cfg)), _ptr(pool, torch.int16),
        _ptr(bank, bf16, allow_none=True), _ptr(expert_rows, i32),
        _ptr(expert_count, i32), _ptr(Wg, bf16), _ptr(Wu, bf16), _ptr(Wd, bf16),
        _ptr(ws, u8), ws.numel(), _ptr(ypool, bf16), _ptr(status, i32), _stream(stream)))


def dispatch_expert_waves(cfg, z, idx, ws, pool, slot_of, drop, expert_rows, expert_count, stats,
                          Wg, Wu, Wd, ffn_ws, ypool, status, stream=None):
    """dispatch_pooled then expert_ffn_grouped, with the later waves' pool rows
    copied inside the gate/up launch while wave 0's experts compute."""
    _check("moe_dispatch_expert_waves", lib().moe_dispatch_expert_waves(
        ctypes.byref(make_config(cfg)), _ptr(z, bf16), _ptr(idx, i32), _ptr(ws, u8),
        ws.numel(), _ptr(pool, torch.int16), _ptr(slot_of, i32), _ptr(drop, u8),
        _ptr(expert_rows, i32), _ptr(expert_count, i32), _ptr(stats, torch.int64),
        _ptr(Wg, bf16), _ptr(Wu, bf16), _ptr(Wd, bf16), _ptr(ffn_ws, u8), ffn_ws.numel(),
        _ptr(ypool, bf16), _ptr(status, i32), _stream(stream)))


def dispatch_shared_overlap(cfg, z, idx, ws, pool, slot_of, drop, expert_rows, expert_count,
                            stats, x, Wsg, Wsu, a, status, stream=None, bank=None):
    """dispatch_pooled plus the shared experts' activations a, the pool rows
    copied while the shared gate/up product computes; then call combine with
    Wsg = Wsu = None."""
    _check("moe_dispatch_shared_overlap", lib().moe_dispatch_shared_overlap(
        ctypes.byref(make_config(cfg)), _ptr(z, bf16), _ptr(idx, i32), _ptr(ws, u8),
        ws.numel(), _ptr(pool, torch.int16), _ptr(slot_of, i32), _ptr(drop, u8),
        _ptr(expert_rows, i32), _ptr(expert_count, i32), _ptr(stats, torch.int64),
        _ptr(bank, bf16, allow_none=True),
        _ptr(x, bf16, allow_none=True), _ptr(Wsg, bf16, allow_none=True),
        _ptr(Wsu, bf16, allow_none=True), _ptr(a, bf16, allow_none=True), _ptr(status, i32),
        _stream(stream)))


def dispatch_ragged(cfg, z, idx, ws, pool, slot_of, drop, expert_offsets, expert_rows,
                    expert_count, stats, stream=None, bank=None):
    _check("moe_dispatch_ragged", lib().moe_dispatch_ragged(
        ctypes.byref(make_config(cfg)), _ptr(z, bf16), _ptr(idx, i32), _ptr(ws, u8),
        ws.numel(), _ptr(pool, torch.int16), _ptr(slot_of, i32), _ptr(drop, u8),
        _ptr(expert_offsets, i32), _ptr(expert_rows, i32), _ptr(expert_count, i32),
        _ptr(stats, torch.int64), _ptr(bank, bf16, allow_none=True), _stream(stream)))


def dispatch_ragged_shared_overlap(cfg, z, idx, ws, pool, slot_of, drop, expert_offsets,
                                   expert_rows, expert_count, stats, x, Wsg, Wsu, a, status,
                                   stream=None, bank=None):
    """dispatch_ragged plus the shared experts' activations a, the pack run
    inside the shared gate/up product; then call combine with Wsg = Wsu = None."""
    _check("moe_dispatch_ragged_shared_overlap", lib().moe_dispatch_ragged_shared_overlap(
        ctypes.byref(make_config(cfg)), _ptr(z, bf16), _ptr(idx, i32), _ptr(ws, u8),
        ws.numel(), _ptr(pool, torch.int16), _ptr(slot_of, i32), _ptr(drop, u8),
        _ptr(expert_offsets, i32), _ptr(expert_rows, i32), _ptr(expert_count, i32),
        _ptr(stats, torch.int64), _ptr(bank, bf16, allow_none=True),
        _ptr(x, bf16, allow_none=True), _ptr(Wsg, bf16, allow_none=True),
        _ptr(Wsu, bf16, allow_none=True), _ptr(a, bf16, allow_none=True), _ptr(status, i32),
        _stream(stream)))


def expert_ffn_ragged(cfg, pool, expert_offsets, expert_rows, expert_count, Wg, Wu, Wd, ws,
                      ypool, status, stream=None, bank=None):
    _check("moe_expert_ffn_ragged", lib().moe_expert_ffn_ragged(
        ctypes.byref(make_config(cfg)), _ptr(pool, torch.int16),
        _ptr(bank, bf16, allow_none=True), _ptr(expert_offsets, i32),
        _ptr(expert_rows, i32), _ptr(expert_count, i32), _ptr(Wg, bf16), _ptr(Wu, bf16),
        _ptr(Wd, bf16), _ptr(ws, u8), ws.numel(), _ptr(ypool, bf16), _ptr(status, i32),
        _stream(stream)))


def balance_update(cfg, idx, hist, alpha, bias, stream=None):
    _check("moe_balance_update", lib().moe_balance_update(
        ctypes.byref(make_config(cfg)), _ptr(idx, i32), _ptr(hist, torch.int64),
        float(alpha), _ptr(bias, f32), _stream(stream)))


def balance_update_window(cfg, idx, hist, ring, step, alpha, bias, stream=None):
    """moe_balance_update over exactly the past ring.shape[0] batches (ring
    [N, E] int64 and step [1] int64 live on the device, zero at the start)."""
    _check("moe_balance_update_window", lib().moe_balance_update_window(
        ctypes.byref(make_config(cfg)), _ptr(idx, i32), _ptr(hist, torch.int64),
        _ptr(ring, torch.int64), int(ring.shape[0]), _ptr(step, torch.int64), float(alpha),
        _ptr(bias, f32), _stream(stream)))


def combine(cfg, ypool, slot_of, w, W_lu, x, Wsg, Wsu, Wsd, c, a, out, status, stream=None):
    _check("moe_combine", lib().moe_combine(
        ctypes.byref(make_config(cfg)), _ptr(ypool, bf16), _ptr(slot_of, i32), _ptr(w, f32),
        _ptr(W_lu, bf16), _ptr(x, bf16, allow_none=True), _ptr(Wsg, bf16, allow_none=True),
        _ptr(Wsu, bf16, allow_none=True), _ptr(Wsd, bf16, allow_none=True),
        _ptr(c, bf16), _ptr(a, bf16, allow_none=True), _ptr(out, bf16), _ptr(status, i32),
        _stream(stream)))


def stats_dict(stats_tensor) -> dict:
    """Decode a moe_drop_stats_t record held in an int64 tensor of STATS_WORDS."""
    raw = bytes(stats_tensor.detach().cpu().numpy().tobytes())
    s = DropStats.from_buffer_copy(raw)
    return {f: getattr(s, f) for f, _ in DropStats._fields_}


# ---------------------------------------------------------------- whole layer

def layer_buffers(tensors: dict) -> LayerBuffers:
    """moe_layer_buffers_t from tensors named as its fields (None: NULL); the
    two sizes are taken from the scratch tensors."""
    b = LayerBuffers()
    for f in LAYER_BUFFER_FIELDS:
        if f.endswith("_bytes"):
            t = tensors.get(f[: -len("_bytes")])
            setattr(b, f, t.numel() * t.element_size() if t is not None else 0)
            continue
        t = tensors.get(f)
        if t is not None:
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{f}: contiguous device tensor required")
            setattr(b, f, t.data_ptr())
    return b


def layer_forward(cfg, buffers: LayerBuffers, x, out, stream=None):
    _check("moe_layer_forward", lib().moe_layer_forward(
        ctypes.byref(make_config(cfg)), ctypes.byref(buffers), _ptr(x, bf16), _ptr(out, bf16),
        _stream(stream)))


class HostPipe:
    """moe_host_pipe_*: batches from host memory through moe_layer_forward,
    the copies on the pipeline's own streams.  x_dev, out_dev, stats_dev:
    lists of device staging tensors (the ring)."""

    def __init__(self, cfg, x_dev, out_dev, stats_dev):
        self.cfg = make_config(cfg)
        n = len(x_dev)
        arr = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts])
        self._keep = (x_dev, out_dev, stats_dev)
        self.h = ctypes.c_void_p()
        _check("moe_host_pipe_create", lib().moe_host_pipe_create(
            ctypes.byref(self.cfg), n, arr(x_dev), arr(out_dev), arr(stats_dev),
            ctypes.byref(self.h)))

    def submit(self, buffers: LayerBuffers, x_host, out_host, stats_host=None, stream=None):
        for t in (x_host, out_host) + ((stats_host,) if stats_host is not None else ()):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("host tensors required (pinned for overlap)")
        _check("moe_host_pipe_submit", lib().moe_host_pipe_submit(
            self.h, ctypes.byref(buffers), ctypes.c_void_p(x_host.data_ptr()),
            ctypes.c_void_p(out_host.data_ptr()),
            ctypes.c_void_p(stats_host.data_ptr()) if stats_host is not None else None,
            _stream(stream)))

    def synchronize(self):
        _check("moe_host_pipe_sync", lib().moe_host_pipe_sync(self.h))

    def close(self):
        if self.h:
            rc = lib().moe_host_pipe_destroy(self.h)
            self.h = ctypes.c_void_p()
            _check("moe_host_pipe_destroy", rc)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------- timing trace

def trace_begin(n: int):
    _check("moe_trace_begin", lib().moe_trace_begin(n))


def trace_mark(stream=None):
    _check("moe_trace_mark", lib().moe_trace_mark(_stream(stream)))


def trace_end() -> list:
    """Stop tracing; return [(kernel name, ms since the previous event)]."""
    n = lib().moe_trace_end()
    out = []
    name = ctypes.c_char_p()
    ms = ctypes.c_float()
    for i in range(n):
        _check("moe_trace_event", lib().moe_trace_event(i, ctypes.byref(name), ctypes.byref(ms)))
        out.append((name.value.decode(), float(ms.value)))
    return out


# ---------------------------------------------------------------- backward pass

def backward_plan(cfg, ragged=False) -> BackwardWs:
    w = BackwardWs()
    fn = "moe_backward_plan_ragged" if ragged else "moe_backward_plan"
    _check(fn, getattr(lib(), fn)(ctypes.byref(make_config(cfg)), ctypes.byref(w)))
    return w


def layer_backward(cfg, tensors: dict, ws, status, stream=None):
    """tensors: every BackwardArgs field by name (torch tensors, or None for
    the shared-expert ones when there are none)."""
    args = BackwardArgs()
    for f in BWD_ARG_FIELDS:
        t = tensors.get(f)
        setattr(args, f, None if t is None else t.data_ptr())
    args.ws = ws.data_ptr()
    args.ws_bytes = ws.numel()
    args.status = status.data_ptr()
    eoff = tensors.get("expert_offsets")
    args.expert_offsets = None if eoff is None else eoff.data_ptr()
    bank = tensors.get("bank")
    args.bank = None if bank is None else bank.data_ptr()
    fn = "moe_layer_backward" if eoff is None else "moe_layer_backward_ragged"
    _check(fn, getattr(lib(), fn)(ctypes.byref(make_config(cfg)), ctypes.byref(args),
                                  _stream(stream)))
