"""One pooled-wave MoE layer on the GPU: device buffers plus the five calls.

``PooledWaveMoE`` owns every buffer the C ABI asks the caller for (allocated
once through PyTorch's caching allocator) and runs the layer as

    moe_route_project (= moe_router_topk + moe_latent_proj in one pass over x)
        -> moe_dispatch_pooled -> moe_expert_ffn_grouped -> moe_combine

(``pipeline="waves"``: the middle two are the single wave-pipelined call
moe_dispatch_expert_waves; ``pipeline="shared"``: moe_dispatch_shared_overlap
copies the pool rows while the shared experts' gate/up runs, then
moe_expert_ffn_grouped and moe_combine with the shared activations given,
moe_dispatch_ragged_shared_overlap likewise for the dropless layout; same
results either way)

on one CUDA stream, with no host synchronisation, so the whole forward can be
captured in a CUDA graph.  Intermediates stay readable as attributes.
"""
from __future__ import annotations

import torch

from . import abi


class PooledWaveMoE:
    """``balance_alpha``: if set, after each batch's routing the
    quantile-balancing bias is recomputed from the running selection
    histogram (``self.hist``) into the router bias, so it applies from the
    next batch on; with ``balance_window`` = N the histogram spans exactly
    the past N batches.  ``pipeline``: None (the calls one after another),
    "waves" (dispatch and experts as one wave-pipelined call: the later
    waves' pool rows copied while wave 0's experts run; capped layout only)
    or "shared" (the pool rows copied while the shared experts' gate/up
    runs; either layout).  ``expert_bank``: the dispatch also writes the received
    rows grouped by expert (``self.bank``: [E, c_recv, L] capped, [T*k, L]
    dropless in the flat row list's order), from which the expert products
    load whole tiles (either layout, except the "waves" pipeline); False
    gathers each expert's rows from the pool instead."""

    PIPELINES = (None, "waves", "shared")

    def __init__(self, cfg, weights: dict, device="cuda", balance_alpha=None,
                 dropless=False, pipeline=None, balance_window=None, expert_bank=True):
        self.cfg = cfg
        self.dropless = dropless
        if pipeline not in self.PIPELINES:
            raise ValueError(f"pipeline must be one of {self.PIPELINES}")
        if pipeline == "waves" and dropless:
            raise ValueError("the wave pipeline is built for the capped layout")
        self.pipeline = pipeline
        self.plan = abi.plan_ragged(cfg) if dropless else abi.plan(cfg)
        self.device = torch.device(device)
        dev = self.device
        T, d, L, E, k = cfg.T, cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.top_k
        p = self.plan
        self.w = {n: (t.to(dev).contiguous() if t is not None else None)
                  for n, t in weights.items() if n != "x"}
        e = lambda *s, dt: torch.empty(s, dtype=dt, device=dev)
        self.logits = e(T, E, dt=torch.float32)
        self.idx = e(T, k, dt=torch.int32)
        self.gate_w = e(T, k, dt=torch.float32)
        self.tie = e(T, dt=torch.uint8)
        self.z = e(T, L, dt=torch.bfloat16)
        self.ws_dispatch = e(max(1, p.ws_dispatch_bytes), dt=torch.uint8)
        self.pool = e(p.pool_rows, p.pool_row_bytes // 2, dt=torch.int16)
        self.slot_of = e(T, k, dt=torch.int32)
        self.drop = e(T, k, dt=torch.uint8)
        if dropless:    # flat row list with per-expert offsets
            self.expert_rows = e(T * k, dt=torch.int32)
            self.expert_offsets = e(E + 1, dt=torch.int32)
        else:
            self.expert_rows = e(E, p.c_recv, dt=torch.int32)
        self.expert_count = e(E, dt=torch.int32)
        self.stats = torch.zeros(abi.STATS_WORDS, dtype=torch.int64, device=dev)
        self.ws_ffn = e(max(1, p.ws_ffn_bytes), dt=torch.uint8)
        # the received rows grouped by local expert (written by the pack)
        if not expert_bank or pipeline == "waves":
            self.bank = None
        elif dropless:
            self.bank = e(max(1, T * k), L, dt=torch.bfloat16)
        else:
            self.bank = e(E, max(1, p.c_recv), L, dt=torch.bfloat16)
        self.ypool = e(p.pool_rows, L, dt=torch.bfloat16)
        self.c = e(T, L, dt=torch.bfloat16)
        self.a = e(T, max(1, cfg.n_shared * cfg.h_shared), dt=torch.bfloat16)
        self.out = e(T, d, dt=torch.bfloat16)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.balance_alpha = balance_alpha
        self.balance_window = balance_window
        if balance_alpha is not None:
            if self.w.get("bias") is None:
                self.w["bias"] = torch.zeros(E, dtype=torch.float32, device=dev)
            self.hist = torch.zeros(E, dtype=torch.int64, device=dev)
            if balance_window:   # exact window of the past N batches
                self.ring = torch.zeros(balance_window, E, dtype=torch.int64, device=dev)
                self.bstep = torch.zeros(1, dtype=torch.int64, device=dev)

    # -- the five steps -------------------------------------------------
    def route(self, x, stream=None):
        abi.router_topk(self.cfg, x, self.w["Wr"], self.w.get("bias"), self.logits, self.idx,
                        self.gate_w, self.tie, self.status, stream)

    def latent(self, x, stream=None):
        abi.latent_proj(x, self.w["W_ld"], self.z, self.status, stream)

    def dispatch(self, stream=None):
        if self.dropless:
            abi.dispatch_ragged(self.cfg, self.z, self.idx, self.ws_dispatch, self.pool,
                                self.slot_of, self.drop, self.expert_offsets, self.expert_rows,
                                self.expert_count, self.stats, stream, bank=self.bank)
        else:
            abi.dispatch_pooled(self.cfg, self.z, self.idx, self.ws_dispatch, self.pool,
                                self.slot_of, self.drop, self.expert_rows, self.expert_count,
                                self.stats, stream, bank=self.bank)

    def experts(self, stream=None):
        if self.dropless:
            abi.expert_ffn_ragged(self.cfg, self.pool, self.expert_offsets, self.expert_rows,
                                  self.expert_count, self.w["Wg"], self.w["Wu"], self.w["Wd"],
                                  self.ws_ffn, self.ypool, self.status, stream, bank=self.bank)
        else:
            abi.expert_ffn_grouped(self.cfg, self.pool, self.expert_rows, self.expert_count,
                                   self.w["Wg"], self.w["Wu"], self.w["Wd"], self.ws_ffn,
                                   self.ypool, self.status, stream, bank=self.bank)

    def combine(self, x, out=None, stream=None):
        abi.combine(self.cfg, self.ypool, self.slot_of, self.gate_w, self.w["W_lu"], x,
                    self.w["Wsg"], self.w["Wsu"], self.w["Wsd"], self.c,
                    self.a if self.cfg.n_shared else None,
                    self.out if out is None else out, self.status, stream)

    def route_and_latent(self, x, stream=None):
        """Router top-k and latent projection in one pass over x."""
        abi.route_project(self.cfg, x, self.w["Wr"], self.w.get("bias"), self.w["W_ld"],
                          self.logits, self.idx, self.gate_w, self.tie, self.z, self.status,
                          stream)

    def forward(self, x, out=None, stream=None):
        """Enqueue the whole layer on ``stream``; returns the output tensor
        (``out`` if given, else the layer's own output buffer)."""
        self.route_and_latent(x, stream)
        if self.balance_alpha is not None and self.balance_window:
            abi.balance_update_window(self.cfg, self.idx, self.hist, self.ring, self.bstep,
                                      self.balance_alpha, self.w["bias"], stream)
        elif self.balance_alpha is not None:
            abi.balance_update(self.cfg, self.idx, self.hist, self.balance_alpha,
                               self.w["bias"], stream)
        if self.pipeline == "waves":
            abi.dispatch_expert_waves(self.cfg, self.z, self.idx, self.ws_dispatch, self.pool,
                                      self.slot_of, self.drop, self.expert_rows,
                                      self.expert_count, self.stats, self.w["Wg"], self.w["Wu"],
                                      self.w["Wd"], self.ws_ffn, self.ypool, self.status, stream)
            self.combine(x, out, stream)
        elif self.pipeline == "shared" and self.cfg.n_shared:
            if self.dropless:
                abi.dispatch_ragged_shared_overlap(
                    self.cfg, self.z, self.idx, self.ws_dispatch, self.pool, self.slot_of,
                    self.drop, self.expert_offsets, self.expert_rows, self.expert_count,
                    self.stats, x, self.w["Wsg"], self.w["Wsu"], self.a, self.status, stream,
                    bank=self.bank)
            else:
                abi.dispatch_shared_overlap(self.cfg, self.z, self.idx, self.ws_dispatch,
                                            self.pool, self.slot_of, self.drop, self.expert_rows,
                                            self.expert_count, self.stats, x, self.w["Wsg"],
                                            self.w["Wsu"], self.a, self.status, stream,
                                            bank=self.bank)
            self.experts(stream)
            abi.combine(self.cfg, self.ypool, self.slot_of, self.gate_w, self.w["W_lu"], None,
                        None, None, self.w["Wsd"], self.c, self.a,
                        self.out if out is None else out, self.status, stream)
        else:
            self.dispatch(stream)
            self.experts(stream)
            self.combine(x, out, stream)
        return self.out if out is None else out

    def capture(self, x, out=None):
        """Record one forward on ``x`` (into ``out`` if given) as a CUDA graph.

        Every step of the layer is a kernel launch or an async memset on the
        stream, with no host synchronisation and no allocation, so the whole
        forward replays from the graph: ``g.replay()`` runs it again on
        whatever ``x`` then holds.  Two eager forwards run first (outside the
        capture) so that one-time launch attributes are already set."""
        dev = self.device
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for _ in range(2):
                self.forward(x, out)
        torch.cuda.current_stream(dev).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.forward(x, out)
        return g

    def backward(self, x, dout, stream=None) -> dict:
        """Gradients of the last forward with respect to x and every weight,
        for the upstream gradient dout [T, d] (capped or dropless layout).
        Returns {"x": dx (bf16), "Wr": ..., ...} with fp32 weight gradients."""
        cfg, dev = self.cfg, self.device
        T, d, L, E, H = cfg.T, cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.h_expert
        ns, Hs = cfg.n_shared, cfg.h_shared
        if not hasattr(self, "bwd_ws"):
            self.bwd_layout = abi.backward_plan(cfg, ragged=self.dropless)
            self.bwd_ws = torch.empty(max(1, self.bwd_layout.total), dtype=torch.uint8, device=dev)
            f = lambda *sh: torch.empty(sh, dtype=torch.float32, device=dev)
            self.grads = {"x": torch.empty(T, d, dtype=torch.bfloat16, device=dev),
                          "Wr": f(E, d), "W_ld": f(L, d), "Wg": f(E, H, L), "Wu": f(E, H, L),
                          "Wd": f(E, L, H), "W_lu": f(d, L), "Wsg": f(ns, Hs, d),
                          "Wsu": f(ns, Hs, d), "Wsd": f(ns, d, Hs)}
        hoff = self.plan.h_offset_bytes
        h_rows = self.plan.pool_rows if self.dropless else E * self.plan.c_recv
        h = self.ws_ffn[hoff:hoff + h_rows * H * 2].view(torch.bfloat16)
        g = self.grads
        tensors = dict(x=x, Wr=self.w["Wr"], W_ld=self.w["W_ld"], Wg=self.w["Wg"], Wu=self.w["Wu"],
                       Wd=self.w["Wd"], W_lu=self.w["W_lu"], Wsg=self.w["Wsg"], Wsu=self.w["Wsu"],
                       Wsd=self.w["Wsd"], idx=self.idx, w=self.gate_w, pool=self.pool,
                       slot_of=self.slot_of, expert_rows=self.expert_rows,
                       expert_count=self.expert_count, h=h, ypool=self.ypool, c=self.c,
                       a=self.a if ns else None, dout=dout, dx=g["x"], dWr=g["Wr"],
                       dW_ld=g["W_ld"], dWg=g["Wg"], dWu=g["Wu"], dWd=g["Wd"], dW_lu=g["W_lu"],
                       dWsg=g["Wsg"] if ns else None, dWsu=g["Wsu"] if ns else None,
                       dWsd=g["Wsd"] if ns else None,
                       expert_offsets=self.expert_offsets if self.dropless else None,
                       bank=None if self.dropless else self.bank)
        abi.layer_backward(cfg, tensors, self.bwd_ws, self.status, stream)
        return g

    def backward_intermediate(self, name):
        """A view of one backward intermediate in the scratch (tests)."""
        off = getattr(self.bwd_layout, name)
        return self.bwd_ws[off:]

    # -- views ------------------------------------------------------------
    def buffers(self):
        """The layer's weights and buffers as moe_layer_buffers_t (capped layout)."""
        if self.dropless:
            raise ValueError("moe_layer_forward runs the capped layout")
        t = {k: v for k, v in self.w.items() if v is not None and v.numel() > 0}
        t.update(logits=self.logits, idx=self.idx, w=self.gate_w, tie=self.tie, z=self.z,
                 ws_dispatch=self.ws_dispatch, pool=self.pool, slot_of=self.slot_of,
                 drop=self.drop, expert_rows=self.expert_rows, expert_count=self.expert_count,
                 stats=self.stats, bank=self.bank, ws_ffn=self.ws_ffn, ypool=self.ypool,
                 c=self.c, a=self.a if self.cfg.n_shared else None, status=self.status)
        return abi.layer_buffers(t)

    def forward_native(self, x, out=None, stream=None):
        """The whole forward as one library call (moe_layer_forward: the pool
        fill inside the shared experts' gate/up launch); same results as
        forward() with pipeline="shared"."""
        out = self.out if out is None else out
        abi.layer_forward(self.cfg, self.buffers(), x, out, stream)
        return out

    def pool_payload(self):
        return self.pool[:, : self.cfg.d_latent].view(torch.bfloat16)

    def pool_tags(self):
        L = self.cfg.d_latent
        return self.pool[:, L:L + 8].contiguous().view(torch.int32)

    def drop_stats(self) -> dict:
        return abi.stats_dict(self.stats)


class HostPipeline:
    """Runs host-resident batches through a layer with the copies overlapped,
    in the library (moe_host_pipe_*, over moe_layer_forward: the pool fill
    inside the shared experts' gate/up launch, the layer's bank if it has
    one).  Batch i's host->device copy runs on the library's own stream while
    batch i-1 computes on the caller's stream and batch i-2's output (and
    drop statistics) copy back on a second stream of the library's;
    ``depth`` device staging buffers per direction keep the three in flight.
    Host tensors should be pinned for the copies to be asynchronous.  The
    layer's balancing-bias update is not applied on this path.
    """

    def __init__(self, layer: "PooledWaveMoE", depth: int = 2):
        if layer.dropless:
            raise ValueError("the host pipeline runs the capped layout")
        self.m = layer
        self.depth = depth
        cfg, dev = layer.cfg, layer.device
        self.xd = [torch.empty(cfg.T, cfg.d_model, dtype=torch.bfloat16, device=dev)
                   for _ in range(depth)]
        self.od = [torch.empty(cfg.T, cfg.d_model, dtype=torch.bfloat16, device=dev)
                   for _ in range(depth)]
        self.sd = [torch.empty_like(layer.stats) for _ in range(depth)]
        self.buffers = layer.buffers()
        self.pipe = abi.HostPipe(cfg, self.xd, self.od, self.sd)

    def submit(self, x_host, out_host, stats_host=None, stream=None):
        """Enqueue one batch: x_host -> layer -> out_host (all asynchronous)."""
        self.pipe.submit(self.buffers, x_host, out_host, stats_host, stream)

    def synchronize(self):
        self.pipe.synchronize()

    def close(self):
        self.pipe.close()
