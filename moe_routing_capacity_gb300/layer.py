"""One pooled-wave MoE layer on the GPU: device buffers plus the five calls.

``PooledWaveMoE`` owns every buffer the C ABI asks the caller for (allocated
once through PyTorch's caching allocator) and runs the layer as

    moe_router_topk -> moe_latent_proj -> moe_dispatch_pooled
        -> moe_expert_ffn_grouped -> moe_combine

on one CUDA stream, with no host synchronisation, so the whole forward can be
captured in a CUDA graph.  Intermediates stay readable as attributes.
"""
from __future__ import annotations

import torch

from . import abi


class PooledWaveMoE:
    def __init__(self, cfg, weights: dict, device="cuda"):
        self.cfg = cfg
        self.plan = abi.plan(cfg)
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
        self.pool = e(p.pool_rows, L + 8, dt=torch.int16)
        self.slot_of = e(T, k, dt=torch.int32)
        self.drop = e(T, k, dt=torch.uint8)
        self.expert_rows = e(E, p.c_recv, dt=torch.int32)
        self.expert_count = e(E, dt=torch.int32)
        self.stats = torch.zeros(abi.STATS_WORDS, dtype=torch.int64, device=dev)
        self.ws_ffn = e(max(1, p.ws_ffn_bytes), dt=torch.uint8)
        self.ypool = e(p.pool_rows, L, dt=torch.bfloat16)
        self.c = e(T, L, dt=torch.bfloat16)
        self.a = e(T, max(1, cfg.n_shared * cfg.h_shared), dt=torch.bfloat16)
        self.out = e(T, d, dt=torch.bfloat16)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    # -- the five steps -------------------------------------------------
    def route(self, x, stream=None):
        abi.router_topk(self.cfg, x, self.w["Wr"], self.w.get("bias"), self.logits, self.idx,
                        self.gate_w, self.tie, self.status, stream)

    def latent(self, x, stream=None):
        abi.latent_proj(x, self.w["W_ld"], self.z, self.status, stream)

    def dispatch(self, stream=None):
        abi.dispatch_pooled(self.cfg, self.z, self.idx, self.ws_dispatch, self.pool, self.slot_of,
                            self.drop, self.expert_rows, self.expert_count, self.stats, stream)

    def experts(self, stream=None):
        abi.expert_ffn_grouped(self.cfg, self.pool, self.expert_rows, self.expert_count,
                               self.w["Wg"], self.w["Wu"], self.w["Wd"], self.ws_ffn, self.ypool,
                               self.status, stream)

    def combine(self, x, stream=None):
        abi.combine(self.cfg, self.ypool, self.slot_of, self.gate_w, self.w["W_lu"], x,
                    self.w["Wsg"], self.w["Wsu"], self.w["Wsd"], self.c,
                    self.a if self.cfg.n_shared else None, self.out, self.status, stream)

    def forward(self, x, stream=None):
        """Enqueue the whole layer on ``stream``; returns the output buffer."""
        self.route(x, stream)
        self.latent(x, stream)
        self.dispatch(stream)
        self.experts(stream)
        self.combine(x, stream)
        return self.out

    # -- views ------------------------------------------------------------
    def pool_payload(self):
        return self.pool[:, : self.cfg.d_latent].view(torch.bfloat16)

    def pool_tags(self):
        L = self.cfg.d_latent
        return self.pool[:, L:].contiguous().view(torch.int32)

    def drop_stats(self) -> dict:
        return abi.stats_dict(self.stats)
