"""Seeded synthetic workloads for the pooled-wave MoE layer.

This module only *draws inputs*: layer sizes, seeds and random tensors.  It
holds none of the layer's arithmetic (no capacities, routing, dispatch or
expert maths), so the CUDA library and the CPU oracle can both take their
inputs from it without sharing any of the method's code.

Recipe (one generator per tensor, seeded from the config seed and the
tensor's name):

* token states ``x``: i.i.d. N(0, 1), or, for the long-context workload, an
  AR(1) process along the sequence, ``x_t = rho x_{t-1} + sqrt(1-rho^2) e_t``
  with ``x_0 = e_0`` (stationary, unit variance per feature);
* every weight ``W ~ N(0, 1/fan_in)``;
* router bias: none, or for the skewed workload ``bias_e = log p_e`` with
  ``p_e`` proportional to ``(e+1)^-alpha`` (a Zipf prior over the experts in
  index order, so hot experts sit on the low destination ranks);
* all tensors are rounded once to bfloat16 (the bias stays float32).

Layouts (row-major, weights stored out-features-major like ``nn.Linear``):
``x [T,d]``, ``Wr [E,d]``, ``bias [E]``, ``W_ld [L,d]``, ``Wg, Wu [E,H,L]``,
``Wd [E,L,H]``, ``W_lu [d,L]``, ``Wsg, Wsu [n_s,Hs,d]``, ``Wsd [n_s,d,Hs]``.

The pages run the layer on Marin's trained weights and training text, neither
of which is available; these draws stand in for them.
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class LayerConfig:
    """Sizes of one MoE layer (notation of the pooled-wave design).

    T tokens, model width d, latent width L, E routed experts on n_ranks
    logical ranks (S = D = n_ranks), top-k routing, W waves, n_s shared
    experts; H / Hs are the routed / shared SwiGLU hidden sizes; cf_send and
    cf_recv are the sender and receiver capacity factors.
    """

    name: str
    T: int
    d_model: int
    d_latent: int
    n_experts: int
    n_ranks: int
    top_k: int
    n_waves: int
    n_shared: int
    h_expert: int
    h_shared: int
    cf_send: float = 1.10
    cf_recv: float = 1.15
    seed: int = 0
    x_kind: str = "normal"      # "normal" | "ar1"
    ar_rho: float = 0.9
    bias_kind: str = "none"     # "none" | "zipf"
    zipf_alpha: float = 1.2
    n_seqs: int = 1             # sequences the T tokens come from (descriptive)

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


# The five workloads: the tiny case, the 2x4096 mid layer, the full-width
# 535B-A23B layer (384 experts, top-8, 64 ranks), the Zipf-skewed variant and
# the 65536-token single-sequence AR(1) variant.
TINY = LayerConfig("tiny", T=256, d_model=128, d_latent=64, n_experts=24, n_ranks=4,
                   top_k=2, n_waves=3, n_shared=1, h_expert=128, h_shared=128, seed=0)
MID = LayerConfig("mid", T=8192, d_model=2048, d_latent=1024, n_experts=48, n_ranks=8,
                  top_k=8, n_waves=3, n_shared=2, h_expert=1024, h_shared=1024, seed=1,
                  n_seqs=2)
FULL = LayerConfig("full", T=16384, d_model=6144, d_latent=3072, n_experts=384, n_ranks=64,
                   top_k=8, n_waves=3, n_shared=2, h_expert=1024, h_shared=2048, seed=2,
                   n_seqs=4)
SKEW = FULL.with_(name="skew", bias_kind="zipf")
LONG = FULL.with_(name="long", T=65536, seed=3, x_kind="ar1", n_seqs=1)

# The full-width layer's per-expert shapes (d=6144, L=3072, H=1024, top-8,
# 6 experts a rank, about 340 received rows per expert) on 96 experts and 16
# ranks with T=4096: the expert GEMMs run in the same regime on a few GB of
# device memory, small enough for multi-pass profiler captures.
SLICE = FULL.with_(name="full_slice", T=4096, n_experts=96, n_ranks=16, seed=4, n_seqs=1)

# The full layer's routing (T=16384, 384 experts on 64 ranks, top-8, three
# waves, the same capacity factors) at narrow widths (d=512, L=256, H=128):
# the router top-k, dispatch and combine kernels see the full routing's
# shapes and launch sizes on a few hundred MB of device memory.
ROUTE_SLICE = FULL.with_(name="route_slice", d_model=512, d_latent=256, h_expert=128,
                         h_shared=128, seed=5)

CONFIGS = {c.name: c for c in (TINY, MID, FULL, SKEW, LONG, SLICE, ROUTE_SLICE)}

# Inputs with fewer elements than this are drawn on the host (so CPU-only and
# GPU test runs see identical values); larger ones are drawn on the target
# device by torch's own generator.
HOST_DRAW_LIMIT = 400_000_000


def _tensor_seed(seed: int, name: str) -> int:
    return (seed * 1_000_003 + zlib.crc32(name.encode())) % (2**63 - 1)


def _gen(device: torch.device, seed: int, name: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_tensor_seed(seed, name))
    return g


def input_numel(cfg: LayerConfig) -> int:
    T, d, L, E, H = cfg.T, cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.h_expert
    ns, Hs = cfg.n_shared, cfg.h_shared
    return T * d + E * d + L * d + 3 * E * H * L + d * L + 3 * ns * Hs * d


def draw_device(cfg: LayerConfig, device) -> torch.device:
    device = torch.device(device)
    if device.type == "cpu" or input_numel(cfg) < HOST_DRAW_LIMIT:
        return torch.device("cpu")
    return device


def _normal_bf16(shape, std: float, g: torch.Generator, dev: torch.device,
                 chunk_dim0: int | None = None) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    n0 = shape[0]
    step = max(1, n0 if chunk_dim0 is None else chunk_dim0)
    for a in range(0, n0, step):
        b = min(n0, a + step)
        blk = torch.randn((b - a,) + tuple(shape[1:]), generator=g, device=dev,
                          dtype=torch.float32)
        out[a:b] = (blk * std).to(torch.bfloat16)
    return out


def _ar1_bf16(T: int, d: int, rho: float, g: torch.Generator, dev: torch.device,
              block: int = 256) -> torch.Tensor:
    """AR(1) draws along the token axis, blocked: within a block of B steps,
    x_blk = M @ e_blk + rho^(1..B) x_prev, with M[i,j] = rho^(i-j) c_j."""
    c = math.sqrt(1.0 - rho * rho)
    out = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    i = torch.arange(block, device=dev, dtype=torch.float64)
    expo = (i[:, None] - i[None, :]).clamp(min=0)
    M = torch.where(i[:, None] >= i[None, :], rho ** expo, torch.zeros((), dtype=torch.float64,
                                                                        device=dev))
    Mc = (M * c).to(torch.float32)
    carry_w = (rho ** (i + 1)).to(torch.float32)[:, None]
    prev = None
    for a in range(0, T, block):
        b = min(T, a + block)
        n = b - a
        e = torch.randn((n, d), generator=g, device=dev, dtype=torch.float32)
        if prev is None:
            Mb = Mc[:n, :n].clone()
            Mb[:, 0] = (rho ** i[:n]).to(torch.float32)   # x_0 = e_0: unit variance from the start
            xb = Mb @ e
        else:
            xb = Mc[:n, :n] @ e + carry_w[:n] * prev[None, :]
        prev = xb[-1].clone()
        out[a:b] = xb.to(torch.bfloat16)
    return out


def zipf_bias(n_experts: int, alpha: float) -> torch.Tensor:
    e = torch.arange(1, n_experts + 1, dtype=torch.float64)
    p = e.pow(-alpha)
    p = p / p.sum()
    return p.log().to(torch.float32)


def make_inputs(cfg: LayerConfig, device="cpu") -> dict:
    """Draw every input of one layer call; tensors end up on ``device``."""
    device = torch.device(device)
    dev = draw_device(cfg, device)
    T, d, L, E, H = cfg.T, cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.h_expert
    ns, Hs = cfg.n_shared, cfg.h_shared
    s = cfg.seed
    t = {}
    if cfg.x_kind == "ar1":
        t["x"] = _ar1_bf16(T, d, cfg.ar_rho, _gen(dev, s, "x"), dev)
    else:
        t["x"] = _normal_bf16((T, d), 1.0, _gen(dev, s, "x"), dev, chunk_dim0=4096)
    t["Wr"] = _normal_bf16((E, d), d ** -0.5, _gen(dev, s, "Wr"), dev)
    t["bias"] = zipf_bias(E, cfg.zipf_alpha).to(dev) if cfg.bias_kind == "zipf" else None
    t["W_ld"] = _normal_bf16((L, d), d ** -0.5, _gen(dev, s, "W_ld"), dev)
    t["Wg"] = _normal_bf16((E, H, L), L ** -0.5, _gen(dev, s, "Wg"), dev, chunk_dim0=32)
    t["Wu"] = _normal_bf16((E, H, L), L ** -0.5, _gen(dev, s, "Wu"), dev, chunk_dim0=32)
    t["Wd"] = _normal_bf16((E, L, H), H ** -0.5, _gen(dev, s, "Wd"), dev, chunk_dim0=32)
    t["W_lu"] = _normal_bf16((d, L), L ** -0.5, _gen(dev, s, "W_lu"), dev)
    t["Wsg"] = _normal_bf16((ns, Hs, d), d ** -0.5, _gen(dev, s, "Wsg"), dev)
    t["Wsu"] = _normal_bf16((ns, Hs, d), d ** -0.5, _gen(dev, s, "Wsu"), dev)
    t["Wsd"] = _normal_bf16((ns, d, Hs), Hs ** -0.5, _gen(dev, s, "Wsd"), dev)
    if dev != device:
        t = {k: (v.to(device) if v is not None else None) for k, v in t.items()}
    return t
