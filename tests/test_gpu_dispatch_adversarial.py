"""The pooled-wave dispatch on adversarial routings, bit for bit against the
oracle: every token on the same k experts, every token on the experts of one
destination rank (or the fewest that hold k experts), one wave only, and
blocks of consecutive tokens all choosing one expert first.  The routing is
fed straight to moe_dispatch_pooled (no router), so the decisions cannot
hide behind near-ties."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_routing_capacity_gb300 import abi
from moe_routing_capacity_gb300 import workloads as wl

from helpers import dispatch_rules_hold

pytestmark = pytest.mark.gpu


def _routings(cfg, rng):
    T, k, E, D, W = cfg.T, cfg.top_k, cfg.n_experts, cfg.n_ranks, cfg.n_waves
    E_l = E // D
    E_w = E_l // W
    out = {}
    # every token on the same k experts
    out["same_k"] = np.tile(np.arange(k), (T, 1))
    # every token on the experts of destination 0 (or of the fewest leading
    # destinations that hold k experts)
    first = np.arange(-(-k // E_l) * E_l)
    out["one_dst"] = np.stack([rng.choice(first, k, replace=False) for _ in range(T)])
    # every token on the experts of wave 0 of every destination
    wave0 = np.array([d * E_l + j for d in range(D) for j in range(E_w)])
    out["one_wave"] = np.stack([rng.choice(wave0, k, replace=False) for _ in range(T)])
    # token t's first choice is the expert of its block of 64 tokens, the rest random
    blk = np.stack([np.concatenate([[(t // 64) % E],
                                    rng.choice(np.setdiff1d(np.arange(E), [(t // 64) % E]),
                                               k - 1, replace=False)]) for t in range(T)])
    out["blocked"] = blk
    return {n: v.astype(np.int32) for n, v in out.items()}


def _gpu_dispatch(cfg, idx, z):
    p = abi.plan(cfg)
    dev = "cuda"
    ws = torch.empty(max(1, p.ws_dispatch_bytes), dtype=torch.uint8, device=dev)
    o = dict(pool=torch.zeros(p.pool_rows, p.pool_row_bytes // 2, dtype=torch.int16, device=dev),
             slot_of=torch.zeros(cfg.T, cfg.top_k, dtype=torch.int32, device=dev),
             drop=torch.zeros(cfg.T, cfg.top_k, dtype=torch.uint8, device=dev),
             expert_rows=torch.zeros(cfg.n_experts, p.c_recv, dtype=torch.int32, device=dev),
             expert_count=torch.zeros(cfg.n_experts, dtype=torch.int32, device=dev),
             stats=torch.zeros(abi.STATS_WORDS, dtype=torch.int64, device=dev))
    abi.dispatch_pooled(cfg, z.cuda(), torch.from_numpy(idx).cuda(), ws, o["pool"], o["slot_of"],
                        o["drop"], o["expert_rows"], o["expert_count"], o["stats"])
    torch.cuda.synchronize()
    return {n: (t.cpu() if n != "stats" else abi.stats_dict(t)) for n, t in o.items()}


@pytest.mark.parametrize("cfg", [wl.TINY, wl.TINY.with_(seed=71, T=512, n_experts=48, n_ranks=8,
                                                          top_k=4, d_latent=128),
                                 wl.MID], ids=["tiny", "small48", "mid"])
def test_adversarial_routings_bit_exact(cfg):
    rng = np.random.default_rng(cfg.seed + 100)
    g = torch.Generator().manual_seed(cfg.seed + 100)
    z = torch.randn(cfg.T, cfg.d_latent, generator=g).to(torch.bfloat16)
    plan = O.make_plan(cfg)
    for name, idx in _routings(cfg, rng).items():
        ref = O.dispatch(idx, plan)
        got = _gpu_dispatch(cfg, idx, z)
        assert (got["slot_of"].numpy() == ref["slot_of"]).all(), name
        assert (got["drop"].numpy() == ref["drop"]).all(), name
        assert (got["expert_count"].numpy() == ref["count"]).all(), name
        assert (got["expert_rows"].numpy() == ref["expert_rows"]).all(), name
        st = got["stats"]
        assert st["status"] == 0, name
        assert (st["kept"], st["dropped_send"], st["dropped_recv"]) == (
            ref["stats"]["kept"], ref["stats"]["dropped_send"], ref["stats"]["dropped_recv"]), name
        dispatch_rules_hold(idx, got["slot_of"].numpy(), got["drop"].numpy(),
                            got["expert_rows"].numpy(), got["expert_count"].numpy(), plan)
        # payload and tag of every filled pool row
        L = cfg.d_latent
        pool = got["pool"]
        rows = np.nonzero(ref["send_row"].reshape(-1) >= 0)[0]
        payload, tags = O.pack_pool(z.float().numpy(), idx, ref, plan,
                                    rows=ref["send_row"].reshape(-1)[rows])
        gt = pool[ref["send_row"].reshape(-1)[rows], L:L + 8].contiguous().view(torch.int32).numpy()
        assert (gt == tags).all(), name
        gp = pool[ref["send_row"].reshape(-1)[rows], :L].view(torch.bfloat16).float().numpy()
        assert (gp == payload.astype(np.float32)).all(), name
        if name == "same_k":   # closed form: per expert min(sender-kept rows, c_recv)
            assert (ref["count"][:cfg.top_k] > 0).all()
