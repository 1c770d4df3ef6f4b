"""The allocation-free dispatch entry point against the regular one.

``moe_dispatch_pooled_noalloc`` serves callers that cannot allocate device
memory (a host application that reserved the device's memory up front, a
latency-critical path that cannot afford an allocation's synchronisation, a
plug-in handed tensors but no allocator): it keeps the dispatch scratch in a
fixed array inside the library.  Its results must equal those of
``moe_dispatch_pooled`` with caller-provided scratch, bit for bit (integer
and copy work), on two calls in a row with different routings, so that
nothing left in the shared array from one call leaks into the next.

This file is named to be collected last.
"""
import pytest
import torch

from moe_routing_capacity_gb300 import abi
from moe_routing_capacity_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _routing(cfg, seed, skew):
    g = torch.Generator().manual_seed(seed)
    E, k = cfg.n_experts, cfg.top_k
    if skew:
        w = torch.arange(1, E + 1, dtype=torch.float64).pow(-1.2)
    else:
        w = torch.ones(E, dtype=torch.float64)
    idx = torch.multinomial(w.expand(cfg.T, E), k, replacement=False, generator=g)
    z = torch.randn(cfg.T, cfg.d_latent, generator=g).to(torch.bfloat16)
    return idx.to(torch.int32).cuda(), z.cuda()


def _outputs(cfg):
    p = abi.plan(cfg)
    dev = "cuda"
    return dict(
        pool=torch.zeros(p.pool_rows, p.pool_row_bytes // 2, dtype=torch.int16, device=dev),
        slot_of=torch.zeros(cfg.T, cfg.top_k, dtype=torch.int32, device=dev),
        drop=torch.zeros(cfg.T, cfg.top_k, dtype=torch.uint8, device=dev),
        expert_rows=torch.zeros(cfg.n_experts, p.c_recv, dtype=torch.int32, device=dev),
        expert_count=torch.zeros(cfg.n_experts, dtype=torch.int32, device=dev),
        stats=torch.zeros(abi.STATS_WORDS, dtype=torch.int64, device=dev),
    )


def _same(a, b, L):
    for key in ("slot_of", "drop", "expert_rows", "expert_count", "stats"):
        assert torch.equal(a[key], b[key]), key
    tags_a = a["pool"][:, L:L + 8]
    assert torch.equal(tags_a, b["pool"][:, L:L + 8])
    filled = tags_a.contiguous().view(torch.int32)[:, 0] >= 0
    assert torch.equal(a["pool"][filled, :L], b["pool"][filled, :L])


@pytest.mark.parametrize("name", ["mid", "full"])
def test_noalloc_dispatch_equals_dispatch_twice(name):
    cfg = wl.CONFIGS[name]
    p = abi.plan(cfg)
    assert p.ws_dispatch_bytes <= abi.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(p.ws_dispatch_bytes, dtype=torch.uint8, device="cuda")
    for call, (seed, skew) in enumerate(((1, False), (2, True))):
        idx, z = _routing(cfg, seed, skew)
        want = _outputs(cfg)
        abi.dispatch_pooled(cfg, z, idx, ws, want["pool"], want["slot_of"], want["drop"],
                            want["expert_rows"], want["expert_count"], want["stats"])
        got = _outputs(cfg)
        abi.dispatch_pooled_noalloc(cfg, z, idx, got["pool"], got["slot_of"], got["drop"],
                                    got["expert_rows"], got["expert_count"], got["stats"])
        torch.cuda.synchronize()
        _same(got, want, cfg.d_latent)
        st = abi.stats_dict(got["stats"])
        assert st["status"] == 0 and st["assignments"] == cfg.T * cfg.top_k
        if skew:
            assert st["dropped_send"] + st["dropped_recv"] > 0


def test_noalloc_dispatch_rejects_oversized_config():
    cfg = wl.FULL.with_(T=16384 * 8)        # 1M assignments: ~12.8 MB of scratch
    assert abi.plan(cfg).ws_dispatch_bytes > abi.NOALLOC_SCRATCH_BYTES
    import ctypes
    rc = abi.lib().moe_dispatch_pooled_noalloc(ctypes.byref(abi.make_config(cfg)), None, None,
                                               None, None, None, None, None, None, None)
    assert rc == abi.MOE_ENOSPC
