"""The whole-layer forward in one library call (moe_layer_forward) and the
host-memory pipeline over it (moe_host_pipe_*), through the C ABI.

moe_layer_forward must give the same bits as the same calls made one by one
(the layer object's forward with the pool fill inside the shared experts'
gate/up launch), with and without shared experts and with and without the
per-expert bank.  The pipeline must return, for each of several different
batches taken from pinned host memory, exactly that batch's output and drop
statistics, with the copies and the compute of neighbouring batches in
flight together.
"""
import pytest
import torch

from moe_routing_capacity_gb300 import workloads as wl
from moe_routing_capacity_gb300.layer import HostPipeline, PooledWaveMoE

pytestmark = pytest.mark.gpu

PAIRS = wl.LayerConfig("pairs", T=4096, d_model=256, d_latent=256, n_experts=24, n_ranks=4,
                       top_k=2, n_waves=3, n_shared=1, h_expert=128, h_shared=128, seed=5)


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("tiny_noshared", {}), ("pairs", {}),
                                     ("pairs", {"expert_bank": False}), ("mid", {})])
def test_layer_forward_equals_the_calls(name, kw):
    cfg = {"tiny": wl.TINY, "tiny_noshared": wl.TINY.with_(n_shared=0), "pairs": PAIRS,
           "mid": wl.MID}[name]
    inp = wl.make_inputs(cfg, "cuda")
    x = inp["x"]
    ref = PooledWaveMoE(cfg, inp, "cuda", pipeline="shared", **kw)
    ref.forward(x)
    m = PooledWaveMoE(cfg, inp, "cuda", pipeline="shared", **kw)
    out = torch.empty_like(ref.out)
    m.forward_native(x, out)
    torch.cuda.synchronize()
    assert int(ref.status.item()) == 0 and int(m.status.item()) == 0
    assert torch.equal(_bits(out), _bits(ref.out))
    for n in ("idx", "slot_of", "drop", "expert_rows", "expert_count", "c"):
        assert torch.equal(_bits(getattr(m, n)), _bits(getattr(ref, n))), n
    assert m.drop_stats() == ref.drop_stats()


@pytest.mark.parametrize("name", ["tiny", "pairs"])
def test_host_pipeline_returns_each_batch(name):
    cfg = {"tiny": wl.TINY, "pairs": PAIRS}[name]
    inp = wl.make_inputs(cfg, "cuda")
    m = PooledWaveMoE(cfg, inp, "cuda", pipeline="shared")
    g = torch.Generator(device="cuda").manual_seed(11)
    n = 5
    xs = [inp["x"]] + [torch.randn(cfg.T, cfg.d_model, generator=g, device="cuda").to(torch.bfloat16)
                       for _ in range(n - 1)]
    want, want_stats = [], []
    for x in xs:
        m.forward(x)
        want.append(m.out.clone())
        want_stats.append(m.stats.clone())
    torch.cuda.synchronize()
    xh = [x.cpu().pin_memory() for x in xs]
    oh = [torch.empty(cfg.T, cfg.d_model, dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    sh = [torch.empty(m.stats.numel(), dtype=torch.int64).pin_memory() for _ in range(n)]
    pipe = HostPipeline(m, depth=2)
    for i in range(n):
        pipe.submit(xh[i], oh[i], sh[i])
    pipe.synchronize()
    torch.cuda.synchronize()
    assert int(m.status.item()) == 0
    for i in range(n):
        assert torch.equal(_bits(oh[i]), _bits(want[i].cpu())), i
        assert torch.equal(sh[i], want_stats[i].cpu()), i
    pipe.close()
