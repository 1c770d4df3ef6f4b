"""The layer forward replayed from a CUDA graph equals the eager forward, bit
for bit, on new inputs written into the captured input buffer (every step
of the path is a stream-ordered launch; nothing in it synchronises the host
or allocates)."""
import pytest
import torch

from moe_routing_capacity_gb300 import workloads as wl
from moe_routing_capacity_gb300.layer import PooledWaveMoE

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,dropless", [("tiny", False), ("mid", False), ("mid", True)])
def test_graph_replay_equals_eager(name, dropless):
    cfg = wl.CONFIGS[name]
    inp = wl.make_inputs(cfg, "cuda")
    m = PooledWaveMoE(cfg, inp, "cuda", dropless=dropless)
    x_buf = inp["x"].clone()
    out_g = torch.empty(cfg.T, cfg.d_model, dtype=torch.bfloat16, device="cuda")
    g = m.capture(x_buf, out_g)
    gen = torch.Generator(device="cuda").manual_seed(11)
    for step in range(3):
        x_new = torch.randn(cfg.T, cfg.d_model, generator=gen, device="cuda").to(torch.bfloat16)
        x_buf.copy_(x_new)
        g.replay()
        torch.cuda.synchronize()
        got = out_g.clone()
        stats_g = m.drop_stats()
        want = m.forward(x_new).clone()
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), step
        assert stats_g == m.drop_stats()
        assert int(m.status.item()) == 0
