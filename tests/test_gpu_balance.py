"""GPU parity of the quantile-balancing bias update (devpress.csdn.net,
appendix A.2): histogram counts bit-exact, bias within fp32 rounding of the
oracle's float64 value, and the bias taking effect on the next batch."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_routing_capacity_gb300 import abi
from moe_routing_capacity_gb300 import workloads as wl
from moe_routing_capacity_gb300.layer import PooledWaveMoE

from helpers import LOGIT_ATOL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("E,k,T", [(24, 2, 256), (384, 8, 16384), (48, 8, 0)])
def test_balance_update_matches_oracle(E, k, T):
    cfg = wl.TINY.with_(T=T, n_experts=E, top_k=k, n_ranks=4 if T else 4)
    g = torch.Generator().manual_seed(E + k)
    hist = torch.zeros(E, dtype=torch.int64, device="cuda")
    bias = torch.full((E,), 7.0, dtype=torch.float32, device="cuda")
    h_o = np.zeros(E, dtype=np.int64)
    for step in range(2):
        w = torch.arange(1, E + 1, dtype=torch.float64).pow(-1.0 - 0.5 * step)
        idx = (torch.multinomial(w.expand(max(T, 1), E), k, generator=g)[:T]
               .to(torch.int32).contiguous())
        abi.balance_update(cfg, idx.cuda(), hist, 3.5, bias)
        torch.cuda.synchronize()
        h_o, b_o = O.balance_update(idx.numpy(), h_o, 3.5, E)
        assert (hist.cpu().numpy() == h_o).all()
        np.testing.assert_allclose(bias.cpu().numpy(), b_o, rtol=1e-6, atol=1e-9)


def test_balance_bias_applies_from_next_batch():
    cfg = wl.TINY.with_(seed=31, T=512, n_ranks=4)
    inp = wl.make_inputs(cfg, "cpu")
    m = PooledWaveMoE(cfg, inp, "cuda", balance_alpha=5.0)
    g = torch.Generator().manual_seed(4)
    Wr = inp["Wr"].float().numpy()
    h_o = np.zeros(cfg.n_experts, dtype=np.int64)
    b_o = np.zeros(cfg.n_experts)
    for step in range(3):
        x = torch.randn(cfg.T, cfg.d_model, generator=g).to(torch.bfloat16)
        m.forward(x.cuda())
        torch.cuda.synchronize()
        # this batch was routed with the bias from the batches before it
        l_o = O.router_logits(x.float().numpy(), Wr, b_o.astype(np.float32))
        assert np.abs(m.logits.cpu().numpy() - l_o).max() <= LOGIT_ATOL
        idx_o, _, tie_o = O.router_topk(l_o, cfg.top_k)
        assert (m.idx.cpu().numpy() == idx_o).all()      # no near-ties at these seeds
        h_o, b_o = O.balance_update(idx_o, h_o, 5.0, cfg.n_experts)
        assert (m.hist.cpu().numpy() == h_o).all()
        np.testing.assert_allclose(m.w["bias"].cpu().numpy(), b_o, rtol=1e-6, atol=1e-9)


def test_balance_bias_evens_skewed_routing():
    """Token states leaning towards a few experts' router rows: with the
    balancing bias fed back, selections spread out over the next batches."""
    cfg = wl.TINY.with_(seed=32, T=1024, n_ranks=4, top_k=2)
    inp = wl.make_inputs(cfg, "cpu")
    lean = inp["Wr"][:3].float().sum(0)
    lean = lean / lean.norm()
    g = torch.Generator().manual_seed(8)
    xs = [(torch.randn(cfg.T, cfg.d_model, generator=g) + 2.5 * lean).to(torch.bfloat16)
          for _ in range(8)]

    def imbalance(alpha):
        m = PooledWaveMoE(cfg, inp, "cuda", balance_alpha=alpha)
        for x in xs:
            m.forward(x.cuda())
        counts = torch.bincount(m.idx.flatten().long(), minlength=cfg.n_experts).float()
        torch.cuda.synchronize()
        return float(counts.max() / counts.mean()), m.drop_stats()

    base, st0 = imbalance(0.0)
    bal, st1 = imbalance(20.0)
    assert base > 2.0            # the lean really skews the routing
    assert bal < 0.75 * base
    assert st1["dropped_send"] + st1["dropped_recv"] < st0["dropped_send"] + st0["dropped_recv"]


@pytest.mark.parametrize("E,k,T,window", [(24, 2, 256, 1), (24, 2, 256, 3), (384, 8, 16384, 2),
                                          (48, 8, 0, 2)])
def test_balance_window_matches_oracle(E, k, T, window):
    """H over exactly the past `window` batches: counts bit-exact over more
    batches than the window holds, bias within fp32 rounding."""
    cfg = wl.TINY.with_(T=T, n_experts=E, top_k=k, n_ranks=4)
    g = torch.Generator().manual_seed(E + k + window)
    hist = torch.zeros(E, dtype=torch.int64, device="cuda")
    ring = torch.zeros(window, E, dtype=torch.int64, device="cuda")
    step = torch.zeros(1, dtype=torch.int64, device="cuda")
    bias = torch.full((E,), 7.0, dtype=torch.float32, device="cuda")
    h_o = np.zeros(E, dtype=np.int64)
    r_o = np.zeros((window, E), dtype=np.int64)
    s_o = 0
    for b in range(window + 3):
        w = torch.arange(1, E + 1, dtype=torch.float64).pow(-0.5 - 0.3 * (b % 3))
        idx = (torch.multinomial(w.expand(max(T, 1), E), k, generator=g)[:T]
               .to(torch.int32).contiguous())
        abi.balance_update_window(cfg, idx.cuda(), hist, ring, step, 2.5, bias)
        torch.cuda.synchronize()
        h_o, r_o, s_o, b_o = O.balance_update_window(idx.numpy(), h_o, r_o, s_o, 2.5, E)
        assert (hist.cpu().numpy() == h_o).all(), b
        assert (ring.cpu().numpy() == r_o).all(), b
        assert int(step.item()) == s_o
        np.testing.assert_allclose(bias.cpu().numpy(), b_o, rtol=1e-6, atol=1e-9)


def test_balance_window_in_the_layer():
    """The layer with a window of 2 batches: each batch is routed with the
    bias from the two batches before it."""
    cfg = wl.TINY.with_(seed=33, T=512, n_ranks=4)
    inp = wl.make_inputs(cfg, "cpu")
    m = PooledWaveMoE(cfg, inp, "cuda", balance_alpha=5.0, balance_window=2)
    g = torch.Generator().manual_seed(6)
    Wr = inp["Wr"].float().numpy()
    E = cfg.n_experts
    h_o, r_o, s_o, b_o = np.zeros(E, dtype=np.int64), np.zeros((2, E), dtype=np.int64), 0, np.zeros(E)
    for step in range(4):
        x = torch.randn(cfg.T, cfg.d_model, generator=g).to(torch.bfloat16)
        m.forward(x.cuda())
        torch.cuda.synchronize()
        l_o = O.router_logits(x.float().numpy(), Wr, b_o.astype(np.float32))
        assert np.abs(m.logits.cpu().numpy() - l_o).max() <= LOGIT_ATOL
        idx_o, _, _ = O.router_topk(l_o, cfg.top_k)
        assert (m.idx.cpu().numpy() == idx_o).all()      # no near-ties at these seeds
        h_o, r_o, s_o, b_o = O.balance_update_window(idx_o, h_o, r_o, s_o, 5.0, E)
        assert (m.hist.cpu().numpy() == h_o).all()
        np.testing.assert_allclose(m.w["bias"].cpu().numpy(), b_o, rtol=1e-6, atol=1e-9)
