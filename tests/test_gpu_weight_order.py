"""The expert products with the up weights below the gate weights in memory.

The gate/up products read Wg and Wu through one tensor map whose outermost
dimension steps from the lower-addressed tensor to the other, and the dX
product of the backward reads its two K segments the same way; which tensor
comes first decides which TMEM lanes hold the gate rows and which map index
each segment takes.  With Wu placed below Wg (both halves of one buffer) the
forward must match the path that gathers the rows from the pool bit for bit
and the oracle, and every gradient must match the oracle's derivative and,
bit for bit, a run with the usual order.  The widths (L = 256, H = 256) take
the row-group kernels for every routed-expert product of both passes; the
experts receive 201-295 rows (one- and two-chunk groups), and no token's
routing is a near-tie, so the oracle's routing is the GPU's.
"""
import pytest
import torch

import oracle as O
from moe_routing_capacity_gb300 import workloads as wl
from moe_routing_capacity_gb300.layer import PooledWaveMoE

from helpers import check_close
from test_gpu_backward import check_grad
from test_gpu_parity import compare_full, run_gpu

pytestmark = pytest.mark.gpu

CFG = wl.LayerConfig("order", T=3072, d_model=256, d_latent=256, n_experts=24, n_ranks=4,
                     top_k=2, n_waves=3, n_shared=1, h_expert=256, h_shared=128, seed=10)


def _inputs(up_first):
    """Device inputs with Wg and Wu the two halves of one allocation: Wu the
    lower one when up_first, else Wg."""
    inp = wl.make_inputs(CFG, "cuda")
    buf = torch.empty((2,) + tuple(inp["Wg"].shape), dtype=torch.bfloat16, device="cuda")
    lo, hi = ("Wu", "Wg") if up_first else ("Wg", "Wu")
    buf[0].copy_(inp[lo])
    buf[1].copy_(inp[hi])
    inp[lo], inp[hi] = buf[0], buf[1]
    assert inp[lo].data_ptr() < inp[hi].data_ptr()
    return inp


def test_forward_with_up_weights_first():
    inp = _inputs(up_first=True)
    m, ref, rep = compare_full(CFG, inp, expert_bank=True)
    b = run_gpu(CFG, inp, expert_bank=False)
    kept = m.slot_of[m.slot_of >= 0].long()
    assert torch.equal(m.ypool[kept].view(torch.int16), b.ypool[kept].view(torch.int16))
    assert torch.equal(m.out.view(torch.int16), b.out.view(torch.int16))
    print(rep)


def _grads(inp, dout):
    m = PooledWaveMoE(CFG, inp, "cuda", pipeline="shared")
    x = inp["x"]
    m.forward(x)
    g = m.backward(x, dout)
    torch.cuda.synchronize()
    assert int(m.status.item()) == 0
    return m, {k: v.clone() for k, v in g.items()}


def test_backward_with_up_weights_first():
    dout = torch.randn(CFG.T, CFG.d_model, generator=torch.Generator().manual_seed(3)).to(
        torch.bfloat16).cuda()
    a_inp = _inputs(up_first=True)
    m, ga = _grads(a_inp, dout)
    _, gb = _grads(_inputs(up_first=False), dout)
    for k in ga:
        va, vb = ga[k], gb[k]
        w = torch.int32 if va.dtype == torch.float32 else torch.int16
        assert torch.equal(va.view(w), vb.view(w)), k
    host = {k: (v.float().cpu().numpy() if v is not None else None) for k, v in a_inp.items()}
    fwd = O.layer(CFG, host)
    assert (fwd["tie"] == 0).all() and (m.idx.cpu().numpy() == fwd["idx"]).all()
    ref = O.layer_backward(CFG, host, fwd, dout.float().cpu().numpy())
    rep = {}
    check_close("dx", ga["x"].float().cpu().numpy(), ref["x"], rep)
    for name in ("Wr", "W_ld", "Wg", "Wu", "Wd", "W_lu", "Wsg", "Wsu", "Wsd"):
        check_grad("d" + name, ga[name].cpu().numpy(), ref[name], rep)
    print(rep)
