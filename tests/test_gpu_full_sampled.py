"""Full-size parity: the full-width layer (384 experts, top-8, 64 logical
ranks, d=6144, L=3072), its Zipf-skewed variant and the 65536-token AR(1)
long-context variant, run exactly as the benchmark runs them.

The oracle recomputes the routing and the whole dispatch for every token
(integer results compared bit-exactly, near-ties excepted) and the floating-
point path for a sample of tokens, one by one.  Properties that hold at any
size (caps, conservation, the pack being a copy) are checked on everything.
Inputs are drawn on the device by torch's seeded generator; the oracle gets
host copies of those inputs, never a value the library computed.
"""
import numpy as np
import pytest
import torch

import oracle as O
from moe_routing_capacity_gb300 import workloads as wl
from moe_routing_capacity_gb300.layer import PooledWaveMoE

from helpers import LOGIT_ATOL, check_close, dispatch_rules_hold, tie_margin_ok

pytestmark = pytest.mark.gpu

N_SAMPLE = 24


def _f64(t):
    return t.detach().double().cpu().numpy()


def _sample_tokens(T, n, seed):
    rng = np.random.default_rng(seed)
    pick = set([0, T - 1]) | set(rng.choice(T, n - 2, replace=False).tolist())
    return np.array(sorted(pick))


@pytest.mark.parametrize("name", ["full", "skew", "long"])
def test_full_size_sampled(name):
    cfg = wl.CONFIGS[name]
    inp = wl.make_inputs(cfg, "cuda")
    m = PooledWaveMoE(cfg, inp, "cuda")
    x = inp["x"]
    m.forward(x)
    torch.cuda.synchronize()
    assert int(m.status.item()) == 0
    st = m.drop_stats()
    assert st["status"] == 0
    p = O.make_plan(cfg)
    T, k, L = cfg.T, cfg.top_k, cfg.d_latent

    # ---- routing for every token
    xh = _f64(x)
    bias = inp["bias"].cpu().numpy() if inp["bias"] is not None else None
    l32 = O.router_logits(xh, _f64(inp["Wr"]), bias)
    idx_o, w_o, tie_o = O.router_topk(l32, k)
    lg = m.logits.cpu().numpy()
    assert np.abs(lg.astype(np.float64) - l32).max() <= LOGIT_ATOL
    idx = m.idx.cpu().numpy()
    clear = tie_o == 0
    assert (idx[clear] == idx_o[clear]).all()
    lerr = float(np.abs(lg.astype(np.float64) - l32).max())
    stable = tie_margin_ok(l32, k, idx_o, 2 * lerr + 1e-7)
    assert (m.tie.cpu().numpy()[stable] == tie_o[stable]).all()

    # ---- dispatch for every assignment
    d = O.dispatch(idx_o, p)
    slot_of, drop = m.slot_of.cpu().numpy(), m.drop.cpu().numpy()
    rows, count = m.expert_rows.cpu().numpy(), m.expert_count.cpu().numpy()
    flips = np.nonzero((idx != idx_o).any(axis=1))[0]
    if flips.size == 0:
        assert (slot_of == d["slot_of"]).all() and (drop == d["drop"]).all()
        assert (rows == d["expert_rows"]).all() and (count == d["count"]).all()
        for key in ("kept", "dropped_send", "dropped_recv"):
            assert st[key] == d["stats"][key]
    else:
        t0 = int(flips[0])
        assert (slot_of[:t0] == d["slot_of"][:t0]).all() and (drop[:t0] == d["drop"][:t0]).all()
        dispatch_rules_hold(idx, slot_of, drop, rows, count, p)
    assert st["kept"] + st["dropped_send"] + st["dropped_recv"] == T * k
    assert st["max_send_fill"] <= p.c_send and st["max_expert_rows"] <= p.c_recv

    # ---- properties of the pool at full size (checked on the device)
    tags = m.pool_tags()
    filled = tags[:, 0] >= 0
    assert int(filled.sum()) == st["kept"] + st["dropped_recv"]
    tok = tags[filled, 1].long()
    assert torch.equal(m.pool_payload()[filled], m.z[tok])
    e_tag = tags[filled, 0]
    assert bool((m.idx[tok, tags[filled, 2].long()] == e_tag).all())

    # ---- floating point on sampled tokens, one by one
    W_ld = _f64(inp["W_ld"])
    W_lu = _f64(inp["W_lu"])
    Wsg, Wsu, Wsd = _f64(inp["Wsg"]), _f64(inp["Wsu"]), _f64(inp["Wsd"])
    same = (idx == idx_o).all(axis=1) & (drop == d["drop"]).all(axis=1)
    toks = [t for t in _sample_tokens(T, N_SAMPLE, cfg.seed) if same[t]]
    assert len(toks) >= N_SAMPLE // 2
    rep = {}
    z_o = O.latent_down(xh[toks], W_ld)
    check_close("z", m.z[toks].double().cpu().numpy(), z_o, rep)
    Yg, Yo = [], []
    c_o = []
    for i, t in enumerate(toks):
        acc = np.zeros(L)
        for j in range(k):
            r = int(d["slot_of"][t, j])
            if r < 0:
                continue
            e = int(idx_o[t, j])
            y = O.expert_ffn(z_o[i:i + 1], _f64(inp["Wg"][e]), _f64(inp["Wu"][e]),
                             _f64(inp["Wd"][e]))[0]
            Yo.append(y)
            Yg.append(m.ypool[r].double().cpu().numpy())
            acc = acc + w_o[t, j] * y
        c_o.append(acc)
    check_close("Y", np.stack(Yg), np.stack(Yo), rep)
    c_o = O.bf16_round(np.stack(c_o))
    check_close("c", m.c[toks].double().cpu().numpy(), c_o, rep)
    a_o = O.shared_act(xh[toks], Wsg, Wsu)
    check_close("a", m.a[toks].double().cpu().numpy(), a_o, rep)
    out_o = O.output(c_o, a_o, W_lu, Wsd)
    check_close("out", m.out[toks].double().cpu().numpy(), out_o, rep)
    drop_rate = (st["dropped_send"] + st["dropped_recv"]) / (T * k)
    print(f"\n{name}: drop rate {drop_rate:.4f} (send {st['dropped_send']}, recv "
          f"{st['dropped_recv']}), near-ties {int((~clear).sum())}, flips {flips.size}, {rep}")
