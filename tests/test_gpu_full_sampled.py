"""Full-size parity: the full-width layer (384 experts, top-8, 64 logical
ranks, d=6144, L=3072), its Zipf-skewed variant and the 65536-token AR(1)
long-context variant, run exactly as the benchmark runs them (the pool fill
inside the shared experts' gate/up launch), and the full layer once more
with the calls one after another.

The oracle recomputes the routing, the whole dispatch and every pool tag
(integer results compared bit-exactly, near-ties excepted), and the
floating-point path for a sample of tokens plus one whole block of 256
consecutive tokens.  Properties that hold at any size (caps, conservation,
the pack being a copy) are checked on everything.  Inputs are drawn on the
device by torch's seeded generator; the oracle gets host copies of those
inputs, never a value the library computed.
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
BLOCK = 256


def _f64(t):
    return t.detach().double().cpu().numpy()


def _f32(t):
    return t.detach().float().cpu().numpy()


def _sample_tokens(T, n, seed):
    rng = np.random.default_rng(seed)
    pick = set([0, T - 1]) | set(rng.choice(T, n - 2, replace=False).tolist())
    return np.array(sorted(pick))


@pytest.mark.parametrize("name,pipeline", [("full", "shared"), ("full", None),
                                           ("skew", "shared"), ("long", "shared")])
def test_full_size_against_oracle(name, pipeline):
    cfg = wl.CONFIGS[name]
    inp = wl.make_inputs(cfg, "cuda")
    m = PooledWaveMoE(cfg, inp, "cuda", pipeline=pipeline)
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

    # ---- dispatch for every assignment, every pool tag
    d = O.dispatch(idx_o, p)
    slot_of, drop = m.slot_of.cpu().numpy(), m.drop.cpu().numpy()
    rows, count = m.expert_rows.cpu().numpy(), m.expert_count.cpu().numpy()
    tags = m.pool_tags()
    tags_g = tags.cpu().numpy()
    flips = np.nonzero((idx != idx_o).any(axis=1))[0]
    # A token whose routing differs (a near-tie, both orders correct) moves
    # sender slots only in the (source, destination, wave) slices its
    # assignments touch; that can change which rows of any expert of such a
    # slice's (destination, wave) are sender-kept, hence those experts'
    # receiver ranks.  An expert that never reaches c_recv (on either side)
    # drops nothing at the receiver, so its decisions stay exact outside the
    # touched slices.  Everything else is compared bit for bit.
    E_l, E_w, W, S = p.E_l, p.E_w, p.W, p.S
    bad_slice = np.zeros((p.D, W, S), dtype=bool)
    bad_e = np.zeros(p.E, dtype=bool)
    for t in flips:
        for e in set(idx[t].tolist()) | set(idx_o[t].tolist()):
            bad_slice[e // E_l, (e % E_l) // E_w, t // p.T_s] = True
            bad_e[e] = True
    dw_bad = bad_slice.any(axis=2)                       # [D, W]
    for e in range(p.E):
        if dw_bad[e // E_l, (e % E_l) // E_w]:
            bad_e[e] = True
    recv_safe = (count < p.c_recv) & (d["count"] < p.c_recv)
    if flips.size == 0:
        for key in ("kept", "dropped_send", "dropped_recv"):
            assert st[key] == d["stats"][key]
    same_tok = ~np.isin(np.arange(T), flips)
    e_o = idx_o.astype(np.int64)
    sl = bad_slice[e_o // E_l, (e_o % E_l) // E_w, (np.arange(T) // p.T_s)[:, None]]
    # a sender drop depends only on its own slice; a sender-kept row's
    # receiver decision on its expert's whole sequence
    exact = same_tok[:, None] & ~sl & ((d["drop"] == O.DROP_SEND) | ~bad_e[e_o] | recv_safe[e_o])
    assert exact.mean() > 0.95
    np.testing.assert_array_equal(slot_of[exact], d["slot_of"][exact])
    np.testing.assert_array_equal(drop[exact], d["drop"][exact])
    for e in np.nonzero(~bad_e)[0]:
        assert count[e] == d["count"][e], e
        np.testing.assert_array_equal(rows[e], d["expert_rows"][e])
    # every pool tag: the oracle's pool with a one-column payload (its tags
    # depend only on the dispatch; its first payload column is the oracle's
    # z column 0, floating point, so within the tolerance)
    z0 = O.latent_down(xh, _f64(inp["W_ld"][:1]))
    pay_o, tags_o = O.pack_pool(z0, idx_o, d, p)
    row_ok = ~np.repeat(bad_slice.reshape(-1), p.c_send)
    assert row_ok.mean() > 0.95
    np.testing.assert_array_equal(tags_g[row_ok], tags_o[row_ok])
    filled_o = (tags_o[:, 0] >= 0) & row_ok
    pay0 = m.pool_payload()[:, 0].double().cpu().numpy()
    check_close("pool payload column 0", pay0[filled_o], pay_o[filled_o, 0])
    if flips.size:
        t0 = int(flips[0])
        assert (slot_of[:t0] == d["slot_of"][:t0]).all() and (drop[:t0] == d["drop"][:t0]).all()
        dispatch_rules_hold(idx, slot_of, drop, rows, count, p)
    assert st["kept"] + st["dropped_send"] + st["dropped_recv"] == T * k
    assert st["max_send_fill"] <= p.c_send and st["max_expert_rows"] <= p.c_recv

    # ---- properties of the pool at full size (checked on the device)
    filled = tags[:, 0] >= 0
    assert int(filled.sum()) == st["kept"] + st["dropped_recv"]
    tok = tags[filled, 1].long()
    assert torch.equal(m.pool_payload()[filled], m.z[tok])
    e_tag = tags[filled, 0]
    assert bool((m.idx[tok, tags[filled, 2].long()] == e_tag).all())

    # ---- floating point: sampled tokens plus one whole block of consecutive
    # tokens (the second source's first BLOCK tokens); routed experts grouped
    # so that each expert's weights are widened once
    W_ld = _f64(inp["W_ld"])
    W_lu = _f64(inp["W_lu"])
    Wsg, Wsu, Wsd = _f64(inp["Wsg"]), _f64(inp["Wsu"]), _f64(inp["Wsd"])
    same = (idx == idx_o).all(axis=1) & (drop == d["drop"]).all(axis=1)
    b0 = p.T_s
    block = np.arange(b0, b0 + BLOCK)
    toks = np.array(sorted(set(_sample_tokens(T, N_SAMPLE, cfg.seed).tolist())
                           | set(block.tolist())))
    toks = toks[same[toks]]
    assert same[block].mean() > 0.95 and toks.size >= BLOCK
    pos = {int(t): i for i, t in enumerate(toks)}
    rep = {}
    z_o = O.latent_down(xh[toks], W_ld)
    check_close("z", m.z[torch.from_numpy(toks).cuda()].double().cpu().numpy(), z_o, rep)
    by_e = {}
    for t in toks:
        for j in range(k):
            if d["slot_of"][t, j] >= 0:
                by_e.setdefault(int(idx_o[t, j]), []).append((int(t), j))
    Y_o = {}
    for e, tj in sorted(by_e.items()):
        X = z_o[[pos[t] for t, _ in tj]]
        Ye = O.expert_ffn(X, _f32(inp["Wg"][e]), _f32(inp["Wu"][e]), _f32(inp["Wd"][e]))
        for (t, j), y in zip(tj, Ye):
            Y_o[(t, j)] = y
    keys = sorted(Y_o)
    ysel = torch.tensor([int(d["slot_of"][t, j]) for t, j in keys], device="cuda")
    check_close("Y", m.ypool[ysel].double().cpu().numpy(), np.stack([Y_o[q] for q in keys]), rep)
    c_o = []
    for t in toks:
        acc = np.zeros(L)
        for j in range(k):
            if d["slot_of"][t, j] >= 0:
                acc = acc + w_o[t, j] * Y_o[(int(t), j)]
        c_o.append(acc)
    c_o = O.bf16_round(np.stack(c_o))
    tsel = torch.from_numpy(toks).cuda()
    check_close("c", m.c[tsel].double().cpu().numpy(), c_o, rep)
    a_o = O.shared_act(xh[toks], Wsg, Wsu)
    check_close("a", m.a[tsel].double().cpu().numpy(), a_o, rep)
    out_o = O.output(c_o, a_o, W_lu, Wsd)
    check_close("out", m.out[tsel].double().cpu().numpy(), out_o, rep)
    drop_rate = (st["dropped_send"] + st["dropped_recv"]) / (T * k)
    print(f"\n{name}/{pipeline}: drop rate {drop_rate:.4f} (send {st['dropped_send']}, recv "
          f"{st['dropped_recv']}), near-ties {int((~clear).sum())}, flips {flips.size}, "
          f"exact assignments {exact.mean():.4f}, exact pool rows {row_ok.mean():.4f}, "
          f"exact expert lists {int((~bad_e).sum())}/{p.E}, "
          f"{toks.size} tokens compared, {rep}")
