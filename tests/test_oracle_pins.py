"""Pins of the CPU oracle against facts other than itself.

Each test checks one oracle function against something independent: a
library routine on a special case, brute-force enumeration on tiny inputs,
closed forms worked by hand from the pages' constants, or invariants the
pages state (kept rows never exceed either fixed buffer, drops are counted,
the shared experts still see every token).
"""
import json
import math
import os
from collections import Counter

import numpy as np
import pytest
import torch

import oracle as O
from moe_routing_capacity_gb300 import workloads as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _cfg(**kw):
    base = dict(name="t", T=16, d_model=8, d_latent=8, n_experts=6, n_ranks=2, top_k=2,
                n_waves=3, n_shared=1, h_expert=8, h_shared=8)
    base.update(kw)
    return wl.LayerConfig(**base)


# ------------------------------------------------------------------ numerics

def test_bf16_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)]
    # exact halfway points between neighbouring bf16 values (ties to even)
    base = rng.integers(1 << 7, 1 << 8, 4000).astype(np.float64)
    ex = rng.integers(-20, 20, 4000)
    vals.append(np.ldexp(base + 0.5, ex - 7))
    vals.append(-np.ldexp(base + 0.5, ex - 7))
    # subnormal range, near overflow, zeros
    vals.append(np.ldexp(rng.random(2000), -rng.integers(126, 149, 2000)))
    vals.append(np.array([3.38e38, 3.3895e38, 3.4e38, -3.4e38, 0.0, -0.0, 1e-45]))
    a = np.concatenate(vals).astype(np.float32)
    want = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(a.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_silu_against_library_logistic():
    from scipy.special import expit
    g = np.linspace(-40, 40, 10001)
    np.testing.assert_allclose(O.silu(g), g * expit(g), rtol=1e-14, atol=1e-300)


# ------------------------------------------------------------------ router

def _topk_brute(row, k):
    """Repeatedly take the largest remaining logit, lowest expert id on ties."""
    left = list(range(len(row)))
    out = []
    for _ in range(k):
        best = left[0]
        for e in left[1:]:
            if row[e] > row[best]:
                best = e
        out.append(best)
        left.remove(best)
    return out


def test_topk_matches_brute_force_with_exact_ties():
    rng = np.random.default_rng(1)
    # few distinct values -> many exact ties, exercising the lower-id rule
    l = rng.integers(-3, 4, size=(300, 12)).astype(np.float32)
    for k in (1, 2, 5, 12):
        idx, w, tie = O.router_topk(l, k)
        for t in range(l.shape[0]):
            assert list(idx[t]) == _topk_brute(list(l[t]), k)
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)


def test_gate_weights_two_way_closed_form():
    # softmax of two logits is the logistic of their difference
    l = np.array([[2.0, -1.0, 0.5], [0.25, 0.0, 3.0]], dtype=np.float32)
    idx, w, _ = O.router_topk(l, 2)
    assert idx.tolist() == [[0, 2], [2, 0]]
    d0 = 2.0 - 0.5
    d1 = 3.0 - 0.25
    np.testing.assert_allclose(w[0], [1 / (1 + math.exp(-d0)), 1 / (1 + math.exp(d0))], rtol=1e-14)
    np.testing.assert_allclose(w[1], [1 / (1 + math.exp(-d1)), 1 / (1 + math.exp(d1))], rtol=1e-14)


def test_tie_flags_on_constructed_gaps():
    eps = O.TIE_EPS
    l = np.array([
        [5.0, 4.0, 3.0, 2.0],                 # clear
        [5.0, 4.0, 4.0 - eps / 2, 2.0],       # k=2: boundary gap < eps
        [5.0, 5.0 - eps / 4, 3.0, 2.0],       # inner gap < eps
        [5.0, 5.0, 5.0, 2.0],                 # both
        [5.0, 4.0, 4.0 - 2 * eps, 1.0],       # gap 2*eps: not a tie
    ], dtype=np.float32)
    _, _, tie = O.router_topk(l, 2)
    assert tie.tolist() == [0, 1, 2, 3, 0]
    _, _, tie4 = O.router_topk(l, 4)          # k == E: no boundary to test
    assert tie4.tolist() == [0, 2, 2, 2, 0]         # row 1: its close pair is now inside


def test_router_logits_exact_on_integer_inputs():
    rng = np.random.default_rng(2)
    x = rng.integers(-4, 5, (5, 7)).astype(np.float64)
    Wr = rng.integers(-4, 5, (6, 7)).astype(np.float64)
    b = np.array([0.5, -0.25, 0, 1, 2, -3], dtype=np.float32)
    l = O.router_logits(x, Wr, b)
    for t in range(5):
        for e in range(6):
            s = 0.0
            for i in range(7):
                s += x[t, i] * Wr[e, i]
            assert l[t, e] == np.float32(s + float(b[e]))


# ------------------------------------------------------------------ capacities

def test_pages_constants_are_the_full_workload():
    g = json.load(open(os.path.join(GOLD, "pages_constants.json")))
    c = wl.FULL
    assert c.n_experts == g["routed_experts"] and c.top_k == g["top_k"]
    assert c.n_shared == g["shared_experts"] and c.d_model == g["model_width"]
    assert c.d_latent == g["latent_width"] and c.n_ranks == g["expert_parallel_gpus"]
    assert c.n_experts // c.n_ranks == g["experts_per_gpu"] and c.n_waves == g["waves"]
    assert c.cf_send == g["sender_capacity_factor"] and c.cf_recv == g["receiver_capacity_factor"]


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLD, "capacities.json")))["cases"],
                         ids=lambda c: c["name"])
def test_capacity_closed_forms(case):
    cfg = _cfg(T=case["T"], n_ranks=case["ranks"], n_experts=case["E"], top_k=case["k"],
               n_waves=case["W"], cf_send=float(case["cf_send"]), cf_recv=float(case["cf_recv"]))
    p = O.make_plan(cfg)
    assert (p.c_send, p.c_recv, p.pool_rows) == (case["c_send"], case["c_recv"], case["pool_rows"])


# ------------------------------------------------------------------ dispatch, brute force

def _lex_first_maximal(keys, cap):
    """Among all subsets that respect `cap` per key and to which no element
    can be added, the one whose membership vector (in priority order, 1 > 0)
    is largest.  Exhaustive over 2^n subsets."""
    n = len(keys)
    best = None
    for mask in range(1 << n):
        cnt = Counter(keys[i] for i in range(n) if mask >> i & 1)
        if any(v > cap for v in cnt.values()):
            continue
        if any(cnt[keys[i]] < cap for i in range(n) if not mask >> i & 1):
            continue
        vec = tuple((mask >> i) & 1 for i in range(n))
        if best is None or vec > best:
            best = vec
    return best


def _random_routing(rng, T, E, k):
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("seed", range(40))
def test_dispatch_equals_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    T, ranks, E, W = 4, 2, 6, [1, 3][seed % 2]
    k = [2, 3][seed % 3 == 0]
    cf_s = [1.1, 2.0, 0.5][seed % 3]
    cf_r = [0.7, 1.1, 2.0][(seed // 3) % 3]
    cfg = _cfg(T=T, n_ranks=ranks, n_experts=E, top_k=k, n_waves=W, cf_send=cf_s, cf_recv=cf_r)
    p = O.make_plan(cfg)
    # skew half the cases towards expert 0/1 so caps bind
    idx = _random_routing(rng, T, E, k)
    if seed % 2:
        idx = np.stack([np.r_[0, rng.choice(np.arange(1, E), k - 1, replace=False)]
                        for _ in range(T)]).astype(np.int32)
    d = O.dispatch(idx, p)

    prio = [(t, j) for t in range(T) for j in range(k)]
    send_key = []
    for t, j in prio:
        e = int(idx[t, j])
        send_key.append((t // p.T_s, e // p.E_l, (e % p.E_l) // p.E_w))
    want_send = _lex_first_maximal(send_key, p.c_send)
    got_send = tuple(int(d["drop"][t, j] != O.DROP_SEND) for t, j in prio)
    assert got_send == want_send

    kept = [i for i in range(len(prio)) if want_send[i]]
    recv_key = [int(idx[prio[i]]) for i in kept]
    want_recv = _lex_first_maximal(recv_key, p.c_recv) if kept else ()
    got_recv = tuple(int(d["drop"][prio[i]] == O.DROP_KEPT) for i in kept)
    assert got_recv == want_recv

    # slots: position among earlier sender-kept rows of the same key; rows by layout
    for a, i in enumerate(kept):
        n = sum(1 for b in kept[:a] if send_key[b] == send_key[i])
        s, dst, wv = send_key[i]
        row = ((dst * W + wv) * p.S + s) * p.c_send + n
        assert d["send_row"][prio[i]] == row
        if d["drop"][prio[i]] == O.DROP_KEPT:
            assert d["slot_of"][prio[i]] == row
        else:
            assert d["slot_of"][prio[i]] == -1
    # expert rows: the r-th receiver-kept assignment of e sits at expert_rows[e, r]
    for e in range(E):
        mine = [prio[i] for a, i in enumerate(kept) if want_recv[a] and recv_key[a] == e]
        assert d["count"][e] == len(mine)
        for r, tj in enumerate(mine):
            assert d["expert_rows"][e, r] == d["slot_of"][tj]
        assert (d["expert_rows"][e, len(mine):] == -1).all()


# ------------------------------------------------------------------ dispatch, invariants

def _check_invariants(idx, p, d):
    T, k = idx.shape
    st = d["stats"]
    assert st["kept"] + st["dropped_send"] + st["dropped_recv"] == T * k
    assert (d["drop"] == O.DROP_KEPT).sum() == st["kept"]
    assert (d["drop"] == O.DROP_SEND).sum() == st["dropped_send"]
    assert (d["drop"] == O.DROP_RECV).sum() == st["dropped_recv"]
    assert (d["send_fill"] <= p.c_send).all()
    assert (d["count"] <= p.c_recv).all()
    assert d["count"].sum() == st["kept"]
    rows = d["send_row"][d["send_row"] >= 0]
    assert np.unique(rows).size == rows.size                 # no two rows share a slot
    assert ((rows >= 0) & (rows < p.pool_rows)).all()
    for e in range(p.E):
        r = d["expert_rows"][e, :d["count"][e]]
        dst, _, wv = O.placement(e, p)
        slice_ = r // (p.S * p.c_send)
        assert (slice_ == dst * p.W + wv).all()               # rows sit in e's (dst, wave) slice
        assert np.unique(r).size == r.size


@pytest.mark.parametrize("kind", ["uniform", "zipf", "one-destination"])
def test_dispatch_invariants_medium(kind):
    rng = np.random.default_rng(7)
    cfg = _cfg(T=2048, n_ranks=8, n_experts=48, top_k=8, n_waves=3)
    p = O.make_plan(cfg)
    if kind == "uniform":
        idx = _random_routing(rng, cfg.T, cfg.n_experts, cfg.top_k)
    elif kind == "zipf":
        pr = np.arange(1, 49, dtype=np.float64) ** -1.2
        pr /= pr.sum()
        idx = np.stack([rng.choice(48, 8, replace=False, p=pr) for _ in range(cfg.T)]).astype(np.int32)
    else:
        idx = np.tile(np.arange(8, dtype=np.int32), (cfg.T, 1))   # experts 0..7: destinations 0, 1
    d = O.dispatch(idx, p)
    _check_invariants(idx, p, d)
    if kind != "uniform":
        assert d["stats"]["dropped_send"] > 0


def test_all_tokens_on_one_expert_closed_form():
    # k=1, every token picks expert 0: each source keeps min(T_s, c_send) rows,
    # then the receiver keeps min(S * that, c_recv)
    cfg = _cfg(T=64, n_ranks=4, n_experts=12, top_k=1, n_waves=3, cf_send=2.0, cf_recv=1.15)
    p = O.make_plan(cfg)
    idx = np.zeros((64, 1), dtype=np.int32)
    d = O.dispatch(idx, p)
    per_src = min(p.T_s, p.c_send)
    assert d["stats"]["dropped_send"] == 64 - p.S * per_src
    assert d["stats"]["kept"] == min(p.S * per_src, p.c_recv)
    assert d["count"][0] == d["stats"]["kept"] and d["count"][1:].sum() == 0


def test_unbounded_factors_drop_nothing():
    rng = np.random.default_rng(3)
    cfg = _cfg(T=512, n_ranks=4, n_experts=24, top_k=4, cf_send=float("inf"), cf_recv=float("inf"))
    p = O.make_plan(cfg)
    idx = np.zeros((512, 4), dtype=np.int32)
    idx[:] = np.arange(4)                                          # worst case: all on experts 0..3
    d = O.dispatch(idx, p)
    assert d["stats"]["kept"] == 512 * 4
    idx = _random_routing(rng, 512, 24, 4)
    assert O.dispatch(idx, p)["stats"]["kept"] == 512 * 4


def test_empty_batch():
    cfg = _cfg(T=0, n_ranks=2)
    p = O.make_plan(cfg)
    assert p.pool_rows == 0 and p.c_send == 0
    d = O.dispatch(np.zeros((0, 2), dtype=np.int32), p)
    assert d["stats"] == dict(assignments=0, kept=0, dropped_send=0, dropped_recv=0)


# ------------------------------------------------------------------ pack

def test_pack_tags_and_payload():
    rng = np.random.default_rng(4)
    cfg = _cfg(T=32, n_ranks=2, n_experts=6, top_k=2, n_waves=3, cf_send=1.1, cf_recv=1.1)
    p = O.make_plan(cfg)
    idx = _random_routing(rng, 32, 6, 2)
    d = O.dispatch(idx, p)
    z = rng.standard_normal((32, 8))
    payload, tags = O.pack_pool(z, idx, d, p)
    filled = 0
    for t in range(32):
        for j in range(2):
            r = d["send_row"][t, j]
            if r >= 0:
                filled += 1
                assert tags[r].tolist() == [idx[t, j], t, j, 0]
                np.testing.assert_array_equal(payload[r], z[t])
    empty = (tags[:, 0] == -1)
    assert empty.sum() == p.pool_rows - filled
    assert np.isnan(payload[empty]).all()


# ------------------------------------------------------------------ whole layer

def _tiny_inputs(cfg):
    return {k: (v.float().numpy() if v is not None else None)
            for k, v in wl.make_inputs(cfg, "cpu").items()}


def _golden_layer(name):
    g = json.load(open(os.path.join(GOLD, name)))
    cfg = _cfg(**g["config"])
    t = {k: np.array(g[k], dtype=np.float64) for k in
         ("x", "Wr", "W_ld", "Wg", "Wu", "Wd", "W_lu", "Wsg", "Wsu", "Wsd")}
    t["bias"] = None
    return O.layer(cfg, t), g["expect"]


def test_worked_example_by_hand():
    r, ex = _golden_layer("worked_example.json")
    np.testing.assert_array_equal(r["logits"], ex["logits"])
    assert r["idx"].tolist() == ex["idx"]
    np.testing.assert_array_equal(r["w"], ex["w"])
    np.testing.assert_array_equal(r["z"], ex["z"])
    assert (r["plan"].c_send, r["plan"].c_recv, r["plan"].pool_rows) == \
        (ex["c_send"], ex["c_recv"], ex["pool_rows"])
    assert r["disp"]["slot_of"].tolist() == ex["slot_of"]
    np.testing.assert_array_equal(r["Y"][0], ex["Y_row0"])
    np.testing.assert_array_equal(r["Y"][1], ex["Y_row1"])
    np.testing.assert_array_equal(r["c"], ex["c"])
    np.testing.assert_array_equal(r["a"], ex["a"])
    np.testing.assert_array_equal(r["out"], ex["out"])


def test_partial_drop_by_hand():
    """A token whose second assignment overflows the receiver's one-row cap
    keeps its first expert's output at the unchanged gate weight (no
    renormalisation), and its shared term; the dropped row is counted."""
    r, ex = _golden_layer("partial_drop.json")
    np.testing.assert_array_equal(r["logits"], ex["logits"])
    assert r["idx"].tolist() == ex["idx"]
    np.testing.assert_allclose(r["w"], ex["w"], rtol=1e-15, atol=0)
    np.testing.assert_array_equal(r["z"], ex["z"])
    assert (r["plan"].c_send, r["plan"].c_recv, r["plan"].pool_rows) == \
        (ex["c_send"], ex["c_recv"], ex["pool_rows"])
    d = r["disp"]
    assert d["slot_of"].tolist() == ex["slot_of"]
    assert d["drop"].tolist() == ex["drop"]
    assert d["expert_rows"].tolist() == ex["expert_rows"]
    assert d["count"].tolist() == ex["count"]
    assert d["stats"] == ex["stats"]
    assert r["tags"].tolist() == ex["tags"]
    assert sorted(r["Y"]) == sorted(int(k) for k in ex["Y"])
    for row, y in ex["Y"].items():
        np.testing.assert_array_equal(r["Y"][int(row)], y)
    np.testing.assert_array_equal(r["c"], ex["c"])
    for wrong in ("c_if_renormalised", "c_if_wrong_rank_dropped"):
        assert not np.array_equal(r["c"], ex[wrong])
    np.testing.assert_array_equal(r["a"], ex["a"])
    np.testing.assert_array_equal(r["out"], ex["out"])


def test_two_shared_experts_by_hand():
    """Two shared experts with distinct weights: each one's activations sit
    in its own slice of a, and out carries the sum of both down-projections."""
    r, ex = _golden_layer("two_shared.json")
    np.testing.assert_array_equal(r["logits"], ex["logits"])
    assert r["idx"].tolist() == ex["idx"]
    np.testing.assert_array_equal(r["w"], ex["w"])
    np.testing.assert_array_equal(r["z"], ex["z"])
    assert (r["plan"].c_send, r["plan"].c_recv, r["plan"].pool_rows) == \
        (ex["c_send"], ex["c_recv"], ex["pool_rows"])
    assert r["disp"]["slot_of"].tolist() == ex["slot_of"]
    np.testing.assert_array_equal(r["c"], ex["c"])
    np.testing.assert_array_equal(r["a"], ex["a"])
    np.testing.assert_array_equal(r["out"], ex["out"])


def test_unbounded_layer_equals_dense_mixture():
    """With no caps nothing drops, and the pooled layer must equal a dense
    per-token mixture evaluated straight from the routing (no pools)."""
    cfg = wl.TINY.with_(cf_send=float("inf"), cf_recv=float("inf"))
    t = _tiny_inputs(cfg)
    r = O.layer(cfg, t)
    assert r["disp"]["stats"]["kept"] == cfg.T * cfg.top_k
    x = t["x"].astype(np.float64)
    z = O.bf16_round(np.einsum("td,ld->tl", x, t["W_ld"].astype(np.float64)))
    idx, w = r["idx"], r["w"]
    Wg, Wu, Wd = (t[n].astype(np.float64) for n in ("Wg", "Wu", "Wd"))
    g = np.einsum("tl,tjhl->tjh", z, Wg[idx])
    u = np.einsum("tl,tjhl->tjh", z, Wu[idx])
    h = O.bf16_round(g / (1 + np.exp(-g)) * u)
    Y = O.bf16_round(np.einsum("tjh,tjlh->tjl", h, Wd[idx]))
    c = O.bf16_round(np.einsum("tj,tjl->tl", w, Y))
    xs = np.einsum("td,shd->tsh", x, t["Wsg"].astype(np.float64))
    us = np.einsum("td,shd->tsh", x, t["Wsu"].astype(np.float64))
    a = O.bf16_round(xs / (1 + np.exp(-xs)) * us)
    out = O.bf16_round(np.einsum("tl,dl->td", c, t["W_lu"].astype(np.float64))
                       + np.einsum("tsh,sdh->td", a, t["Wsd"].astype(np.float64)))
    np.testing.assert_array_equal(r["z"], z)
    np.testing.assert_allclose(r["c"], c, rtol=2 ** -8, atol=0)   # association order only
    np.testing.assert_allclose(r["out"], out, rtol=2 ** -8, atol=1e-12)
    assert (r["out"] != out).mean() < 1e-3


def test_shared_path_reaches_every_token():
    """Routed weights zeroed, or every assignment dropped: the output is the
    shared experts alone, for every token."""
    cfg = wl.TINY
    t = _tiny_inputs(cfg)
    x = t["x"].astype(np.float64)
    a = O.shared_act(x, t["Wsg"], t["Wsu"])
    shared = O.bf16_round(sum(a[:, s * cfg.h_shared:(s + 1) * cfg.h_shared]
                              @ t["Wsd"][s].astype(np.float64).T for s in range(cfg.n_shared)))
    r0 = O.layer(cfg, t, gate_w=np.zeros((cfg.T, cfg.top_k)))
    np.testing.assert_array_equal(r0["out"], shared)
    # caps of one row: almost everything drops, the dropped tokens keep the shared term
    cfg_min = cfg.with_(cf_send=0.01, cf_recv=0.01)
    r1 = O.layer(cfg_min, t)
    assert r1["disp"]["stats"]["kept"] <= cfg.n_experts
    none_kept = (r1["disp"]["drop"] != O.DROP_KEPT).all(axis=1)
    assert none_kept.sum() > cfg.T // 2
    np.testing.assert_array_equal(r1["out"][none_kept], shared[none_kept])
    np.testing.assert_array_equal(r1["c"][none_kept], 0.0)


def test_tiny_layer_invariants():
    cfg = wl.TINY
    t = _tiny_inputs(cfg)
    r = O.layer(cfg, t)
    _check_invariants(r["idx"], r["plan"], r["disp"])
    assert r["out"].shape == (cfg.T, cfg.d_model)
    assert np.isfinite(r["out"]).all()
    # every pool tag matches the routing
    for t_ in range(cfg.T):
        for j in range(cfg.top_k):
            row = r["disp"]["send_row"][t_, j]
            if row >= 0:
                assert r["tags"][row].tolist() == [r["idx"][t_, j], t_, j, 0]


def test_skewed_bias_raises_drops():
    """A Zipf prior on the logits concentrates load on low experts, so the
    fixed caps drop more (the pages' point that uneven routing drops rows)."""
    base = wl.TINY.with_(T=512)
    t = _tiny_inputs(base)
    r0 = O.layer(base, t)
    t["bias"] = wl.zipf_bias(base.n_experts, 1.2).numpy()
    r1 = O.layer(base, t)
    d0 = r0["disp"]["stats"]["dropped_send"] + r0["disp"]["stats"]["dropped_recv"]
    d1 = r1["disp"]["stats"]["dropped_send"] + r1["disp"]["stats"]["dropped_recv"]
    assert d1 > 2 * d0


# ------------------------------------------------------------------ balancing bias

def test_balance_update_closed_form():
    # 4 experts; selections 0,0,0,1,1,2 (expert 3 never): H = [3, 2, 1, 0],
    # f = [1/2, 1/3, 1/6, 0], b = -alpha (f - 1/4)
    idx = np.array([[0, 1], [0, 2], [0, 1]])
    h, b = O.balance_update(idx, np.zeros(4, dtype=np.int64), 0.5, 4)
    assert h.tolist() == [3, 2, 1, 0]
    np.testing.assert_allclose(b, [-0.5 * (1/2 - 1/4), -0.5 * (1/3 - 1/4),
                                   -0.5 * (1/6 - 1/4), -0.5 * (0 - 1/4)], rtol=1e-15)
    # accumulates over batches
    h2, b2 = O.balance_update(np.array([[3, 2]]), h, 0.5, 4)
    assert h2.tolist() == [3, 2, 2, 1]
    np.testing.assert_allclose(b2, -0.5 * (np.array([3, 2, 2, 1]) / 8 - 0.25), rtol=1e-15)


def test_balance_update_invariants():
    rng = np.random.default_rng(9)
    E = 24
    idx = _random_routing(rng, 500, E, 4)
    h, b = O.balance_update(idx, np.zeros(E, dtype=np.int64), 0.01, E)
    assert h.sum() == 500 * 4
    assert abs(b.sum()) < 1e-15                      # sum_i (f_i - 1/E) = 0
    assert ((b < 0) == (h > h.sum() / E)).all()      # over-selected experts pushed down
    flat = np.tile(np.arange(E), 10).reshape(-1, 4)  # perfectly balanced selections
    _, b0 = O.balance_update(flat, np.zeros(E, dtype=np.int64), 1.0, E)
    np.testing.assert_allclose(b0, 0.0, atol=1e-17)
    _, bz = O.balance_update(np.zeros((0, 4), dtype=np.int64), np.zeros(E, dtype=np.int64), 1.0, E)
    assert (bz == 0).all()


def test_balance_window_closed_form():
    # window of 2 batches over 3 batches that select expert 0, then 1, then 2
    # (three assignments each): after batch 3, H holds batches 2 and 3 only
    E, alpha = 4, 0.5
    h = np.zeros(E, dtype=np.int64)
    ring = np.zeros((2, E), dtype=np.int64)
    step = 0
    for e in (0, 1, 2):
        h, ring, step, b = O.balance_update_window(np.full((3, 1), e), h, ring, step, alpha, E)
    assert step == 3
    assert h.tolist() == [0, 3, 3, 0]
    np.testing.assert_allclose(b, [alpha / 4, -alpha / 4, -alpha / 4, alpha / 4], rtol=1e-15)
    # window of one batch: H is the last batch's counts
    h1, r1, _, _ = O.balance_update_window(np.array([[1, 3], [3, 3]]), np.array([5, 0, 0, 0]),
                                           np.array([[5, 0, 0, 0]]), 7, alpha, E)
    assert h1.tolist() == [0, 1, 0, 3] and r1.tolist() == [[0, 1, 0, 3]]


def test_balance_window_longer_than_history_is_plain_accumulation():
    rng = np.random.default_rng(4)
    E = 12
    h_w = h_a = np.zeros(E, dtype=np.int64)
    ring = np.zeros((10, E), dtype=np.int64)
    step = 0
    for _ in range(6):
        idx = _random_routing(rng, 40, E, 3)
        h_w, ring, step, b_w = O.balance_update_window(idx, h_w, ring, step, 0.1, E)
        h_a, b_a = O.balance_update(idx, h_a, 0.1, E)
        assert (h_w == h_a).all()
        np.testing.assert_array_equal(b_w, b_a)


# ------------------------------------------------------------------ dropless ragged dispatch

@pytest.mark.parametrize("seed", range(6))
def test_ragged_dispatch_structure(seed):
    rng = np.random.default_rng(200 + seed)
    cfg = _cfg(T=96, n_ranks=4, n_experts=24, top_k=3, n_waves=[1, 3][seed % 2])
    p = O.make_plan(cfg)
    idx = _random_routing(rng, cfg.T, cfg.n_experts, cfg.top_k)
    if seed >= 3:
        idx[:, 0] = 0                      # everyone also picks expert 0 (kept anyway)
        idx = np.stack([np.r_[0, rng.choice(np.arange(1, 24), 2, replace=False)] for _ in range(96)])
    d = O.dispatch_ragged(idx, p)
    rows = d["slot_of"].reshape(-1)
    assert sorted(rows.tolist()) == list(range(cfg.T * cfg.top_k))      # a permutation: no gaps
    assert (d["drop"] == 0).all()
    # brute force: rows grouped by (dst, wave, src) in that order, priority inside
    prio = [(t, j) for t in range(cfg.T) for j in range(cfg.top_k)]
    def blk(tj):
        e = int(idx[tj]); dst = e // p.E_l; wv = (e % p.E_l) // p.E_w
        return (dst, wv, tj[0] // p.T_s)
    order = sorted(prio, key=lambda tj: (blk(tj), tj))
    for r, tj in enumerate(order):
        assert d["slot_of"][tj] == r
    for e in range(p.E):
        mine = [d["slot_of"][tj] for tj in prio if idx[tj] == e]
        got = d["expert_rows"][d["expert_offsets"][e]:d["expert_offsets"][e + 1]]
        assert got.tolist() == mine


def test_ragged_layer_equals_unbounded_capped_layer():
    """Without caps nothing drops in either layout, so every token's result
    is the same whether the pools are padded (cf = inf) or ragged."""
    cfg = wl.TINY.with_(cf_send=float("inf"), cf_recv=float("inf"))
    t = _tiny_inputs(cfg)
    a = O.layer(cfg, t)
    b = O.layer_ragged(cfg, t)
    assert a["disp"]["stats"]["kept"] == b["disp"]["stats"]["kept"] == cfg.T * cfg.top_k
    np.testing.assert_array_equal(a["c"], b["c"])
    np.testing.assert_array_equal(a["out"], b["out"])
    for tt in range(cfg.T):
        for j in range(cfg.top_k):
            np.testing.assert_array_equal(a["Y"][int(a["disp"]["slot_of"][tt, j])],
                                          b["Y"][int(b["disp"]["slot_of"][tt, j])])


# ------------------------------------------------------------------ backward pass

def test_backward_matches_central_differences():
    """Every gradient of the float64 (rounding-free) layer against central
    differences of the forward: d<out, dout>/dparam at random entries."""
    cfg = _cfg(T=16, n_ranks=2, n_experts=6, top_k=2, n_waves=3, n_shared=2, h_expert=8,
               h_shared=8, cf_send=float("inf"), cf_recv=float("inf"))
    t = {k: (v.double().numpy() if v is not None else None)
         for k, v in wl.make_inputs(cfg.with_(seed=5), "cpu").items()}
    fwd = O.layer(cfg, t, rnd=O.exact)
    rng = np.random.default_rng(11)
    dout = rng.standard_normal(fwd["out"].shape)
    g = O.layer_backward(cfg, t, fwd, dout, rnd=O.exact)

    def loss(tt):
        r = O.layer(cfg, tt, rnd=O.exact)
        assert (r["idx"] == fwd["idx"]).all()            # no selection change within +-eps
        return (r["out"] * dout).sum()

    for name in ["x", "Wr", "W_ld", "Wg", "Wu", "Wd", "W_lu", "Wsg", "Wsu", "Wsd"]:
        for _ in range(4):
            idx = tuple(int(rng.integers(0, n)) for n in t[name].shape)
            tt = {k: (v.copy() if v is not None else None) for k, v in t.items()}
            eps = 1e-5
            tt[name][idx] += eps
            up = loss(tt)
            tt[name][idx] -= 2 * eps
            down = loss(tt)
            fd = (up - down) / (2 * eps)
            assert abs(fd - g[name][idx]) <= 1e-6 * (1 + abs(fd)), (name, idx, fd, g[name][idx])


def test_backward_dropped_assignments_get_no_expert_gradient():
    """A dropped assignment contributes nothing forward, so its expert and
    gate-weight gradients vanish; the shared path still gets its gradient."""
    cfg = _cfg(T=32, n_ranks=2, n_experts=6, top_k=2, cf_send=0.01, cf_recv=0.01)
    t = {k: (v.double().numpy() if v is not None else None)
         for k, v in wl.make_inputs(cfg.with_(seed=6), "cpu").items()}
    fwd = O.layer(cfg, t)
    dout = np.ones(fwd["out"].shape)
    g = O.layer_backward(cfg, t, fwd, dout)
    dropped = fwd["disp"]["slot_of"] < 0
    assert dropped.any()
    assert (g["dw"][dropped] == 0).all()
    never = np.setdiff1d(np.arange(6), fwd["idx"][~dropped])
    for e in never:
        assert (g["Wd"][e] == 0).all() and (g["Wg"][e] == 0).all()
    assert np.abs(g["Wsg"]).sum() > 0
