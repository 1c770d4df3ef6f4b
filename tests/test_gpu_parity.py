"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer results (top-k ids away from near-ties, pool slots, drop decisions,
expert row lists, tags, drop counts) must be bit-exact; floating-point
results must meet the bf16 tolerance in ``helpers``.  Where a near-tie let
the GPU's fp32 logits order two experts differently from the oracle's, the
dispatch is compared bit-exactly up to the first such token and checked
against the rules for the GPU's own routing after it.
"""
import numpy as np
import pytest
import torch

import oracle as O
from moe_routing_capacity_gb300 import workloads as wl
from moe_routing_capacity_gb300.layer import PooledWaveMoE

from helpers import (LOGIT_ATOL, check_close, dispatch_rules_hold, tie_margin_ok)

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64) if t.is_floating_point() \
        else t.detach().cpu().numpy()


def _host_inputs(inp):
    return {k: (v.float().cpu().numpy() if v is not None else None) for k, v in inp.items()}


def run_gpu(cfg, inp, **layer_kw):
    m = PooledWaveMoE(cfg, inp, "cuda", **layer_kw)
    x = inp["x"].cuda()
    m.forward(x)
    torch.cuda.synchronize()
    assert int(m.status.item()) == 0, "device status word set"
    st = m.drop_stats()
    assert st["status"] == 0, st
    return m


def compare_full(cfg, inp, report=None, **layer_kw):
    """Element-by-element comparison of every stage (sizes the oracle
    finishes in seconds); layer_kw selects a variant of the GPU layer."""
    report = {} if report is None else report
    ref = O.layer(cfg, _host_inputs(inp))
    m = run_gpu(cfg, inp, **layer_kw)
    p = ref["plan"]
    # router
    lg = _np(m.logits)
    assert np.abs(lg - ref["logits"]).max() <= LOGIT_ATOL
    idx = _np(m.idx)
    tie = _np(m.tie)
    clear = ref["tie"] == 0
    assert (idx[clear] == ref["idx"][clear]).all(), "top-k ids differ away from near-ties"
    lerr = float(np.abs(lg - ref["logits"]).max())
    stable = tie_margin_ok(ref["logits"], cfg.top_k, ref["idx"], 2 * lerr + 1e-7)
    assert (tie[stable] == ref["tie"][stable]).all(), "near-tie flags differ"
    same_route = clear | (idx == ref["idx"]).all(axis=1)
    check_close("w", _np(m.gate_w)[same_route], ref["w"][same_route], report)
    report["near_tie_tokens"] = int((~clear).sum())
    # latent
    check_close("z", _np(m.z), ref["z"], report)
    # dispatch
    slot_of, drop = _np(m.slot_of), _np(m.drop)
    rows, count = _np(m.expert_rows), _np(m.expert_count)
    st = m.drop_stats()
    assert st["kept"] + st["dropped_send"] + st["dropped_recv"] == cfg.T * cfg.top_k
    flips = np.nonzero((idx != ref["idx"]).any(axis=1))[0]
    report["routing_flips"] = int(flips.size)
    if flips.size == 0:
        d = ref["disp"]
        assert (slot_of == d["slot_of"]).all()
        assert (drop == d["drop"]).all()
        assert (rows == d["expert_rows"]).all()
        assert (count == d["count"]).all()
        for key in ("kept", "dropped_send", "dropped_recv"):
            assert st[key] == d["stats"][key], key
        assert st["max_send_fill"] == int(d["send_fill"].max(initial=0))
        assert st["max_expert_rows"] == int(d["count"].max(initial=0))
        tags = _np(m.pool_tags())
        np.testing.assert_array_equal(tags, ref["tags"])
    else:
        t0 = int(flips[0])
        d = ref["disp"]
        assert (slot_of[:t0] == d["slot_of"][:t0]).all()
        assert (drop[:t0] == d["drop"][:t0]).all()
        dispatch_rules_hold(idx, slot_of, drop, rows, count, p)
    # the pack is a copy: every filled payload row is its token's z row
    tags = _np(m.pool_tags())
    filled = tags[:, 0] >= 0
    zg = m.z.view(torch.int16).cpu().numpy()
    payload = m.pool[:, : cfg.d_latent].cpu().numpy()
    assert (payload[filled] == zg[tags[filled, 1]]).all()
    assert ((tags[filled, 0][:, None] == idx[tags[filled, 1]]).any(axis=1)).all()
    # experts: rows computed on both sides that carry the same (expert, token, rank)
    Yg = m.ypool.float().cpu().numpy().astype(np.float64)
    computed = set(slot_of[slot_of >= 0].tolist())
    same_tag = (tags == ref["tags"]).all(axis=1)
    ok_rows = [r for r in ref["Y"] if r in computed and same_tag[r]]
    if ok_rows:
        check_close("Y", Yg[ok_rows], np.stack([ref["Y"][r] for r in ok_rows]), report)
    # combine, shared, output: tokens whose routing and drop decisions agree
    tok = np.nonzero((idx == ref["idx"]).all(axis=1) & (drop == ref["disp"]["drop"]).all(axis=1))[0]
    report["compared_tokens"] = int(tok.size)
    check_close("c", _np(m.c)[tok], ref["c"][tok], report)
    if cfg.n_shared:
        check_close("a", _np(m.a), ref["a"], report)
    check_close("out", _np(m.out)[tok], ref["out"][tok], report)
    return m, ref, report


def test_tiny_layer_matches_oracle():
    cfg = wl.TINY
    _, _, rep = compare_full(cfg, wl.make_inputs(cfg, "cpu"))
    print(rep)


@pytest.mark.parametrize("kw", [
    dict(),                                               # the tiny workload, seed 0
    dict(seed=11, T=200, n_ranks=4, d_model=136, d_latent=72, h_expert=136, h_shared=72),
    dict(seed=12, top_k=1),
    dict(seed=13, n_waves=1),
    dict(seed=14, n_waves=2, n_experts=16),
    dict(seed=15, n_shared=0),
    dict(seed=16, n_shared=3, h_shared=64),
    dict(seed=17, cf_send=float("inf"), cf_recv=float("inf")),
    dict(seed=18, cf_send=0.3, cf_recv=0.5),
    dict(seed=19, top_k=6, cf_send=1.0, cf_recv=1.0),
    dict(seed=20, T=1024, n_ranks=8, n_experts=48, top_k=4, d_model=256, d_latent=128,
         h_expert=256, h_shared=128),
    dict(seed=25, n_experts=768, top_k=2),      # E > 384: router GEMM + separate top-k kernel
    dict(seed=26, n_experts=48, top_k=20),      # k > 16: same fallback
    dict(seed=27, n_experts=384, n_ranks=4, top_k=16, cf_send=2.0, cf_recv=2.0),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()) or "tiny")
def test_small_variants_match_oracle(kw):
    cfg = wl.TINY.with_(**kw)
    compare_full(cfg, wl.make_inputs(cfg, "cpu"))


def test_skewed_bias_all_on_few_experts():
    """A Zipf prior plus a large bias on expert 0: capacity drops dominate."""
    cfg = wl.TINY.with_(seed=21, bias_kind="zipf")
    inp = wl.make_inputs(cfg, "cpu")
    inp["bias"] = inp["bias"].clone()
    inp["bias"][0] += 50.0
    m, ref, rep = compare_full(cfg, inp)
    st = m.drop_stats()
    assert st["dropped_send"] + st["dropped_recv"] > 0
    assert int(_np(m.expert_count)[0]) == min(ref["plan"].c_recv, int(ref["disp"]["recv_demand"][0]))


def test_exact_arithmetic_routing_is_bit_exact():
    """Small-integer inputs make every fp32 logit exact on both sides, so the
    routing (ties broken to the lower id) and the whole dispatch must match
    bit for bit with no near-tie exceptions."""
    cfg = wl.TINY.with_(seed=22, T=512, n_ranks=4, top_k=4)
    inp = wl.make_inputs(cfg, "cpu")
    g = torch.Generator().manual_seed(5)
    inp["x"] = (torch.randint(-4, 5, inp["x"].shape, generator=g) / 8.0).to(torch.bfloat16)
    inp["Wr"] = (torch.randint(-4, 5, inp["Wr"].shape, generator=g) / 64.0).to(torch.bfloat16)
    ref = O.layer(cfg, _host_inputs(inp))
    m = run_gpu(cfg, inp)
    np.testing.assert_array_equal(_np(m.logits), ref["logits"])
    np.testing.assert_array_equal(_np(m.idx), ref["idx"])
    np.testing.assert_array_equal(_np(m.tie), ref["tie"])
    np.testing.assert_array_equal(_np(m.slot_of), ref["disp"]["slot_of"])
    np.testing.assert_array_equal(_np(m.drop), ref["disp"]["drop"])
    np.testing.assert_array_equal(_np(m.expert_rows), ref["disp"]["expert_rows"])
    np.testing.assert_array_equal(_np(m.pool_tags()), ref["tags"])
    assert (ref["tie"] != 0).any()      # exact ties happen and are broken the same way


def test_mid_layer_matches_oracle():
    cfg = wl.MID
    _, _, rep = compare_full(cfg, wl.make_inputs(cfg, "cpu"))
    print(rep)


def test_empty_batch():
    cfg = wl.TINY.with_(T=0)
    inp = wl.make_inputs(cfg, "cpu")
    m = PooledWaveMoE(cfg, inp, "cuda")
    m.forward(inp["x"].cuda())
    torch.cuda.synchronize()
    st = m.drop_stats()
    assert st["assignments"] == 0 and st["kept"] == 0 and st["status"] == 0
    assert int(m.status.item()) == 0


def test_results_are_deterministic():
    cfg = wl.TINY.with_(seed=23, T=1024, n_ranks=8, n_experts=48, top_k=8)
    inp = wl.make_inputs(cfg, "cpu")
    m = PooledWaveMoE(cfg, inp, "cuda")
    x = inp["x"].cuda()
    outs = []
    for _ in range(2):
        m.forward(x)
        torch.cuda.synchronize()
        # bit patterns (rows no expert writes hold whatever was there, NaNs included)
        outs.append([t.clone().view(torch.uint8) for t in (m.idx, m.slot_of, m.drop,
                                                            m.expert_rows, m.pool, m.ypool,
                                                            m.out)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_host_pipeline_matches_forward():
    """Host batches through the overlapped-copy runner give the same bits as
    the plain forward on device-resident inputs."""
    from moe_routing_capacity_gb300.layer import HostPipeline
    cfg = wl.TINY.with_(seed=24, T=512, n_ranks=4)
    inp = wl.make_inputs(cfg, "cpu")
    m = PooledWaveMoE(cfg, inp, "cuda")
    g = torch.Generator().manual_seed(9)
    xs = [torch.randn(cfg.T, cfg.d_model, generator=g).to(torch.bfloat16).pin_memory()
          for _ in range(5)]
    want = []
    for xh in xs:
        m.forward(xh.cuda())
        torch.cuda.synchronize()
        want.append((m.out.cpu().clone(), m.stats.cpu().clone()))
    pipe = HostPipeline(m, depth=2)
    outs = [torch.empty(cfg.T, cfg.d_model, dtype=torch.bfloat16).pin_memory() for _ in xs]
    sts = [torch.empty(m.stats.numel(), dtype=torch.int64).pin_memory() for _ in xs]
    for xh, oh, sh in zip(xs, outs, sts):
        pipe.submit(xh, oh, sh)
    pipe.synchronize()
    for (wo, ws), oh, sh in zip(want, outs, sts):
        assert torch.equal(oh.view(torch.int16), wo.view(torch.int16))
        assert torch.equal(sh, ws)


@pytest.mark.parametrize("E", [48, 384, 768])
def test_route_project_equals_separate_calls(E):
    """The one-pass router + latent projection gives the same bits as
    moe_router_topk followed by moe_latent_proj."""
    cfg = wl.TINY.with_(seed=28, T=640, n_ranks=4, d_model=384, d_latent=512, n_experts=E,
                        top_k=8 if E > 48 else 4, bias_kind="zipf")
    inp = wl.make_inputs(cfg, "cuda")
    a = PooledWaveMoE(cfg, inp, "cuda")
    b = PooledWaveMoE(cfg, inp, "cuda")
    x = inp["x"]
    a.route_and_latent(x)
    b.route(x)
    b.latent(x)
    torch.cuda.synchronize()
    for name in ("logits", "idx", "gate_w", "tie", "z"):
        ta, tb = getattr(a, name), getattr(b, name)
        assert torch.equal(ta.view(torch.uint8), tb.view(torch.uint8)), name
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
