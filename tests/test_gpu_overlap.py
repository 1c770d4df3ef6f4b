"""The overlapped dispatch paths against the plain sequence of calls.

"waves" (moe_dispatch_expert_waves): the later waves' payload rows are
copied into the pools inside the expert gate/up launch while wave 0's
experts compute.  "shared" (moe_dispatch_shared_overlap): every payload row
is copied by extra warps of the shared experts' gate/up launch.  Either way
the results must be those of moe_dispatch_pooled, moe_expert_ffn_grouped
and moe_combine bit for bit -- pool tags of every row, payloads of every
filled row, sender and receiver decisions, row lists, drop counts, the
computed expert rows, the shared activations and the layer output -- and
must meet the oracle like the plain path does.
"""
import numpy as np
import pytest
import torch

from moe_routing_capacity_gb300 import workloads as wl
from moe_routing_capacity_gb300.layer import PooledWaveMoE

from test_gpu_parity import compare_full

pytestmark = pytest.mark.gpu


def _bits(t):
    t = t.detach()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.view(torch.int16)
    elif t.dtype == torch.float32:
        t = t.view(torch.int32)
    return t.cpu().numpy()


PIPES = ["waves", "shared"]


def run_both(cfg, inp, pipeline, steps=1):
    x = inp["x"].cuda()
    plain = PooledWaveMoE(cfg, inp, "cuda")
    piped = PooledWaveMoE(cfg, inp, "cuda", pipeline=pipeline)
    for _ in range(steps):
        plain.forward(x)
        piped.forward(x)
    torch.cuda.synchronize()
    for m in (plain, piped):
        assert int(m.status.item()) == 0, "device status word set"
        assert m.drop_stats()["status"] == 0
    return plain, piped


def assert_same(cfg, plain, piped):
    L = cfg.d_latent
    for name in ("idx", "slot_of", "drop", "expert_rows", "expert_count", "z"):
        np.testing.assert_array_equal(_bits(getattr(piped, name)), _bits(getattr(plain, name)),
                                      err_msg=name)
    assert piped.drop_stats() == plain.drop_stats()
    tags = _bits(plain.pool_tags())
    np.testing.assert_array_equal(_bits(piped.pool_tags()), tags, err_msg="tags")
    filled = tags[:, 0] >= 0
    np.testing.assert_array_equal(_bits(piped.pool[:, :L])[filled], _bits(plain.pool[:, :L])[filled],
                                  err_msg="payload rows")
    slot = _bits(plain.slot_of)
    rows = np.unique(slot[slot >= 0])
    if rows.size:
        np.testing.assert_array_equal(_bits(piped.ypool)[rows], _bits(plain.ypool)[rows],
                                      err_msg="expert rows of ypool")
    np.testing.assert_array_equal(_bits(piped.c), _bits(plain.c), err_msg="c")
    if cfg.n_shared:
        np.testing.assert_array_equal(_bits(piped.a), _bits(plain.a), err_msg="a")
    np.testing.assert_array_equal(_bits(piped.out), _bits(plain.out), err_msg="out")


@pytest.mark.parametrize("pipeline", PIPES)
@pytest.mark.parametrize("kw", [
    dict(),                                             # tiny: 3 waves of 2 experts
    dict(seed=13, n_waves=1),                           # one wave: nothing to overlap
    dict(seed=14, n_waves=2, n_experts=16),             # 2 waves
    dict(seed=30, n_waves=6),                           # one expert a wave
    dict(seed=15, n_shared=0),                          # no shared experts to overlap with
    dict(seed=16, n_shared=3, h_shared=64),
    dict(seed=11, T=200, n_ranks=4, d_model=136, d_latent=72, h_expert=136, h_shared=72),
    dict(seed=18, cf_send=0.3, cf_recv=0.5),            # heavy drops on both sides
    dict(seed=17, cf_send=float("inf"), cf_recv=float("inf")),
    dict(seed=27, n_experts=384, n_ranks=4, top_k=16, cf_send=2.0, cf_recv=2.0),
    dict(seed=20, T=1024, n_ranks=8, n_experts=48, top_k=4, d_model=256, d_latent=128,
         h_expert=256, h_shared=128),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()) or "tiny")
def test_overlap_equals_separate_calls(kw, pipeline):
    cfg = wl.TINY.with_(**kw)
    plain, piped = run_both(cfg, wl.make_inputs(cfg, "cpu"), pipeline)
    assert_same(cfg, plain, piped)


@pytest.mark.parametrize("pipeline", PIPES)
def test_overlap_skew_empty_experts(pipeline):
    """Zipf prior plus a large bias on expert 0: most experts of the later
    waves receive nothing, some CTAs have no tile at all."""
    cfg = wl.TINY.with_(seed=21, bias_kind="zipf")
    inp = wl.make_inputs(cfg, "cpu")
    inp["bias"] = inp["bias"].clone()
    inp["bias"][0] += 50.0
    plain, piped = run_both(cfg, inp, pipeline)
    assert_same(cfg, plain, piped)


@pytest.mark.parametrize("pipeline", PIPES)
def test_overlap_empty_batch(pipeline):
    cfg = wl.TINY.with_(T=0)
    inp = wl.make_inputs(cfg, "cpu")
    m = PooledWaveMoE(cfg, inp, "cuda", pipeline=pipeline)
    m.forward(inp["x"].cuda())
    torch.cuda.synchronize()
    st = m.drop_stats()
    assert st["assignments"] == 0 and st["status"] == 0
    assert int(m.status.item()) == 0


@pytest.mark.parametrize("pipeline", PIPES)
def test_overlap_tiny_matches_oracle(pipeline):
    cfg = wl.TINY
    compare_full(cfg, wl.make_inputs(cfg, "cpu"), pipeline=pipeline)


@pytest.mark.parametrize("pipeline", PIPES)
def test_overlap_mid_matches_oracle(pipeline):
    cfg = wl.MID
    compare_full(cfg, wl.make_inputs(cfg, "cpu"), pipeline=pipeline)


@pytest.mark.parametrize("pipeline", PIPES)
@pytest.mark.parametrize("name", ["mid", "full", "long", "skew"])
def test_overlap_equals_separate_calls_large(name, pipeline):
    """At the bench's size, repeated steps (counters reset each step)."""
    cfg = wl.CONFIGS[name]
    plain, piped = run_both(cfg, wl.make_inputs(cfg, "cuda"), pipeline, steps=2)
    assert_same(cfg, plain, piped)


@pytest.mark.parametrize("pipeline", PIPES)
def test_overlap_graph_replay_equals_eager(pipeline):
    cfg = wl.MID
    inp = wl.make_inputs(cfg, "cuda")
    m = PooledWaveMoE(cfg, inp, "cuda", pipeline=pipeline)
    x_buf = inp["x"].clone()
    out_g = torch.empty(cfg.T, cfg.d_model, dtype=torch.bfloat16, device="cuda")
    g = m.capture(x_buf, out_g)
    gen = torch.Generator(device="cuda").manual_seed(12)
    for step in range(2):
        x_new = torch.randn(cfg.T, cfg.d_model, generator=gen, device="cuda").to(torch.bfloat16)
        x_buf.copy_(x_new)
        g.replay()
        torch.cuda.synchronize()
        got = out_g.clone()
        want = m.forward(x_new).clone()
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), step
        assert int(m.status.item()) == 0
