"""GPU parity of the dropless ragged variant (the pages' fallback when drops
stay too high): the CUDA path against the oracle's ragged layer."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_routing_capacity_gb300 import workloads as wl
from moe_routing_capacity_gb300.layer import PooledWaveMoE

from helpers import LOGIT_ATOL, check_close, ragged_rules_hold

pytestmark = pytest.mark.gpu


def _host(inp):
    return {k: (v.float().cpu().numpy() if v is not None else None) for k, v in inp.items()}


def run(cfg, inp, pipeline=None):
    m = PooledWaveMoE(cfg, inp, "cuda", dropless=True, pipeline=pipeline)
    m.forward(inp["x"].cuda())
    torch.cuda.synchronize()
    assert int(m.status.item()) == 0
    st = m.drop_stats()
    assert st["status"] == 0 and st["kept"] == cfg.T * cfg.top_k
    assert st["dropped_send"] == 0 and st["dropped_recv"] == 0
    return m


def compare(cfg, inp, pipeline=None):
    ref = O.layer_ragged(cfg, _host(inp))
    m = run(cfg, inp, pipeline)
    idx = m.idx.cpu().numpy()
    assert np.abs(m.logits.cpu().numpy() - ref["logits"]).max() <= LOGIT_ATOL
    clear = ref["tie"] == 0
    assert (idx[clear] == ref["idx"][clear]).all()
    slot_of = m.slot_of.cpu().numpy()
    eoff, erows = m.expert_offsets.cpu().numpy(), m.expert_rows.cpu().numpy()
    count = m.expert_count.cpu().numpy()
    assert (m.drop.cpu().numpy() == 0).all()
    d = ref["disp"]
    if (idx == ref["idx"]).all():
        assert (slot_of == d["slot_of"]).all()
        assert (eoff == d["expert_offsets"]).all() and (erows == d["expert_rows"]).all()
        assert (count == d["count"]).all()
        np.testing.assert_array_equal(m.pool_tags().cpu().numpy(), ref["tags"])
    else:
        ragged_rules_hold(idx, slot_of, eoff, erows, count, ref["plan"])
    tags = m.pool_tags()
    assert torch.equal(m.pool_payload(), m.z[tags[:, 1].long()])
    same = (idx == ref["idx"]).all(axis=1)
    rows = [int(slot_of[t, j]) for t in np.nonzero(same)[0] for j in range(cfg.top_k)]
    orows = [int(d["slot_of"][t, j]) for t in np.nonzero(same)[0] for j in range(cfg.top_k)]
    Yg = m.ypool.float().cpu().numpy().astype(np.float64)
    check_close("Y", Yg[rows], np.stack([ref["Y"][r] for r in orows]))
    check_close("c", m.c.float().cpu().numpy()[same], ref["c"][same])
    check_close("out", m.out.float().cpu().numpy()[same], ref["out"][same])
    return m


@pytest.mark.parametrize("kw", [
    dict(),
    dict(seed=41, T=200, n_ranks=4, d_model=136, d_latent=72, h_expert=136, h_shared=72),
    dict(seed=42, top_k=6),
    dict(seed=43, n_waves=1, top_k=1),
    dict(seed=44, bias_kind="zipf"),              # heavily skewed: big experts, nothing dropped
    dict(seed=45, T=1024, n_ranks=8, n_experts=48, top_k=8, d_model=256, d_latent=128,
         h_expert=256, h_shared=128),
], ids=lambda kw: ",".join(f"{k}={v}" for k, v in kw.items()) or "tiny")
def test_ragged_small_variants(kw):
    cfg = wl.TINY.with_(**kw)
    compare(cfg, wl.make_inputs(cfg, "cpu"))


def test_ragged_mid():
    compare(wl.MID, wl.make_inputs(wl.MID, "cpu"))


def test_ragged_equals_capped_without_caps():
    """With unbounded factors the capped pools drop nothing either, and each
    expert sees the same rows in the same order: identical bits."""
    cfg = wl.TINY.with_(seed=46, cf_send=float("inf"), cf_recv=float("inf"))
    inp = wl.make_inputs(cfg, "cpu")
    a = PooledWaveMoE(cfg, inp, "cuda")
    b = PooledWaveMoE(cfg, inp, "cuda", dropless=True)
    x = inp["x"].cuda()
    a.forward(x)
    b.forward(x)
    torch.cuda.synchronize()
    assert a.drop_stats()["kept"] == cfg.T * cfg.top_k
    assert torch.equal(a.c.view(torch.int16), b.c.view(torch.int16))
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_ragged_empty_batch():
    cfg = wl.TINY.with_(T=0)
    inp = wl.make_inputs(cfg, "cpu")
    m = PooledWaveMoE(cfg, inp, "cuda", dropless=True)
    m.forward(inp["x"].cuda())
    torch.cuda.synchronize()
    assert m.drop_stats()["assignments"] == 0
    assert (m.expert_offsets.cpu() == 0).all() and (m.expert_count.cpu() == 0).all()


@pytest.mark.parametrize("name", ["full", "skew"])
def test_ragged_full_size_sampled(name):
    cfg = wl.CONFIGS[name]
    inp = wl.make_inputs(cfg, "cuda")
    m = run(cfg, inp)
    p = O.make_plan(cfg)
    xh = inp["x"].double().cpu().numpy()
    bias = inp["bias"].cpu().numpy() if inp["bias"] is not None else None
    l32 = O.router_logits(xh, inp["Wr"].double().cpu().numpy(), bias)
    idx_o, w_o, tie_o = O.router_topk(l32, cfg.top_k)
    idx = m.idx.cpu().numpy()
    assert (idx[tie_o == 0] == idx_o[tie_o == 0]).all()
    d = O.dispatch_ragged(idx_o, p)
    slot_of = m.slot_of.cpu().numpy()
    eoff, erows = m.expert_offsets.cpu().numpy(), m.expert_rows.cpu().numpy()
    if (idx == idx_o).all():
        assert (slot_of == d["slot_of"]).all() and (erows == d["expert_rows"]).all()
        assert (eoff == d["expert_offsets"]).all()
    else:
        t0 = int(np.nonzero((idx != idx_o).any(axis=1))[0][0])
        # blocks before the first flipped token's own block are unaffected only
        # in count, so check the rules for the GPU's routing instead
        ragged_rules_hold(idx, slot_of, eoff, erows, m.expert_count.cpu().numpy(), p)
    # sampled tokens, one by one
    rng = np.random.default_rng(cfg.seed)
    toks = [int(t) for t in rng.choice(cfg.T, 16, replace=False) if (idx[t] == idx_o[t]).all()]
    W_ld = inp["W_ld"].double().cpu().numpy()
    z_o = O.latent_down(xh[toks], W_ld)
    c_o, Yg, Yo = [], [], []
    for i, t in enumerate(toks):
        acc = np.zeros(cfg.d_latent)
        for j in range(cfg.top_k):
            e = int(idx_o[t, j])
            y = O.expert_ffn(z_o[i:i + 1], inp["Wg"][e].double().cpu().numpy(),
                             inp["Wu"][e].double().cpu().numpy(),
                             inp["Wd"][e].double().cpu().numpy())[0]
            Yo.append(y)
            Yg.append(m.ypool[int(slot_of[t, j])].double().cpu().numpy())
            acc = acc + w_o[t, j] * y
        c_o.append(acc)
    check_close("Y", np.stack(Yg), np.stack(Yo))
    c_o = O.bf16_round(np.stack(c_o))
    check_close("c", m.c[toks].double().cpu().numpy(), c_o)
    a_o = O.shared_act(xh[toks], inp["Wsg"].double().cpu().numpy(), inp["Wsu"].double().cpu().numpy())
    out_o = O.output(c_o, a_o, inp["W_lu"].double().cpu().numpy(), inp["Wsd"].double().cpu().numpy())
    check_close("out", m.out[toks].double().cpu().numpy(), out_o)


# Widths the row-group expert kernels take (L a multiple of 256, H of 128);
# a Zipf bias gives experts of several hundred rows (two- and three-group
# experts) next to near-empty ones.
PAIR_SMALL = wl.LayerConfig("ragged-pair", T=3072, d_model=256, d_latent=256, n_experts=24,
                            n_ranks=4, top_k=2, n_waves=3, n_shared=1, h_expert=128,
                            h_shared=128, seed=47, bias_kind="zipf")


def _bank_vs_gathered(cfg, inp):
    x = inp["x"].cuda()
    a = PooledWaveMoE(cfg, inp, "cuda", dropless=True)
    b = PooledWaveMoE(cfg, inp, "cuda", dropless=True, expert_bank=False)
    a.forward(x)
    b.forward(x)
    torch.cuda.synchronize()
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
    assert a.bank is not None and b.bank is None
    # the bank holds each row of the flat row list's token in that order
    tok = a.pool_tags()[a.expert_rows.long(), 1].long()
    assert torch.equal(a.bank.view(torch.int16), a.z[tok].view(torch.int16))
    assert torch.equal(a.ypool.view(torch.int16), b.ypool.view(torch.int16))
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
    return a


@pytest.mark.parametrize("name", ["ragged-pair", "mid", "skew"])
def test_ragged_bank_equals_gathered(name):
    cfg = PAIR_SMALL if name == "ragged-pair" else wl.CONFIGS[name]
    m = _bank_vs_gathered(cfg, wl.make_inputs(cfg, "cuda"))
    counts = m.expert_count.cpu()
    if name != "mid":   # the skewed routings reach the multi-group experts
        assert int(counts.max()) > 416


def test_ragged_bank_small_parity():
    m = compare(PAIR_SMALL, wl.make_inputs(PAIR_SMALL, "cpu"))
    assert m.bank is not None


def test_ragged_bank_equals_capped_bank_without_caps():
    """Both layouts through the row-group kernels: with unbounded factors each
    expert's rows, their order and the row groups are the same, so are the
    bits."""
    cfg = PAIR_SMALL.with_(seed=48, cf_send=float("inf"), cf_recv=float("inf"))
    inp = wl.make_inputs(cfg, "cpu")
    a = PooledWaveMoE(cfg, inp, "cuda")
    b = PooledWaveMoE(cfg, inp, "cuda", dropless=True)
    assert a.bank is not None and b.bank is not None
    x = inp["x"].cuda()
    a.forward(x)
    b.forward(x)
    torch.cuda.synchronize()
    assert a.drop_stats()["kept"] == cfg.T * cfg.top_k
    assert torch.equal(a.c.view(torch.int16), b.c.view(torch.int16))
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def _state(m):
    """Every output of the dropless layer's forward, as raw bits."""
    out = {"out": m.out, "c": m.c, "a": m.a, "ypool": m.ypool, "slot_of": m.slot_of,
           "drop": m.drop, "expert_rows": m.expert_rows, "expert_offsets": m.expert_offsets,
           "expert_count": m.expert_count, "tags": m.pool_tags(), "payload": m.pool_payload()}
    if m.bank is not None:
        out["bank"] = m.bank
    return {k: v.contiguous().view(torch.uint8).clone() for k, v in out.items()}


@pytest.mark.parametrize("name", ["tiny", "ragged-pair", "mid", "full"])
def test_ragged_shared_schedule_equals_sequential(name):
    """The pack inside the shared experts' gate/up launch: every output of the
    dropless forward (decisions, row lists, offsets, pool rows and tags, the
    bank, Y, c, a, out) bit for bit as with the pack as a kernel of its own."""
    cfg = PAIR_SMALL if name == "ragged-pair" else wl.CONFIGS[name]
    inp = wl.make_inputs(cfg, "cuda" if name == "full" else "cpu")
    x = inp["x"].cuda()
    got = {}
    for pipe in (None, "shared"):
        m = PooledWaveMoE(cfg, inp, "cuda", dropless=True, pipeline=pipe)
        m.forward(x)
        torch.cuda.synchronize()
        assert int(m.status.item()) == 0 and m.drop_stats()["status"] == 0
        got[pipe] = _state(m)
        del m
    for k, v in got[None].items():
        assert torch.equal(v, got["shared"][k]), k


def test_ragged_shared_schedule_parity():
    m = compare(PAIR_SMALL, wl.make_inputs(PAIR_SMALL, "cpu"), pipeline="shared")
    assert m.bank is not None


@pytest.mark.parametrize("kw", [dict(n_shared=0), dict(T=0)], ids=["no-shared", "no-tokens"])
def test_ragged_shared_overlap_degenerate(kw):
    """Without shared experts, or without tokens, the overlapped dropless
    dispatch is the plain one: same outputs bit for bit."""
    from moe_routing_capacity_gb300 import abi
    cfg = wl.TINY.with_(seed=49, **kw)
    inp = wl.make_inputs(cfg, "cpu")
    x = inp["x"].cuda()
    got = []
    for overlap in (False, True):
        m = PooledWaveMoE(cfg, inp, "cuda", dropless=True)
        m.route_and_latent(x)
        if overlap:
            ns = cfg.n_shared
            abi.dispatch_ragged_shared_overlap(
                cfg, m.z, m.idx, m.ws_dispatch, m.pool, m.slot_of, m.drop, m.expert_offsets,
                m.expert_rows, m.expert_count, m.stats, x if ns else None,
                m.w["Wsg"] if ns else None, m.w["Wsu"] if ns else None, m.a if ns else None,
                m.status, bank=m.bank)
        else:
            m.dispatch()
        torch.cuda.synchronize()
        assert int(m.status.item()) == 0 and m.drop_stats()["status"] == 0
        st = {"offsets": m.expert_offsets, "count": m.expert_count, "stats": m.stats}
        if cfg.T:
            st.update(slot_of=m.slot_of, drop=m.drop, rows=m.expert_rows, tags=m.pool_tags(),
                      payload=m.pool_payload(), bank=m.bank)
        got.append({k: v.contiguous().view(torch.uint8).clone() for k, v in st.items()})
    for k in got[0]:
        assert torch.equal(got[0][k], got[1][k]), k
