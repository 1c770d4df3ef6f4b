"""The expert products on CTA pairs with each expert's rows on the MMA's N
axis, fed from the per-expert bank that the dispatch's pack writes.

Checked against the oracle element by element on a 4096-token layer whose
widths take that path (L = 256, H = 128): uniform routing (experts of
281-393 rows, each split into two chunks), and a Zipf prior with some
experts ruled out (experts at the receiver cap, experts with a handful of
rows, experts with none).  The bank itself is compared with the pool rows
it groups, and the whole layer with the path that gathers each expert's
rows from the pool, for each pool-fill schedule.
"""
import pytest
import torch

from moe_routing_capacity_gb300 import workloads as wl

from test_gpu_parity import compare_full, run_gpu

pytestmark = pytest.mark.gpu

# widths whose expert products take the bank path; ~341 rows an expert before drops
PAIRS = wl.LayerConfig("pairs", T=4096, d_model=256, d_latent=256, n_experts=24, n_ranks=4,
                       top_k=2, n_waves=3, n_shared=1, h_expert=128, h_shared=128, seed=5)


def _inputs(kind):
    cfg = PAIRS
    inp = wl.make_inputs(cfg, "cpu")
    if kind == "skew":
        b = wl.zipf_bias(cfg.n_experts, 1.2)
        b[[3, 10, 17]] = -1.0e4          # three experts that receive nothing
        inp["bias"] = b
    return cfg, inp


def _bank_matches_pool(m, cfg):
    """bank[e][r] is the payload of pool row expert_rows[e][r], r < count."""
    L = cfg.d_latent
    rows = m.expert_rows.long()
    cnt = m.expert_count.long()
    r_idx = torch.arange(rows.shape[1], device=rows.device)[None, :]
    valid = r_idx < cnt[:, None]
    pool_payload = m.pool[:, :L]
    got = m.bank.view(torch.int16)[valid]
    want = pool_payload[rows[valid]]
    assert torch.equal(got, want)


@pytest.mark.parametrize("kind", ["uniform", "skew"])
def test_bank_path_matches_oracle(kind):
    cfg, inp = _inputs(kind)
    m, ref, rep = compare_full(cfg, inp, expert_bank=True)
    assert m.bank is not None
    cnt = m.expert_count.cpu().numpy()
    if kind == "uniform":
        assert (cnt > 256).sum() >= cfg.n_experts // 2, cnt   # most experts in two chunks
    else:
        p = ref["plan"]
        # experts at the receiver cap, with no rows, and with fewer than 128
        # (chunks narrower than the full-rate MMA width)
        assert (cnt == p.c_recv).any() and (cnt == 0).sum() == 3 and (cnt[cnt > 0] < 128).any(), cnt
    _bank_matches_pool(m, cfg)
    print(kind, rep)


@pytest.mark.parametrize("pipeline", [None, "shared"])
@pytest.mark.parametrize("kind", ["uniform", "skew"])
def test_bank_path_equals_gathered_rows(kind, pipeline):
    cfg, inp = _inputs(kind)
    a = run_gpu(cfg, inp, expert_bank=True, pipeline=pipeline)
    b = run_gpu(cfg, inp, expert_bank=False, pipeline=pipeline)
    assert a.bank is not None and b.bank is None
    _bank_matches_pool(a, cfg)
    kept = a.slot_of[a.slot_of >= 0].long()
    for name in ("slot_of", "drop", "expert_rows", "expert_count"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert torch.equal(a.ypool[kept].view(torch.int16), b.ypool[kept].view(torch.int16))
    for name in ("c", "out"):
        assert torch.equal(getattr(a, name).view(torch.int16), getattr(b, name).view(torch.int16)), name


def test_mid_bank_path_equals_gathered_rows():
    cfg = wl.MID
    inp = wl.make_inputs(cfg, "cpu")
    a = run_gpu(cfg, inp, expert_bank=True)
    b = run_gpu(cfg, inp, expert_bank=False)
    _bank_matches_pool(a, cfg)
    kept = a.slot_of[a.slot_of >= 0].long()
    assert torch.equal(a.ypool[kept].view(torch.int16), b.ypool[kept].view(torch.int16))
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_same_tensor_for_gate_and_up():
    """One tensor passed as both Wg and Wu.  The gate/up product reads the two
    through one tensor map that interleaves them by 16 rows, with the distance
    between the tensors as a stride; at distance 0 no such map exists and the
    product takes the one-chunk-a-tile kernel with two weight boxes a stage.
    It must still match the oracle, and the path that gathers the rows from
    the pool bit for bit."""
    cfg = PAIRS
    inp = wl.make_inputs(cfg, "cuda")
    inp["Wu"] = inp["Wg"]
    # h = silu(g) g is never negative, so Y grows past the range where one
    # bf16 step of Y stays within c's tolerance; a power-of-two scale of Wd
    # (exact in bf16) keeps Y in the usual range
    inp["Wd"] = inp["Wd"] * 0.25
    m, ref, rep = compare_full(cfg, inp, expert_bank=True)
    assert m.w["Wg"].data_ptr() == m.w["Wu"].data_ptr()
    b = run_gpu(cfg, inp, expert_bank=False)
    kept = m.slot_of[m.slot_of >= 0].long()
    assert torch.equal(m.ypool[kept].view(torch.int16), b.ypool[kept].view(torch.int16))
    print(rep)


def _train_grads(cfg, inp, bank, pipeline):
    from moe_routing_capacity_gb300.layer import PooledWaveMoE
    m = PooledWaveMoE(cfg, inp, "cuda", pipeline=pipeline, expert_bank=bank)
    x = inp["x"].cuda()
    m.forward(x)
    g = torch.Generator().manual_seed(11)
    dout = torch.randn(cfg.T, cfg.d_model, generator=g).to(torch.bfloat16).cuda()
    grads = m.backward(x, dout)
    torch.cuda.synchronize()
    assert int(m.status.item()) == 0
    return m, {k: v.clone() for k, v in grads.items()}


@pytest.mark.parametrize("kind", ["uniform", "skew"])
def test_backward_reads_x_from_the_bank(kind):
    """The backward with the forward's bank as its X (only the padding rows
    zeroed) gives the gradients of the one that copies X out of the pool
    rows, bit for bit; the bank's kept rows are left as the forward wrote
    them and its padding rows are zero."""
    cfg, inp = _inputs(kind)
    mb, ga = _train_grads(cfg, inp, True, "shared")
    _, gb = _train_grads(cfg, inp, False, None)
    for k in ga:
        w = torch.int32 if ga[k].dtype == torch.float32 else torch.int16
        assert torch.equal(ga[k].view(w), gb[k].view(w)), k
    _bank_matches_pool(mb, cfg)
    cnt = mb.expert_count.long()
    r_idx = torch.arange(mb.bank.shape[1], device=cnt.device)[None, :]
    pad = r_idx >= cnt[:, None]
    assert int(pad.sum()) > 0
    assert (mb.bank.view(torch.int16)[pad] == 0).all()
