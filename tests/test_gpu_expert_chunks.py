"""The paired expert products at every chunk and group boundary.

A routing is built so that chosen experts receive exactly the given numbers
of rows.  With c_recv = 393 (one group an expert): 0, 1, 7, 8, 9, 15, 16,
17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300 and 393 rows,
chunks of every width class from 16 to 256, one and two chunks a group,
widths rounded up from one row past a multiple of 16.  With c_recv = 2356:
417, 431, 448, 832, 833 and 1100 rows, two and three groups an expert.
The routing goes straight to moe_dispatch_pooled (no router), once writing
the per-expert bank and once not, then to moe_expert_ffn_grouped, which takes
the paired path from the bank or gathers the rows from the pool.  Both must
give the same bits in every computed row, and the first and last row of each
expert must match the oracle's SwiGLU expert on the same input row.
"""
import numpy as np
import pytest
import torch

import oracle as O
from moe_routing_capacity_gb300 import abi
from moe_routing_capacity_gb300 import workloads as wl

from helpers import check_close

pytestmark = pytest.mark.gpu

# widths that take the paired path (L a multiple of 256, H of 128)
ONE_GROUP = (wl.LayerConfig("chunks", T=4096, d_model=256, d_latent=256, n_experts=24, n_ranks=4,
                            top_k=2, n_waves=3, n_shared=1, h_expert=128, h_shared=128, seed=9),
             [0, 1, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300,
              393])
MANY_GROUPS = (wl.LayerConfig("groups", T=8192, d_model=256, d_latent=256, n_experts=8, n_ranks=4,
                              top_k=2, n_waves=2, n_shared=1, h_expert=128, h_shared=128, seed=9),
               [417, 431, 448, 832, 833, 1100])


def _routing(rng, cfg, targets):
    """idx [T, 2] whose receiver-kept counts are `targets` for the first
    experts; the last two experts take the remaining assignments (capped by
    the sender)."""
    T, k, S, E = cfg.T, cfg.top_k, cfg.n_ranks, cfg.n_experts
    T_s = T // S
    per_src = []
    for s in range(S):
        a = []
        for e, n in enumerate(targets):
            a += [e] * (n // S + (1 if s < n % S else 0))
        fill = T_s * k - len(a)
        a += [E - 2 + (i % 2) for i in range(fill)]
        a = np.array(a)
        rng.shuffle(a)
        pairs = a.reshape(T_s, k)
        # distinct experts within a token: swap a clashing second choice
        # with a later token's second choice
        for t in range(T_s):
            if pairs[t, 0] == pairs[t, 1]:
                for u in range(T_s):
                    if u != t and pairs[u, 1] != pairs[t, 0] and pairs[u, 0] != pairs[t, 1]:
                        pairs[t, 1], pairs[u, 1] = pairs[u, 1], pairs[t, 1]
                        break
        per_src.append(pairs)
    idx = np.concatenate(per_src).astype(np.int32)
    assert (idx[:, 0] != idx[:, 1]).all()
    return idx


def _run(cfg, idx, z, w, bank):
    p = abi.plan(cfg)
    dev = "cuda"
    T, k, E, L = cfg.T, cfg.top_k, cfg.n_experts, cfg.d_latent
    ws = torch.empty(max(1, p.ws_dispatch_bytes), dtype=torch.uint8, device=dev)
    o = dict(pool=torch.zeros(p.pool_rows, p.pool_row_bytes // 2, dtype=torch.int16, device=dev),
             slot_of=torch.zeros(T, k, dtype=torch.int32, device=dev),
             drop=torch.zeros(T, k, dtype=torch.uint8, device=dev),
             expert_rows=torch.zeros(E, p.c_recv, dtype=torch.int32, device=dev),
             expert_count=torch.zeros(E, dtype=torch.int32, device=dev),
             stats=torch.zeros(abi.STATS_WORDS, dtype=torch.int64, device=dev))
    b = torch.empty(E, p.c_recv, L, dtype=torch.bfloat16, device=dev) if bank else None
    abi.dispatch_pooled(cfg, z, torch.from_numpy(idx).cuda(), ws, o["pool"], o["slot_of"],
                        o["drop"], o["expert_rows"], o["expert_count"], o["stats"], bank=b)
    ws_ffn = torch.empty(p.ws_ffn_bytes, dtype=torch.uint8, device=dev)
    ypool = torch.zeros(p.pool_rows, L, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    abi.expert_ffn_grouped(cfg, o["pool"], o["expert_rows"], o["expert_count"], w["Wg"], w["Wu"],
                           w["Wd"], ws_ffn, ypool, status, bank=b)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o["ypool"] = ypool
    return o


@pytest.mark.parametrize("case", [ONE_GROUP, MANY_GROUPS], ids=["one_group", "many_groups"])
def test_chunk_boundaries(case):
    cfg, targets = case
    rng = np.random.default_rng(3)
    idx = _routing(rng, cfg, targets)
    inp = wl.make_inputs(cfg, "cuda")
    z = torch.randn(cfg.T, cfg.d_latent, generator=torch.Generator(device="cuda").manual_seed(4),
                    device="cuda").to(torch.bfloat16)
    a = _run(cfg, idx, z, inp, bank=True)
    b = _run(cfg, idx, z, inp, bank=False)
    d = O.dispatch(idx, O.make_plan(cfg))
    cnt = a["expert_count"].cpu().numpy()
    assert cnt[:len(targets)].tolist() == targets, cnt
    assert (cnt == d["count"]).all()
    assert (a["expert_rows"].cpu().numpy() == d["expert_rows"]).all()
    for n in ("slot_of", "drop", "expert_rows", "expert_count"):
        assert torch.equal(a[n], b[n]), n
    kept = a["slot_of"][a["slot_of"] >= 0].long()
    assert torch.equal(a["ypool"][kept].view(torch.int16), b["ypool"][kept].view(torch.int16))
    # against the oracle: the first and the last row of each expert with rows,
    # the input rows taken from z through the oracle's own dispatch
    token_of = {int(r): int(t) for (t, j), r in np.ndenumerate(d["send_row"]) if r >= 0}
    zh = z.double().cpu().numpy()
    got, want = [], []
    for e in range(cfg.n_experts):
        n = int(d["count"][e])
        if n == 0:
            continue
        sel = sorted({int(d["expert_rows"][e, 0]), int(d["expert_rows"][e, n - 1])})
        X = zh[[token_of[r] for r in sel]]
        want.append(O.expert_ffn(X, inp["Wg"][e].float().cpu().numpy(),
                                 inp["Wu"][e].float().cpu().numpy(),
                                 inp["Wd"][e].float().cpu().numpy()))
        got.append(a["ypool"][torch.tensor(sel, device="cuda")].double().cpu().numpy())
    check_close("Y", np.concatenate(got), np.concatenate(want))
