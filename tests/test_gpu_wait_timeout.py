"""A bounded device wait running out, on the GPU, without breaking anything.

The wave-pipelined dispatch (moe_dispatch_expert_waves) has one wait that
spans CTAs: before a CTA's tensor cores start on the experts of wave w, its
row gather waits until every CTA of the cooperative launch has counted its
copies of wave w.  The checked build lets a test shorten that wait's limit
(moe_check_set_wave_wait_limit_ns).  Here the routing sends nothing to the
experts of wave 0, so every CTA's first tile belongs to wave 1 and its gather
has to wait for all 152 CTAs' copies; with a limit of 0 ns the wait runs
out on that legitimate work.  Nothing is broken on purpose: the data, the
launch and every other wait are the normal ones.

Checked: the launch returns (the stream synchronises), the status word holds
MOE_ETIMEOUT, no index check fired while the CTAs unwound, and once the limit
is back at its default the next forward on the same buffers equals a clean
run bit for bit.
"""
import os

import pytest
import torch

from moe_routing_capacity_gb300 import abi, build
from moe_routing_capacity_gb300 import workloads as wl
from moe_routing_capacity_gb300.layer import PooledWaveMoE

pytestmark = pytest.mark.gpu

DEFAULT_LIMIT_NS = 4_000_000_000


@pytest.fixture(scope="module")
def checked_lib():
    if not os.path.exists(build.CHECK_LIB):
        build.build_checked()
    return abi.load_library(build.CHECK_LIB)


def _no_wave0_inputs(cfg):
    """Inputs whose router bias rules out every expert of wave 0 (local ids
    [0, E_w) of each destination), so all routed rows travel in waves 1..W-1."""
    inp = wl.make_inputs(cfg, "cuda")
    E_l = cfg.n_experts // cfg.n_ranks
    E_w = E_l // cfg.n_waves
    bias = torch.zeros(cfg.n_experts, dtype=torch.float32)
    for e in range(cfg.n_experts):
        if e % E_l < E_w:
            bias[e] = -1.0e4
    inp["bias"] = bias.cuda()
    return inp


def test_wave_wait_runs_out_and_the_layer_recovers(checked_lib):
    cfg = wl.TINY.with_(T=4096)
    inp = _no_wave0_inputs(cfg)
    x = inp["x"]
    saved = abi._lib
    abi._lib = checked_lib
    try:
        assert checked_lib.moe_check_status() == 0
        clean = PooledWaveMoE(cfg, inp, "cuda", pipeline="waves")
        clean.forward(x)
        torch.cuda.synchronize()
        assert int(clean.status.item()) == 0
        E_l = cfg.n_experts // cfg.n_ranks
        assert bool(((clean.idx % E_l) >= E_l // cfg.n_waves).all()), "wave 0 still routed"
        assert clean.drop_stats()["kept"] > 0
        ref = {n: getattr(clean, n).clone() for n in ("out", "c", "ypool", "slot_of")}

        m = PooledWaveMoE(cfg, inp, "cuda", pipeline="waves")
        codes = []
        try:
            assert checked_lib.moe_check_set_wave_wait_limit_ns(0) == abi.MOE_OK
            for _ in range(5):
                m.status.zero_()
                m.forward(x)
                torch.cuda.synchronize()          # every CTA returned
                codes.append(int(m.status.item()))
                if codes[-1] == abi.MOE_ETIMEOUT:
                    break
        finally:
            assert checked_lib.moe_check_set_wave_wait_limit_ns(DEFAULT_LIMIT_NS) == abi.MOE_OK
        assert set(codes) <= {abi.MOE_OK, abi.MOE_ETIMEOUT}, codes
        assert codes[-1] == abi.MOE_ETIMEOUT, f"the wait never ran out: {codes}"
        assert checked_lib.moe_check_status() == 0, "an index check fired while unwinding"

        # the same buffers, the default limit: a normal forward again
        m.status.zero_()
        m.forward(x)
        torch.cuda.synchronize()
        assert int(m.status.item()) == 0
        for n, want in ref.items():
            got = getattr(m, n)
            if n == "ypool":   # rows no kept assignment points at are never written
                rows = ref["slot_of"][ref["slot_of"] >= 0].long()
                got, want = got[rows], want[rows]
            assert torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else got,
                               want.view(torch.int16) if want.dtype == torch.bfloat16 else want), n
    finally:
        abi._lib = saved
