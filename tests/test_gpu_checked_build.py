"""The checked build (-DMOE_CHECK=1: every row, slot, expert and tile index a
kernel computes is verified before use, failures recorded in a device word
and the access skipped) on the layer's forward and backward, capped and
dropless, and on the overlapped pool fills (copy warps inside the shared
or the expert gate/up launch), at the tiny and mid sizes and on the full
workload in the bench's schedule: no check fires, and the results equal the
normal build's bit for bit.  This stands in for a memory checker, which is
not available here."""
import os

import pytest
import torch

from moe_routing_capacity_gb300 import abi, build
from moe_routing_capacity_gb300 import workloads as wl
from moe_routing_capacity_gb300.layer import PooledWaveMoE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked_lib():
    if not os.path.exists(build.CHECK_LIB):
        build.build_checked()
    return abi.load_library(build.CHECK_LIB)


def _run(cfg, dropless, lib=None, pipeline=None):
    saved = abi._lib
    if lib is not None:
        abi._lib = lib
    try:
        inp = wl.make_inputs(cfg, "cuda")
        m = PooledWaveMoE(cfg, inp, "cuda", dropless=dropless, pipeline=pipeline)
        x = inp["x"]
        m.forward(x)
        g = torch.Generator(device="cuda").manual_seed(5)
        dout = torch.randn(cfg.T, cfg.d_model, generator=g, device="cuda").to(torch.bfloat16)
        grads = m.backward(x, dout)
        torch.cuda.synchronize()
        code = abi.lib().moe_check_status()
        assert int(m.status.item()) == 0
        out = {"out": m.out.clone(), "slot_of": m.slot_of.clone(), "drop": m.drop.clone(),
               "tags": m.pool_tags().clone()}
        out.update({"d" + k: v.clone() for k, v in grads.items()})
        return out, code
    finally:
        abi._lib = saved


@pytest.mark.parametrize("name,dropless", [("tiny", False), ("tiny", True),
                                           ("mid", False), ("mid", True)])
def test_checked_build_clean_and_identical(checked_lib, name, dropless):
    cfg = wl.CONFIGS[name]
    want, code0 = _run(cfg, dropless)
    assert code0 == 0                      # the normal build never records anything
    got, code = _run(cfg, dropless, checked_lib)
    assert code == 0, f"index check site {code} fired"
    for key, v in want.items():
        a = v.contiguous().view(torch.uint8)
        b = got[key].contiguous().view(torch.uint8)
        assert torch.equal(a, b), key


@pytest.mark.parametrize("pipeline,dropless", [("waves", False), ("shared", False),
                                               ("shared", True)])
@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_checked_build_overlapped_fill(checked_lib, name, pipeline, dropless):
    cfg = wl.CONFIGS[name]
    want, code0 = _run(cfg, dropless, pipeline=pipeline)
    assert code0 == 0
    got, code = _run(cfg, dropless, checked_lib, pipeline=pipeline)
    assert code == 0, f"index check site {code} fired"
    for key, v in want.items():
        assert torch.equal(v.contiguous().view(torch.uint8), got[key].contiguous().view(torch.uint8)), key


@pytest.mark.parametrize("dropless", [False, True], ids=["capped", "dropless"])
def test_checked_build_full_workload(checked_lib, dropless):
    """The full workload in the bench's schedule (pool fill inside the shared
    gate/up, the expert products on CTA pairs over row groups, and the
    backward's grouped expert products), forward and backward, in either
    layout, through the checked build: no index check fires and every output
    and gradient equals the normal build's bit for bit."""
    cfg = wl.CONFIGS["full"]
    want, code0 = _run(cfg, dropless, pipeline="shared")
    assert code0 == 0
    got, code = _run(cfg, dropless, checked_lib, pipeline="shared")
    assert code == 0, f"index check site {code} fired"
    for key in list(want):
        a, b = want.pop(key), got.pop(key)
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), key
        del a, b
