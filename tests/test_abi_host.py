"""Host-side checks of the C ABI library (no GPU needed): it builds, loads and
exports every entry point the header declares; its plan (capacities, pool
size) equals the oracle's; invalid configurations are rejected."""
import ctypes
import math
import os
import re

import pytest

import oracle as O
from moe_routing_capacity_gb300 import abi
from moe_routing_capacity_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_pooled_wave.h")


@pytest.fixture(scope="session", autouse=True)
def built_library():
    if not os.path.exists(abi.LIB_PATH):
        from moe_routing_capacity_gb300 import build
        build.build()
    return abi.lib()


def _declared_all():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", src, re.M)))


def _declared():
    """Entry points every build exports (the checked build's test hooks aside)."""
    return [n for n in _declared_all() if n not in abi.CHECKED_ONLY]


def test_header_and_binding_agree():
    assert sorted(abi.EXPORTS) == _declared()
    assert set(abi.CHECKED_ONLY) <= set(_declared_all())


def test_checked_only_hooks_absent_from_the_normal_build():
    L = abi.lib()
    for name in abi.CHECKED_ONLY:
        assert not hasattr(L, name), name


def test_noalloc_scratch_size_matches_the_header():
    src = open(HEADER).read()
    m = re.search(r"#define\s+MOE_DISPATCH_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "MOE_DISPATCH_NOALLOC_SCRATCH_BYTES not found in the header"
    assert abi.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_library_exports_every_declared_symbol():
    L = abi.lib()
    for name in _declared():
        assert hasattr(L, name), name
    assert L.moe_abi_version() == 6


def test_every_export_declares_its_signature():
    """ctypes passes undeclared integer arguments as 32-bit ints, which is
    wrong for sizes and pointers: every entry point gets its argtypes, and
    their count matches the header's parameter list."""
    L = abi.lib()
    src = open(HEADER).read()
    for name in abi.EXPORTS:
        fn = getattr(L, name)
        assert fn.argtypes is not None, name
        m = re.search(r"^\s*(?:const\s+)?\w+\s*\*?\s*" + name + r"\s*\(([^)]*)\)", src, re.M)
        params = [a for a in m.group(1).split(",") if a.strip() and a.strip() != "void"]
        assert len(fn.argtypes) == len(params), (name, len(fn.argtypes), len(params))


def test_struct_sizes():
    assert ctypes.sizeof(abi.Config) == 64
    assert ctypes.sizeof(abi.Plan) == 64
    assert ctypes.sizeof(abi.DropStats) == 48
    assert abi.STATS_WORDS == 6


def _c_layout(struct, fields, tmp_path):
    """sizeof and each field's offset of a header struct, from a C program
    compiled against the header."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe_pooled_wave.h"',
             "int main(void) {", f'  printf("%zu\\n", sizeof({struct}));']
    lines += [f'  printf("%zu\\n", offsetof({struct}, {f}));' for f in fields]
    lines += ["  return 0;", "}"]
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    return vals[0], vals[1:]


@pytest.mark.parametrize("struct,cls", [("moe_backward_args_t", abi.BackwardArgs),
                                        ("moe_layer_buffers_t", abi.LayerBuffers)])
def test_struct_mirrors_match_header(struct, cls, tmp_path):
    """The binding's ctypes mirrors of the argument structs have the header's
    size and field offsets, field by field."""
    names = [f for f, _ in cls._fields_]
    size, offs = _c_layout(struct, names, tmp_path)
    assert ctypes.sizeof(cls) == size
    assert [getattr(cls, f).offset for f in names] == offs


def test_strerror_names_every_code():
    for c in (abi.MOE_OK, abi.MOE_EINVAL, abi.MOE_ENOSPC, abi.MOE_ECUDA, abi.MOE_ETIMEOUT,
              abi.MOE_ENODEV):
        assert abi.strerror(c) != "unknown error"
    assert abi.strerror(-99) == "unknown error"


@pytest.mark.parametrize("cfg", list(wl.CONFIGS.values()), ids=lambda c: c.name)
def test_plan_matches_oracle(cfg):
    p, q = abi.plan(cfg), O.make_plan(cfg)
    assert (p.c_send, p.c_recv, p.pool_rows) == (q.c_send, q.c_recv, q.pool_rows)
    assert p.tokens_per_rank == q.T_s and p.experts_per_rank == q.E_l
    assert p.experts_per_wave == q.E_w
    # L bf16 payload + 16-byte tag, padded to whole 128-byte lines
    assert p.pool_row_bytes == -(-(2 * cfg.d_latent + 16) // 128) * 128
    assert p.h_offset_bytes % 16 == 0
    assert p.ws_ffn_bytes >= p.h_offset_bytes + cfg.n_experts * p.c_recv * cfg.h_expert * 2


@pytest.mark.parametrize("cfg", list(wl.CONFIGS.values()), ids=lambda c: c.name)
def test_ragged_plan_leaves_room_for_the_row_groups(cfg):
    """The dropless plan: a pool of exactly T*k rows, and below h room for
    the expert products' work lists in the worst case, whatever the routing:
    the gathered path's 128-row tiles (at most rows/128 + E entries of 8
    bytes) and the row-group path's lists (every expert's chunks of at most
    256 rows and groups of at most 416: at most E + rows/256 + 1 and
    E + rows/416 + 1 entries of 16 bytes, plus two counters)."""
    p = abi.plan_ragged(cfg)
    rows, E = cfg.T * cfg.top_k, cfg.n_experts
    assert p.pool_rows == rows and p.c_send == 0 and p.c_recv == 0
    tiles = (rows // 128 + E) * 8 + 16
    lists = (E + rows // 256 + 1 + E + rows // 416 + 1) * 16 + 16
    assert p.h_offset_bytes >= max(tiles, lists)
    assert p.h_offset_bytes % 16 == 0
    assert p.ws_ffn_bytes >= p.h_offset_bytes + rows * cfg.h_expert * 2


def _small(**kw):
    base = dict(name="s", T=64, d_model=64, d_latent=32, n_experts=12, n_ranks=2, top_k=2,
                n_waves=3, n_shared=1, h_expert=32, h_shared=32)
    base.update(kw)
    return wl.LayerConfig(**base)


@pytest.mark.parametrize("kw", [
    dict(cf_send=1.1, cf_recv=1.1), dict(cf_send=0.01, cf_recv=0.01),
    dict(cf_send=float("inf"), cf_recv=float("inf")), dict(cf_send=1.5, cf_recv=1.25),
    dict(T=0), dict(top_k=1), dict(n_waves=1), dict(n_waves=2, n_experts=8),
    dict(T=75, n_ranks=1, n_experts=3, n_waves=3, cf_send=1.1, cf_recv=1.1),
    dict(T=200, n_ranks=4, n_experts=24, top_k=5, cf_send=1.37, cf_recv=0.93),
])
def test_plan_matches_oracle_edge_cases(kw):
    cfg = _small(**kw)
    p, q = abi.plan(cfg), O.make_plan(cfg)
    assert (p.c_send, p.c_recv, p.pool_rows) == (q.c_send, q.c_recv, q.pool_rows)


@pytest.mark.parametrize("kw", [
    dict(T=63),                     # T not divisible by the ranks
    dict(n_experts=13),             # E not divisible by the ranks
    dict(n_experts=8, n_waves=3),   # E/ranks not divisible by the waves
    dict(d_model=60),               # rows not 16-byte multiples
    dict(d_latent=36), dict(h_expert=20), dict(h_shared=12),
    dict(top_k=0), dict(top_k=13), dict(top_k=33, n_experts=64),
    dict(n_shared=4), dict(cf_send=0.0), dict(cf_recv=-1.0), dict(cf_send=float("nan")),
    dict(n_experts=2048, n_ranks=2, n_waves=1, top_k=2),
])
def test_plan_rejects_invalid(kw):
    cfg = _small(**kw)
    with pytest.raises(abi.MoeError) as ei:
        abi.plan(cfg)
    assert ei.value.code == abi.MOE_EINVAL


def test_plans_refuse_rows_past_32_bit_indices():
    """Row lists and slots are int32: a batch whose pool would hold more rows
    than they index is refused by both layouts' plans."""
    cfg = _small(T=2**28, top_k=8)
    for fn in (abi.plan, abi.plan_ragged):
        with pytest.raises(abi.MoeError) as ei:
            fn(cfg)
        assert ei.value.code == abi.MOE_EINVAL


def test_entry_points_validate_before_touching_the_gpu():
    """Null pointers and short scratch are refused on the host, before any
    device call (these run without a GPU)."""
    L = abi.lib()
    c = abi.make_config(_small())
    cp = ctypes.byref(c)
    n = None
    assert L.moe_router_topk(cp, n, n, n, n, n, n, n, n, n) == abi.MOE_EINVAL
    assert L.moe_latent_proj(n, n, 4, 8, 8, n, n, n) == abi.MOE_EINVAL
    assert L.moe_latent_proj(ctypes.c_void_p(16), ctypes.c_void_p(16), 4, 12, 8,
                             ctypes.c_void_p(16), ctypes.c_void_p(16), n) == abi.MOE_EINVAL
    assert L.moe_dispatch_pooled(cp, n, n, n, 0, n, n, n, n, n, n, n, n) == abi.MOE_EINVAL
    p = abi.plan(_small())
    fake = ctypes.c_void_p(1 << 20)
    assert L.moe_dispatch_pooled(cp, fake, fake, fake, p.ws_dispatch_bytes - 1, fake, fake, fake,
                                 fake, fake, fake, n, n) == abi.MOE_ENOSPC
    # a bank that is not 16-byte aligned is refused
    assert L.moe_dispatch_pooled(cp, fake, fake, fake, p.ws_dispatch_bytes, fake, fake, fake,
                                 fake, fake, fake, ctypes.c_void_p((1 << 20) + 8),
                                 n) == abi.MOE_EINVAL
    assert L.moe_expert_ffn_grouped(cp, fake, n, fake, fake, fake, fake, fake, fake,
                                    p.ws_ffn_bytes - 1, fake, fake, n) == abi.MOE_ENOSPC
    assert L.moe_combine(cp, n, n, n, n, n, n, n, n, n, n, n, n, n) == abi.MOE_EINVAL
    # shared activations given (Wsg = Wsu = NULL) but no a: refused
    assert L.moe_combine(cp, fake, fake, fake, fake, n, n, n, fake, fake, n, fake, fake,
                         n) == abi.MOE_EINVAL
    # the overlapped paths: null pointers, then short scratch of either kind
    # (sizes passed as size_t: past the sixth argument they travel on the stack)
    sz = ctypes.c_size_t
    assert L.moe_dispatch_expert_waves(cp, *([n] * 3), sz(0), *([n] * 10), sz(0), n, n,
                                       n) == abi.MOE_EINVAL
    assert L.moe_dispatch_expert_waves(cp, fake, fake, fake, sz(p.ws_dispatch_bytes - 1),
                                       *([fake] * 9), fake, sz(p.ws_ffn_bytes), fake, fake,
                                       n) == abi.MOE_ENOSPC
    assert L.moe_dispatch_expert_waves(cp, fake, fake, fake, sz(p.ws_dispatch_bytes),
                                       *([fake] * 9), fake, sz(p.ws_ffn_bytes - 1), fake, fake,
                                       n) == abi.MOE_ENOSPC
    assert L.moe_dispatch_shared_overlap(cp, *([n] * 3), sz(0), *([n] * 13)) == abi.MOE_EINVAL
    assert L.moe_dispatch_shared_overlap(cp, fake, fake, fake, sz(p.ws_dispatch_bytes - 1),
                                         *([fake] * 6), n, *([fake] * 5), n) == abi.MOE_ENOSPC
    assert L.moe_dispatch_shared_overlap(cp, fake, fake, fake, sz(p.ws_dispatch_bytes),
                                         *([fake] * 6), n, *([fake] * 3), n, fake,
                                         n) == abi.MOE_EINVAL   # no a
    assert L.moe_balance_update_window(cp, fake, fake, fake, 0, fake, ctypes.c_float(1.0), fake,
                                       n) == abi.MOE_EINVAL   # window < 1
    # the dropless entry points: null pointers, short scratch, a misaligned
    # bank, the overlapped dispatch without a
    pr = abi.plan_ragged(_small())
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert L.moe_dispatch_ragged(cp, *([n] * 3), sz(0), *([n] * 10)) == abi.MOE_EINVAL
    assert L.moe_dispatch_ragged(cp, fake, fake, fake, sz(pr.ws_dispatch_bytes - 1),
                                 *([fake] * 7), n, n) == abi.MOE_ENOSPC
    assert L.moe_dispatch_ragged(cp, fake, fake, fake, sz(pr.ws_dispatch_bytes),
                                 *([fake] * 7), odd, n) == abi.MOE_EINVAL
    assert L.moe_dispatch_ragged_shared_overlap(cp, *([n] * 3), sz(0),
                                                *([n] * 15)) == abi.MOE_EINVAL
    assert L.moe_dispatch_ragged_shared_overlap(cp, fake, fake, fake,
                                                sz(pr.ws_dispatch_bytes - 1), *([fake] * 7), n,
                                                *([fake] * 5), n) == abi.MOE_ENOSPC
    assert L.moe_dispatch_ragged_shared_overlap(cp, fake, fake, fake, sz(pr.ws_dispatch_bytes),
                                                *([fake] * 7), n, *([fake] * 3), n, fake,
                                                n) == abi.MOE_EINVAL   # no a
    assert L.moe_expert_ffn_ragged(cp, fake, n, *([fake] * 7), sz(pr.ws_ffn_bytes - 1), fake,
                                   fake, n) == abi.MOE_ENOSPC
    assert L.moe_expert_ffn_ragged(cp, fake, odd, *([fake] * 7), sz(pr.ws_ffn_bytes), fake,
                                   fake, n) == abi.MOE_EINVAL
    # the backward refuses a bank that is not 16-byte aligned
    args = abi.BackwardArgs()
    for f, _ in abi.BackwardArgs._fields_:
        if f not in ("ws_bytes", "expert_offsets", "bank"):
            setattr(args, f, 1 << 20)
    args.ws_bytes = 1 << 40
    args.bank = (1 << 20) + 8
    assert L.moe_layer_backward(cp, ctypes.byref(args), n) == abi.MOE_EINVAL
    bad = abi.make_config(_small(T=63))
    assert L.moe_plan(ctypes.byref(bad), ctypes.byref(abi.Plan())) == abi.MOE_EINVAL


def test_capacity_uses_decimal_factor():
    # 1.1 * 50 is 55 exactly; a float ceil would say 56
    cfg = _small(T=75, n_ranks=1, n_experts=3, n_waves=3, top_k=2, cf_send=1.1, cf_recv=1.1)
    p = abi.plan(cfg)
    assert (p.c_send, p.c_recv) == (55, 55)
    assert not math.isclose(1.1 * 50, 55.0, rel_tol=0, abs_tol=0)


def test_layer_forward_and_host_pipe_refuse_bad_arguments():
    """Refused on the host before any device call."""
    L = abi.lib()
    c = abi.make_config(_small())
    cp = ctypes.byref(c)
    arr0 = (ctypes.c_void_p * 1)()
    h = ctypes.c_void_p()
    assert L.moe_host_pipe_create(cp, 0, arr0, arr0, arr0, ctypes.byref(h)) == abi.MOE_EINVAL
    assert L.moe_host_pipe_create(cp, 1, arr0, arr0, arr0, ctypes.byref(h)) == abi.MOE_EINVAL
    assert not h.value
    assert L.moe_layer_forward(cp, None, None, None, None) == abi.MOE_EINVAL
    assert L.moe_host_pipe_submit(None, None, None, None, None, None) == abi.MOE_EINVAL
    assert L.moe_host_pipe_sync(None) == abi.MOE_EINVAL
    assert L.moe_host_pipe_destroy(None) == abi.MOE_OK
