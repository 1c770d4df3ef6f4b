#!/usr/bin/env python
"""Benchmark: routed tokens/s of one pooled-wave MoE layer forward on GB300.

One step = one whole forward of the layer (router top-k, latent projection,
fixed pooled-wave dispatch with both capacity caps, grouped SwiGLU experts,
combine + up-projection + shared experts) over one batch of T synthetic
tokens of the full-width 535B-A23B layer (d=6144, L=3072, 384 experts on 64
logical ranks, top-8, 2 shared experts).  Inputs and weights are resident in
HBM when the timed region starts; the weights (8.1 GB) exceed L2, so no
separate L2 flush is done.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead (a
bounded token sample of the same workload per step, on the host cores).
Under torchrun each rank runs an independent replica on its own batch
(weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_routing_capacity_gb300 import workloads as wl  # noqa: E402

METRIC = "routed tokens/sec per MoE layer on 1 GB300"
UNIT = "tokens/s"
REF_BUDGET_S = 150.0   # oracle seconds the reference arm spends at most (then one more step)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="full", choices=sorted(wl.CONFIGS))
    ap.add_argument("--cpu-sample", type=int, default=0,
                    help="tokens per oracle sample (0: sized automatically)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-dropless", action="store_true",
                    help="skip timing the dropless ragged variant")
    ap.add_argument("--no-train", action="store_true",
                    help="skip timing forward + backward (one training step of the layer)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the skewed-routing and long-context lines")
    ap.add_argument("--pipeline", default="shared", choices=["none", "waves", "shared"],
                    help="how the dispatch's pool fill is scheduled: a kernel of its own "
                         "(none), wave by wave inside the expert gate/up launch (waves), or "
                         "inside the shared experts' gate/up launch (shared)")
    ap.add_argument("--no-pipelines", action="store_true",
                    help="skip timing the three pool-fill schedules side by side")
    args = ap.parse_args()
    # at least three untimed warm-up steps whatever is asked; the line
    # reports the number run
    args.warmup = max(args.warmup, 3)
    return args


# ------------------------------------------------------------------ helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# Sources a kernel's DRAM traffic depends on: its own translation unit, the
# shared device helpers and layouts, and the entry points that describe its
# operands.  A traffic record taken under other sources is not reported.
KERNEL_SOURCES = {
    "gemm": ("gemm_tc.cu", "common.cuh", "internal.h", "abi.cu"),
    "expert": ("expert_pair.cu", "common.cuh", "internal.h", "abi.cu"),
    "route": ("route.cu", "common.cuh", "internal.h", "abi.cu"),
}


def source_group(kernel: str, bank_path: bool = True) -> str:
    if kernel.startswith("gemm_expert") and bank_path:
        return "expert"
    return "gemm" if kernel.startswith("gemm") else "route"


def code_text(text):
    """C++/CUDA source with its comments removed and whitespace collapsed:
    what a source hash should change with (string literals in these sources
    hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash(kernel="gemm", bank_path=True):
    """Hash of the code (comments and layout left out) of a kernel's
    translation unit, the shared device headers and the entry points."""
    files = KERNEL_SOURCES[source_group(kernel, bank_path)]
    h = hashlib.sha256()
    src = os.path.join(ROOT, "moe_routing_capacity_gb300", "csrc")
    for f in files:
        h.update(code_text(open(os.path.join(src, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def kernel_work(name, cfg, plan, st, pipeline="none", sent_w0=None, bank=False):
    """Algorithmic work of one launch: (amount, unit, bound).  The pack
    kernel's bytes depend on where the pool fill runs: all of it (none) or
    wave 0's rows (waves: sent_w0 sender-kept rows); with the shared
    schedule the whole pack runs inside the shared gate/up launch and the
    pack kernel is not launched.  With the per-expert bank the pack also
    writes every receiver-kept row a second time.  Pack work done inside a
    GEMM launch is not added to its flops."""
    T, d, L, E, k = cfg.T, cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.top_k
    H, Hs, ns = cfg.h_expert, cfg.h_shared, cfg.n_shared
    kept = st["kept"]
    sent = st["kept"] + st["dropped_recv"]
    F = {
        "gemm_router": 2.0 * T * d * E,
        "gemm_latent": 2.0 * T * d * L,
        "gemm_latent_router": 2.0 * T * d * (L + E),
        "gemm_expert_gateup": 2.0 * kept * L * 2 * H,
        "gemm_expert_down": 2.0 * kept * H * L,
        "gemm_shared_gateup": 2.0 * T * d * 2 * ns * Hs,
        "gemm_out": 2.0 * T * (L + ns * Hs) * d,
    }
    if name in F:
        return F[name] / 1e12, "TFLOP", "tensor"
    B = {
        "router_topk": T * E * 4 + T * k * 8 + T,
        # each token's z row read once, every sender-kept row written with its tag,
        # plus the per-assignment decisions
        "dispatch_pack": (T * L * 2 + sent * (2 * L + 16) if pipeline == "none" else
                          T * L * 2 + sent_w0 * (2 * L + 16) if pipeline == "waves" else 0)
                         + T * k * (4 + 8 + 4 + 4 + 1) + kept * 4
                         + (kept * L * 2 if bank and pipeline == "none" else 0),
        "dispatch_init": plan.pool_rows * 16 + E * plan.c_recv * 4,
        # every kept expert row read once, c written once, slots and weights read
        "combine": kept * L * 2 + T * L * 2 + T * k * 8,
    }
    if name in B:
        return B[name] / 1e9, "GB", "hbm"
    return None, None, "latency"


def expert_stream_bytes(name, cfg, st, n_active):
    """DRAM bytes an expert product must move at least: the weights of the
    experts with rows, read once, the rows read once and the output written
    once (gate/up: bank or pool rows of width L in, h out; down: h in, Y
    rows of width L out).  None for other kernels."""
    L, H, kept = cfg.d_latent, cfg.h_expert, st["kept"]
    if name == "gemm_expert_gateup":
        return (n_active * 2 * H * L * 2 + kept * L * 2 + kept * H * 2) / 1e9
    if name == "gemm_expert_down":
        return (n_active * L * H * 2 + kept * H * 2 + kept * L * 2) / 1e9
    return None


def expert_mma_rows(counts, c_recv, bank_path):
    """Rows the expert products multiply per weight row.  Gathered path: each
    expert's rows padded to whole 128-row tiles.  Bank path (CTA pairs, rows
    on the MMA's N axis): an expert's n rows in groups of at most 416 sized
    evenly and rounded up to 16; a group of r rows is one chunk of r rounded
    up to 16 when r <= 256, else two chunks, the first half of r rounded up
    to 32 and the rest rounded up to 16."""
    def up(v, m):
        return (v + m - 1) // m * m

    total = 0
    for n in counts:
        n = max(0, min(int(n), c_recv))
        if not bank_path:
            total += up(n, 128)
            continue
        if n == 0:
            continue
        ng = (n + 415) // 416
        per = up((n + ng - 1) // ng, 16)
        for i in range((n + per - 1) // per):
            r = min(per, n - i * per)
            if r <= 256:
                total += up(r, 16)
            else:
                n0 = up((r + 1) // 2, 32)
                total += n0 + up(r - n0, 16)
    return total


def tensor_peak_for(pk, elapsed_s, clk):
    """Which measured bf16 peak a contraction timed in this region is held
    to: the burst figure (a short loop at the maximum clock) when the timed
    region lasts under a second and the sampled SM clock stayed at its
    maximum with no power cap, else the sustained figure (a seconds-long
    loop under the power cap).  Returns (state, peak, the other peak)."""
    at_max = (clk is None or (clk["sm_mhz"] >= 0.97 * clk["sm_max_mhz"]
                              and "sw_power_cap" not in clk["reasons"]))
    if elapsed_s < 1.0 and at_max:
        return "burst", pk["bf16"], pk["bf16_sustained"]
    return "sustained", pk["bf16_sustained"], pk["bf16"]


class ClockSampler:
    """nvidia-smi samples while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, enabled=True):
        self.p = None
        self.index = index
        if enabled:
            try:
                self.p = subprocess.Popen(
                    ["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except (OSError, FileNotFoundError):
                self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append(dict(sm=float(f[0]), max=float(f[1]), power=float(f[2]),
                                 hw=f[4], hwt=f[5], swt=f[6], swp=f[7]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, nm in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                            ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(nm)
        loaded = [r["sm"] for r in rows if r["power"] > 300] or [r["sm"] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


def oracle_inputs(cfg_full, inputs_dev, n_tokens):
    """Host copies of the inputs for an oracle run on the first n_tokens of
    the batch (a layer of the same widths with T = n_tokens), widened to the
    oracle's float64 once, outside any timing."""
    import numpy as np
    S = cfg_full.n_ranks
    n = max(S, (n_tokens // S) * S)
    # float64 expert weights need 4x their bf16 size in host memory; with less
    # than that available they stay float32 and the oracle widens per expert
    wide = np.float64 if 5 * sum(v.numel() * 8 for k, v in inputs_dev.items()
                                 if v is not None and v.dim() == 3) < mem_available() \
        else np.float32
    host = {}
    for key, v in inputs_dev.items():
        if v is None:
            host[key] = None
        elif key == "x":
            host[key] = v[:n].double().cpu().numpy()
        elif v.dim() == 3:
            a = np.empty(tuple(v.shape), dtype=wide)
            for e in range(v.shape[0]):
                a[e] = v[e].double().cpu().numpy()
            host[key] = a
        else:
            host[key] = v.double().cpu().numpy()
    return cfg_full.with_(T=n), host


def mem_available() -> int:
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def time_oracle(cfg, host):
    import oracle as O
    t0 = time.perf_counter()
    O.layer(cfg, host)
    return time.perf_counter() - t0


def replica_throughput(elapsed_s: float, tokens_per_step: int, steps: int, dev):
    """Whole-job throughput of independent replicas: every rank ran `steps`
    steps of `tokens_per_step` tokens; the job took as long as the slowest
    rank.  Returns (tokens/s over all ranks, max elapsed seconds)."""
    import torch.distributed as dist
    world = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    if world > 1:
        t = torch.tensor([elapsed_s], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_s = float(t.item())
    return world * tokens_per_step * steps / elapsed_s, elapsed_s


def cores_used():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count()


# ------------------------------------------------------------------ arms

def reference_runs_on(rank: int) -> bool:
    """The reference arm (the CPU oracle) runs on rank 0 only; other ranks
    exit without work."""
    return rank == 0


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm (rank 0 only)."""
    if not reference_runs_on(rank):
        return
    cfg = wl.CONFIGS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = wl.make_inputs(cfg, dev)
    total = args.steps + args.warmup
    n_tok = args.cpu_sample or (64 if total > 8 else 256)
    scfg, host = oracle_inputs(cfg, inp, n_tok)
    del inp
    n = scfg.T
    # A full-width oracle pass reads every expert's float64 weights (seconds
    # whatever the sample), so the timed steps stop once the oracle has run
    # for REF_BUDGET_S; the line reports the steps actually timed.
    times = []
    t_start = time.perf_counter()
    for i in range(total):
        if times and time.perf_counter() - t_start > REF_BUDGET_S:
            break
        t = time_oracle(scfg, host)
        if i >= args.warmup:
            times.append(t)
    sec = sum(times)
    value = n * len(times) / sec
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": 1e3 * sec / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": f"{cfg.name}: T={cfg.T} sampled to {n} tokens per step, d={cfg.d_model}, "
                   f"L={cfg.d_latent}, E={cfg.n_experts}, ranks={cfg.n_ranks}, k={cfg.top_k}"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                         "sample": f"{n} tokens per step (T={n} layer of the same widths), "
                                   f"{len(times)} timed steps of the {args.steps} asked (the "
                                   f"arm stops after ~{REF_BUDGET_S:.0f} s of oracle work), "
                                   f"float64 NumPy"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_gb300(args, rank, world, local_rank):
    from moe_routing_capacity_gb300 import abi
    from moe_routing_capacity_gb300.layer import PooledWaveMoE

    cfg = wl.CONFIGS[args.workload]
    if world > 1:
        cfg = cfg.with_(seed=cfg.seed + 1000 * rank)
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = wl.make_inputs(cfg, dev)
    pipeline = args.pipeline
    m = PooledWaveMoE(cfg, inp, dev, pipeline=None if pipeline == "none" else pipeline)
    x = inp["x"]
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        m.forward(x)
    torch.cuda.synchronize()
    assert int(m.status.item()) == 0, "device status word set during warm-up"
    st = m.drop_stats()
    # tokens whose k-th and (k+1)-th (or two adjacent selected) logits are within
    # the near-tie gap: their routing may legitimately differ from the oracle's
    near_ties = int((m.tie != 0).sum().item())
    # MMA rows the expert GEMMs compute (the padding is work the tensor cores
    # do but the algorithmic flop count leaves out)
    n_active = int((m.expert_count > 0).sum().item())
    tile_rows = expert_mma_rows(m.expert_count.tolist(), m.plan.c_recv,
                                m.bank is not None and cfg.d_latent % 256 == 0
                                and cfg.h_expert % 128 == 0)
    # sender-kept rows of wave 0 (what the pack kernel copies when the later
    # waves are filled inside the expert gate/up launch)
    e_w = cfg.n_experts // cfg.n_ranks // cfg.n_waves
    wave = (m.idx.long() % (cfg.n_experts // cfg.n_ranks)) // e_w
    sent_w0 = int(((m.drop != 1) & (wave == 0)).sum().item())

    # ---- timed region: device-resident inputs
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank, enabled=not args.no_clocks)
    time.sleep(0.3 if not args.no_clocks else 0.0)
    n_kern = 16
    abi.trace_begin((n_kern + 1) * args.steps + 8)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        abi.trace_mark(stream)
        m.forward(x)
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    trace = abi.trace_end()
    elapsed = ev0.elapsed_time(ev1) / 1e3
    if world > 1:
        torch.distributed.barrier()
    value, elapsed = replica_throughput(elapsed, cfg.T, args.steps, dev)
    assert int(m.status.item()) == 0, "device status word set during the timed region"

    # ---- per-kernel times from the trace (event after each launch)
    per = {}
    for name, ms in trace:
        if name == "mark":
            continue
        d = per.setdefault(name, [0.0, 0])
        d[0] += ms
        d[1] += 1
    pk = peaks()
    tensor_state, tensor_peak, tensor_other = tensor_peak_for(pk, elapsed, clk)
    kernels = {}
    for name, (ms, n) in sorted(per.items(), key=lambda kv: -kv[1][0]):
        work, unit, bound = kernel_work(name, cfg, m.plan, st, pipeline, sent_w0)
        ms_l = ms / n
        e = {"ms_per_launch": round(ms_l, 4), "launches": n,
             "share": round(ms / max(1e-9, sum(v[0] for v in per.values())), 4)}
        if work is not None:
            ach = work / (ms_l / 1e3)
            peak = tensor_peak if bound == "tensor" else pk["hbm"]
            e.update({"work_per_launch": work, "unit": unit + "/s", "achieved": round(ach, 2),
                      "frac": round(ach / peak, 4)})
        sb = expert_stream_bytes(name, cfg, st, n_active)
        if sb is not None:   # the same launch against its DRAM floor
            gbs = sb / (ms_l / 1e3)
            e["hbm"] = {"bytes_per_launch_gb": round(sb, 4), "achieved_gbs": round(gbs, 1),
                        "frac": round(gbs / pk["hbm"], 4),
                        "floor_ms": round(sb / pk["hbm"] * 1e3, 4)}
        kernels[name] = e
    # the grouped expert FFN as a whole: both products of every expert
    expert_ffn = None
    gu, dn = kernels.get("gemm_expert_gateup", {}), kernels.get("gemm_expert_down", {})
    if "work_per_launch" in gu and "work_per_launch" in dn:
        w_ffn = gu["work_per_launch"] + dn["work_per_launch"]
        ms_ffn = gu["ms_per_launch"] + dn["ms_per_launch"]
        ach = w_ffn / (ms_ffn / 1e3)
        expert_ffn = {"ms": round(ms_ffn, 4), "work": w_ffn, "unit": "TFLOP/s",
                      "achieved": round(ach, 2), "frac": round(ach / tensor_peak, 4),
                      "peak_source": pk["source"] + f" {tensor_state} bf16"}
        if "hbm" in gu and "hbm" in dn:
            gb = gu["hbm"]["bytes_per_launch_gb"] + dn["hbm"]["bytes_per_launch_gb"]
            expert_ffn["hbm"] = {"bytes_gb": round(gb, 4),
                                 "frac": round(gb / (ms_ffn / 1e3) / pk["hbm"], 4)}
    top = next(iter(kernels))
    twork, tunit, tbound = kernel_work(top, cfg, m.plan, st, pipeline, sent_w0)
    # DRAM bytes per launch from the committed ncu record, where it was taken
    # on this workload and pool-fill schedule under the current sources of
    # that kernel
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    recs = json.load(open(tp)) if os.path.exists(tp) else {}
    bank_path = m.bank is not None
    for name, e in kernels.items():
        rec = recs.get(name)
        if (rec and rec.get("source_hash") == source_hash(name, bank_path)
                and rec.get("workload") == cfg.name and rec.get("pool_fill", "none") == pipeline
                and rec.get("bank", bank_path) == bank_path):
            e["traffic"] = rec.get("dram_bytes_per_launch")
            if rec.get("measured_on"):
                e["traffic_from"] = rec["measured_on"]
    traffic = kernels[top].get("traffic")
    if twork is not None:
        ach = kernels[top]["achieved"]
        peak = tensor_peak if tbound == "tensor" else pk["hbm"]
        roof = {"kernel": top, "bound": tbound, "achieved": ach, "peak": peak,
                "unit": "TFLOP/s" if tbound == "tensor" else "GB/s",
                "frac": round(ach / peak, 4), "traffic": traffic,
                "peak_source": pk["source"] + (f" {tensor_state} bf16" if tbound == "tensor"
                                               else " HBM copy")}
        if tbound == "tensor":
            other = "sustained" if tensor_state == "burst" else "burst"
            roof[f"frac_vs_{other}"] = round(ach / tensor_other, 4)
            roof["peak_rule"] = ("burst bf16 peak when the timed region is under 1 s and the "
                                 "sampled SM clock stays at its maximum with no power cap; "
                                 "the sustained one otherwise")
        if top.startswith("gemm_expert") and tile_rows:
            roof["tile_rows"] = tile_rows
            roof["row_util"] = round(st["kept"] / tile_rows, 4)   # kept rows / MMA rows
        if "hbm" in kernels[top]:   # the weight stream's floor beside the tensor figure
            roof["hbm"] = kernels[top]["hbm"]
    else:
        roof = {"kernel": top, "bound": "latency", "achieved": None, "peak": None,
                "unit": None, "frac": None, "traffic": traffic}

    # ---- end to end through the C ABI with host buffers: every step copies
    # its x from pinned host memory and its output + drop stats back, inside
    # the library (moe_host_pipe_submit, the copies overlapped with the
    # neighbouring steps' compute).
    e2e = None
    if not args.no_e2e:
        from moe_routing_capacity_gb300.layer import HostPipeline
        xh = x.cpu().pin_memory()
        oh = [torch.empty(cfg.T, cfg.d_model, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        sh = [torch.empty(m.stats.numel(), dtype=torch.int64).pin_memory() for _ in range(2)]
        pipe = HostPipeline(m, depth=2)
        for i in range(3):
            pipe.submit(xh, oh[i % 2], sh[i % 2])
        pipe.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        # five rounds, the median reported: the host copies share the host's
        # memory and link with whatever else the machine runs
        n_e2e = max(4, min(args.steps, 40))
        rounds = []
        for _ in range(5):
            t0 = time.perf_counter()
            for i in range(n_e2e):
                pipe.submit(xh, oh[i % 2], sh[i % 2])
            pipe.synchronize()
            torch.cuda.synchronize()
            el = time.perf_counter() - t0
            rounds.append(replica_throughput(el, cfg.T, n_e2e, dev)[0])
        assert int(m.status.item()) == 0
        e2e = {"value": sorted(rounds)[2], "unit": UNIT,
               "h2d_bytes_per_step": xh.numel() * xh.element_size(),
               "d2h_bytes_per_step": oh[0].numel() * oh[0].element_size() + sh[0].numel() * 8,
               "steps": 5 * n_e2e, "rounds": [round(r) for r in rounds],
               "timer": "host wall clock around each round of submitted steps; median of 5",
               "path": "moe_host_pipe_submit (C ABI) with pinned host buffers: the whole "
                       "forward per call, H2D / compute / D2H on three streams, double-buffered"}

    # ---- the same step replayed from a CUDA graph (no host launch work)
    graph = None
    try:
        xg = x.clone()
        gr = m.capture(xg)
        torch.cuda.synchronize()
        ng = max(3, min(args.steps, 100))
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(ng):
            gr.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        assert int(m.status.item()) == 0
        gms = g0.elapsed_time(g1) / ng
        graph = {"value": world * cfg.T / (gms / 1e3), "unit": UNIT, "ms_per_step": gms,
                 "steps": ng, "note": "whole forward captured once, replayed"}
        del gr, xg
    except RuntimeError as exc:   # report, do not hide: the line says why
        graph = {"unavailable": str(exc).splitlines()[0][:200]}

    # ---- the three pool-fill schedules side by side on the same batch
    # (rounds in rotated order, median of the rounds per schedule)
    pipes = None
    if not args.no_pipelines:
        arms = {pipeline: m}
        for pn in ("none", "waves", "shared"):
            if pn not in arms:
                arms[pn] = PooledWaveMoE(cfg, inp, dev, pipeline=None if pn == "none" else pn)
                for _ in range(args.warmup):
                    arms[pn].forward(x)
        torch.cuda.synchronize()
        names = ["none", "waves", "shared"]
        n_p = max(3, min(args.steps, 30))
        per_arm = {pn: [] for pn in names}
        # per arm and kernel: the mean launch time of each round
        kern_arm = {pn: {} for pn in names}
        for r in range(7):
            for j in range(3):
                pn = names[(r + j) % 3]
                q0 = torch.cuda.Event(enable_timing=True)
                q1 = torch.cuda.Event(enable_timing=True)
                abi.trace_begin((n_kern + 1) * n_p + 8)
                q0.record(stream)
                for _ in range(n_p):
                    abi.trace_mark(stream)
                    arms[pn].forward(x)
                q1.record(stream)
                torch.cuda.synchronize()
                rtr = abi.trace_end()
                per_arm[pn].append(q0.elapsed_time(q1) / n_p)
                rk = {}
                for name, ms in rtr:
                    if name != "mark":
                        rk.setdefault(name, []).append(ms)
                for name, v in rk.items():
                    kern_arm[pn].setdefault(name, []).append(sum(v) / len(v))
        for pn in names:
            assert int(arms[pn].status.item()) == 0
        same = all(torch.equal(arms[pn].out.view(torch.int16), m.out.view(torch.int16))
                   for pn in names)
        pipes = {pn: {"ms_per_step": round(sorted(v)[3], 4),
                      "value": world * cfg.T / (sorted(v)[3] / 1e3),
                      "kernel_ms": {k2: round(statistics.median(v2), 4)
                                    for k2, v2 in sorted(kern_arm[pn].items())}}
                 for pn, v in per_arm.items()}
        pipes["steps_per_round"] = n_p
        pipes["rounds"] = 7
        pipes["outputs_bit_identical"] = same
        pipes["timer"] = ("CUDA events around each round; kernel_ms: median over the rounds of "
                          "each kernel's mean launch time (library trace)")
        # the pack as a kernel of its own (the sequential schedule): its
        # bandwidth against the HBM copy peak, beside the main arm's kernels
        pk_ms = pipes["none"]["kernel_ms"].get("dispatch_pack")
        if pk_ms:
            pw, pu, _ = kernel_work("dispatch_pack", cfg, m.plan, st, "none",
                                    bank=arms["none"].bank is not None)
            ach = pw / (pk_ms / 1e3)
            kernels["dispatch_pack"] = {
                "ms_per_launch": pk_ms, "launches": 7 * n_p, "work_per_launch": pw,
                "unit": pu + "/s", "achieved": round(ach, 2), "frac": round(ach / pk["hbm"], 4),
                "from": "pipelines.none (the pack as a kernel of its own, the sequential "
                        "schedule); the timed arm runs it inside the shared gate/up launch"}
        # what carrying the pack costs the shared experts' gate/up launch
        sg_with = pipes["shared"]["kernel_ms"].get("gemm_shared_gateup")
        sg_without = pipes["none"]["kernel_ms"].get("gemm_shared_gateup")
        if sg_with and sg_without:
            pw, _, _ = kernel_work("dispatch_pack", cfg, m.plan, st, "none",
                                   bank=arms["shared"].bank is not None)
            marg = sg_with - sg_without
            pipes["pack_in_shared_gateup"] = {
                "with_pack_ms": sg_with, "without_pack_ms": sg_without,
                "marginal_ms": round(marg, 4), "pack_gb": round(pw, 4),
                "pack_kernel_ms": pk_ms,
                "note": "shared gate/up launch time carrying the whole pack (shared schedule) "
                        "minus the same launch without it (sequential schedule)"}
        for pn in names:
            if arms[pn] is not m:
                del arms[pn]
        torch.cuda.empty_cache()

    # ---- the dropless ragged variant on the same batch: the cost of removing drops
    dropless = None
    if not args.no_dropless:
        # the same pool-fill schedule as the main line (the wave pipeline is
        # built for the capped layout only)
        dpipe = "shared" if pipeline == "shared" else None
        md = PooledWaveMoE(cfg, inp, dev, dropless=True, pipeline=dpipe)
        for _ in range(args.warmup):
            md.forward(x)
        torch.cuda.synchronize()
        nd = max(3, min(args.steps, 100))
        abi.trace_begin((n_kern + 1) * nd + 8)
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(nd):
            abi.trace_mark(stream)
            md.forward(x)
        d1.record(stream)
        torch.cuda.synchronize()
        dtr = abi.trace_end()
        assert int(md.status.item()) == 0
        dms = d0.elapsed_time(d1) / nd
        dper = {}
        for name, ms in dtr:
            if name != "mark":
                dper.setdefault(name, []).append(ms)
        dst = md.drop_stats()
        dropless = {"value": world * cfg.T / (dms / 1e3), "unit": UNIT, "ms_per_step": dms,
                    "steps": nd, "pool_rows": md.plan.pool_rows, "pool_fill": dpipe or "none",
                    "kept": dst["kept"], "capped_kept": st["kept"],
                    "expert_ffn_ms": round(sum(sum(v) for k2, v in dper.items()
                                               if k2.startswith("gemm_expert")) / nd, 4)}
        del md

    # ---- the skewed-routing and long-context workloads: throughput and drops
    others = None
    if not args.no_workloads and args.workload == "full":
        others = {}
        for oname in ("skew", "long"):
            ocfg = wl.CONFIGS[oname]
            oinp = wl.make_inputs(ocfg, dev)
            mo = PooledWaveMoE(ocfg, oinp, dev, pipeline=None if pipeline == "none" else pipeline)
            ox = oinp["x"]
            for _ in range(3):
                mo.forward(ox)
            torch.cuda.synchronize()
            no = 20
            o0 = torch.cuda.Event(enable_timing=True)
            o1 = torch.cuda.Event(enable_timing=True)
            o0.record(stream)
            for _ in range(no):
                mo.forward(ox)
            o1.record(stream)
            torch.cuda.synchronize()
            assert int(mo.status.item()) == 0
            oms = o0.elapsed_time(o1) / no
            ost = mo.drop_stats()
            others[oname] = {
                "value": world * ocfg.T / (oms / 1e3), "unit": UNIT, "ms_per_step": oms,
                "steps": no, "T": ocfg.T,
                "drop_rate": (ost["dropped_send"] + ost["dropped_recv"]) / (ocfg.T * ocfg.top_k),
                "dropped_send": ost["dropped_send"], "dropped_recv": ost["dropped_recv"],
                "note": ("Zipf(1.2) prior on the router logits, hot experts on the first ranks"
                         if oname == "skew" else "one 65536-token AR(1) sequence")}
            del mo, oinp, ox

    # ---- one training step of the layer: forward + backward on the same batch
    train = None
    if not args.no_train:
        g = torch.Generator(device=dev).manual_seed(7)
        dout = torch.randn(cfg.T, cfg.d_model, generator=g, device=dev).to(torch.bfloat16)
        for _ in range(2):
            m.forward(x)
            m.backward(x, dout)
        torch.cuda.synchronize()
        assert int(m.status.item()) == 0, "device status word set in the backward"
        nt = max(3, min(args.steps, 30))
        abi.trace_begin(64 * nt + 8)
        t0e = torch.cuda.Event(enable_timing=True)
        t1e = torch.cuda.Event(enable_timing=True)
        t0e.record(stream)
        for _ in range(nt):
            abi.trace_mark(stream)
            m.forward(x)
            m.backward(x, dout)
        t1e.record(stream)
        torch.cuda.synchronize()
        ttr = abi.trace_end()
        assert int(m.status.item()) == 0
        tms = t0e.elapsed_time(t1e) / nt
        bwd = sum(ms for n, ms in ttr if n.startswith("bwd_")) / nt
        tv, _ = replica_throughput(tms / 1e3, cfg.T, 1, dev)
        # GEMM work of the backward: twice the forward's, plus the gate/up
        # recomputes (routed and shared)
        fwd_tf = sum(kernel_work(n, cfg, m.plan, st)[0] or 0.0 for n in per
                     if kernel_work(n, cfg, m.plan, st)[2] == "tensor")
        # the backward's launches, ms a step each (a name launched several
        # times a step is summed)
        bk = {}
        for n, ms in ttr:
            if n.startswith("bwd_"):
                bk[n] = bk.get(n, 0.0) + ms / nt
        train = {"value": tv, "unit": UNIT, "ms_per_step": tms, "steps": nt,
                 "backward_ms": round(bwd, 4),
                 "backward_kernels_ms": {n: round(v, 4) for n, v in
                                         sorted(bk.items(), key=lambda kv: -kv[1])},
                 "forward_tflop": round(fwd_tf, 3),
                 "note": "forward + backward of the layer; weight gradients fp32"}

    # ---- CPU oracle baseline (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_tok = args.cpu_sample or 4096
        scfg, host = oracle_inputs(cfg, inp, n_tok)
        n = scfg.T
        sec = time_oracle(scfg, host)
        del host
        cpu = {"value": n / sec, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
               "sample": f"first {n} tokens of the batch as a T={n} layer of the same widths "
                         f"({n // cfg.n_ranks} per source rank), one float64 NumPy pass, "
                         f"{sec:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{cfg.name}: T={cfg.T} tokens ({cfg.n_seqs} x {cfg.T // max(1, cfg.n_seqs)}), "
                       f"d={cfg.d_model}, L={cfg.d_latent}, E={cfg.n_experts} on {cfg.n_ranks} logical ranks, "
                       f"top-{cfg.top_k}, {cfg.n_waves} waves, {cfg.n_shared} shared (Hs={cfg.h_shared}), "
                       f"H={cfg.h_expert}, cf {cfg.cf_send}/{cfg.cf_recv}",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "pool_fill": pipeline,
                       "expert_path": ("CTA pairs, expert rows on the MMA's N axis from the "
                                       "per-expert bank" if m.bank is not None
                                       else "rows gathered from the pool"),
                       "l2": "inputs larger than L2 (8.1 GB weights per step)"},
            "assignments_per_s": value * cfg.top_k,
            "drops": {"near_tie_tokens": near_ties,
                      "kept": st["kept"], "dropped_send": st["dropped_send"],
                      "dropped_recv": st["dropped_recv"],
                      "drop_rate": (st["dropped_send"] + st["dropped_recv"]) / max(1, st["assignments"])},
            "gpu_launches": sum(v[1] for v in per.values()),
            "roofline": roof, "kernels": kernels, "expert_ffn": expert_ffn, "clocks": clk,
            "e2e": e2e,
            "graph_replay": graph, "pipelines": pipes, "dropless": dropless, "train_step": train,
            "workloads": others,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_gb300(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
