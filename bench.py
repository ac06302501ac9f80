"""Decode throughput of the prerouted int4 MoE stack on GB300.

Workload: the 35B-tier 40-layer stack (d=2048, 256 experts, top-4, expert and
shared intermediate 512, prerouter heads on layers 6-38 with hidden 512, LoRA
r=16 alpha=32 on the shared expert), batch 1, synthetic seeded weights.  One
bench step = one decode step = all 40 layers for one token = one launch of the
persistent engine kernel (edge0_decode_step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  `value` is decode tokens/s with inputs resident in HBM;
`e2e` the same through the C ABI with pinned host buffers copied in and out
every step; `roofline` the engine kernel's achieved HBM GB/s against the
measured copy bandwidth; `cpu_baseline` the CPU oracle on a bounded sample.
--impl reference times the CPU oracle (the reference arm of this build).
Multi-GPU runs are independent replicas (no collective on the data path).
"""
from __future__ import annotations

import argparse
import platform
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from int4_routed_expert_prerouter_gb300 import configs  # noqa: E402

METRIC = "decode tokens/s (1 GB300, 35B-tier MoE stack) and achieved HBM GB/s vs roofline"
CFG = configs.STACK35


# ---------------------------------------------------------------- bytes ----
def algorithmic_bytes_per_token(cfg, own_routed_layers):
    """Bytes a decode step must read once (int4 experts with scales, shared
    expert, head dense parts + gathered one-hot columns, LoRA factors, router of
    each layer that routes itself)."""
    q4 = configs.q4_bytes
    expert = configs.expert_bytes(cfg.d, cfg.I)
    shared = configs.expert_bytes(cfg.d, cfg.Is)
    head = (cfg.H * cfg.d + cfg.E * cfg.d + cfg.E * cfg.H) * 2 + 2 * cfg.K * (cfg.H + cfg.E) * 2
    lora = (2 * (cfg.r * cfg.d + cfg.Is * cfg.r) + (cfg.r * cfg.Is + cfg.d * cfg.r)) * 2
    router = cfg.E * cfg.d * 2
    n_heads = len(cfg.head_owners())
    total = cfg.L * (cfg.K * expert + shared + lora) + n_heads * head + own_routed_layers * router
    del q4
    return total


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = ("int4_routed_expert_prerouter_gb300/csrc/decode1.cu",
                  "int4_routed_expert_prerouter_gb300/csrc/internal.cuh",
                  "int4_routed_expert_prerouter_gb300/csrc/common.cuh",
                  "include/edge0.h")
# the committed DRAM-traffic record of the benched kernel (from an ncu capture)
TRAFFIC_RECORD = "decode1_35b_stack_traffic.txt"


def kernel_source_hash():
    """Hash of the code the benched kernel is compiled from: its sources with the
    comments and whitespace taken out (a comment edit does not change the
    kernel), and of the public header only the constants (#define lines) that
    the kernel uses (a new host-side declaration does not change it either)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        text = open(os.path.join(ROOT, f), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        if f.endswith("edge0.h"):
            text = "\n".join(line for line in text.splitlines() if line.lstrip().startswith("#define"))
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per token of the benched kernel from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", TRAFFIC_RECORD)
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha") != kernel_source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_token"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------- clocks ----
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        load = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in load:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                            ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(load)}


# ------------------------------------------------------ multi-replica -----
def job_times(times_ms, world, device):
    """Replicas (one process per GPU, no collective on the data path) time
    their own regions; the job takes as long as the slowest: the max over ranks
    of each time."""
    local = torch.tensor(times_ms, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(local, op=torch.distributed.ReduceOp.MAX)
    return local.tolist()


def job_throughput(tokens_all_ranks, region_ms):
    """Whole-job throughput: the tokens every rank decoded over the job's time."""
    return tokens_all_ranks / (region_ms / 1e3)


# ------------------------------------------------------------ GPU arm -----
def run_gpu(args, rank, world):
    from int4_routed_expert_prerouter_gb300 import binding, inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    cfg = configs.CONFIGS[args.config]
    if args.layers or args.experts:
        # reduced case for profiler captures only (same per-layer shapes)
        L = args.layers or cfg.L
        cfg = cfg.with_(L=L, E=args.experts or cfg.E, head_owner_last=min(cfg.head_owner_last, L - 2),
                        prerouted=tuple(l for l in cfg.prerouted if l < L - 1))
    model = inputs.make_model(cfg, seed=args.seed, device=dev, small_device=dev)
    dm = binding.DeviceModel(model, dev)
    cpu_model = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu_model = _host_layers(model, args.cpu_layers)
    del model
    torch.cuda.empty_cache()
    st = binding.DecodeState(cfg, device=dev)
    stream = torch.cuda.current_stream(dev)
    B, d = cfg.B, cfg.d
    # one fresh seeded hidden state per step (each step's h_0), updated in place
    n_in = args.warmup + 2 * args.steps
    h_all = torch.empty(n_in, B, d, dtype=torch.float16, device=dev)
    for i in range(n_in):
        h_all[i].copy_(inputs.hidden(cfg, i, seed=args.seed, device=dev))

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    # warm-up (includes step 0, where every layer routes by its own router)
    t = 0
    for _ in range(args.warmup):
        binding.decode_step(dm, st, h_all[t], t)
        t += 1
    barrier()
    err = st.error()
    assert err == 0, f"kernel error during warm-up: {binding.status_string(err)}"

    if args.trace:
        st.set_trace(True)
        binding.decode_step(dm, st, h_all[t], t)
        t += 1
        st.set_trace(False)
        tr = st.read_trace()
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        own = [l for l in range(cfg.L) if l not in cfg.prerouted]
        pre = list(cfg.prerouted)
        print_trace(tr, nsm, ([pre[len(pre) // 2]] if pre else []) + (own[1:2] if len(own) > 1 else own))
        if args.trace_file:
            np.savez_compressed(args.trace_file, consumer=tr[0].numpy(), producer=tr[1].numpy())
    # device-resident timed region: one event pair per launch for the kernel
    # duration, one pair around the region for the step time
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            binding.decode_step(dm, st, h_all[t], t)
            ev[i][1].record(stream)
            t += 1
        t_end.record(stream)
        barrier()
    err = st.error()
    assert err == 0, f"kernel error in the timed region: {binding.status_string(err)}"
    region_ms = t_start.elapsed_time(t_end)
    kern_ms = [a.elapsed_time(b) for a, b in ev]

    # end to end through the C ABI: pinned host input -> device, decode step,
    # device -> pinned host output, every step
    h_host_in = torch.empty(args.steps, B, d, dtype=torch.float16).pin_memory()
    for i in range(args.steps):
        h_host_in[i].copy_(inputs.hidden(cfg, t + i, seed=args.seed))
    h_host_out = torch.empty(args.steps, B, d, dtype=torch.float16).pin_memory()
    h = torch.empty(B, d, dtype=torch.float16, device=dev)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    barrier()
    e_start.record(stream)
    for i in range(args.steps):
        h.copy_(h_host_in[i], non_blocking=True)
        binding.decode_step(dm, st, h, t)
        h_host_out[i].copy_(h, non_blocking=True)
        t += 1
    e_end.record(stream)
    barrier()
    e2e_ms = e_start.elapsed_time(e_end)
    assert st.error() == 0

    region_ms, e2e_ms = job_times([region_ms, e2e_ms], world, dev)
    if rank != 0:
        return None

    tokens = B * args.steps * world
    value = job_throughput(tokens, region_ms)
    e2e_value = tokens / (e2e_ms / 1e3)
    own = cfg.L - len(cfg.prerouted)
    bytes_tok = algorithmic_bytes_per_token(cfg, own)
    mean_kern_s = statistics.mean(kern_ms) / 1e3
    peak, peak_kind = measured_peaks()
    achieved = bytes_tok / mean_kern_s / 1e9
    traffic = profiled_traffic()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(region_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int4xf16",
        "data": "synthetic",
        "config": {
            "workload": (f"{cfg.name}: {cfg.description}" if not (args.layers or args.experts) else
                         f"REDUCED profiling case: {cfg.L} layers, {cfg.E} experts, shapes of {CFG.name}"),
            "layers": cfg.L, "d_model": cfg.d, "experts": cfg.E, "top_k": cfg.K,
            "batch": B, "seq_len": 1, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (%.0f MB of weights read per step > 129 MB)" % (bytes_tok / 1e6),
            "layers_per_s": round(value * cfg.L / world, 1),
        },
        "e2e": {"value": round(e2e_value, 2), "unit": "tokens/s",
                "h2d_bytes_per_step": B * d * 2, "d2h_bytes_per_step": B * d * 2},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": None if traffic is None else int(traffic),
                     "kernel": "edge0::d1::decode1_kernel (one launch per decode step)",
                     "algorithmic_bytes_per_launch": bytes_tok,
                     "mean_launch_us": round(mean_kern_s * 1e6, 2),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
        "clocks": clk.summary(),
    }
    if cpu_model is not None:
        line["cpu_baseline"] = cpu_baseline(cpu_model, args)
    return line


def batched_bytes_per_step(cfg, exec_ids, own_routed):
    """Algorithmic bytes of one batched decode step: each layer's distinct routed
    experts once (however many tokens they serve), the shared expert and LoRA
    factors, every head's dense parts once and its gathered one-hot columns per
    token, and the router of each layer that routes itself.  exec_ids: [L, B, K]
    of the step."""
    expert = configs.expert_bytes(cfg.d, cfg.I)
    shared = configs.expert_bytes(cfg.d, cfg.Is)
    lora = (2 * (cfg.r * cfg.d + cfg.Is * cfg.r) + (cfg.r * cfg.Is + cfg.d * cfg.r)) * 2
    head_dense = (cfg.H * cfg.d + cfg.E * cfg.d + cfg.E * cfg.H) * 2
    head_cols = 2 * cfg.K * (cfg.H + cfg.E) * 2
    total = 0
    for l in range(cfg.L):
        total += len(np.unique(exec_ids[l])) * expert + shared + lora
    total += len(cfg.head_owners()) * (head_dense + cfg.B * head_cols) + own_routed * cfg.E * cfg.d * 2
    return total


def run_batched(args, rank, world, cfg):
    """The batched decode path (cfg.B > 4 sequences): one bench step = one decode
    step of all sequences; with a host tier (cfg.pool_frac), the experts each
    prerouted layer's prediction names are prefetched after every step (part of
    the timed step: it waits for that step's predictions)."""
    from int4_routed_expert_prerouter_gb300 import binding, inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    if args.layers:
        # reduced case for profiler captures only (same per-layer shapes)
        cfg = cfg.with_(L=args.layers, head_owner_last=min(cfg.head_owner_last, args.layers - 2),
                        prerouted=tuple(l for l in cfg.prerouted if l < args.layers - 1))
    model = inputs.make_model(cfg, seed=args.seed, device=dev, small_device=dev)
    dm = binding.DeviceModel(model, dev)
    del model
    torch.cuda.empty_cache()
    pool = binding.ExpertPool(dm, int(cfg.E * cfg.pool_frac)) if cfg.pool_frac else None
    torch.cuda.empty_cache()
    st = binding.DecodeState(cfg, device=dev)
    stream = torch.cuda.current_stream(dev)
    B, d = cfg.B, cfg.d
    prerouted = list(cfg.prerouted)
    n_in = args.warmup + 3 * args.steps
    h_all = torch.empty(n_in, B, d, dtype=torch.float16, device=dev)
    for i in range(n_in):
        h_all[i].copy_(inputs.hidden(cfg, i, seed=args.seed, device=dev))

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    # host-tier arms: the device-planned prefetch of the prerouted layers'
    # predictions, with least-recently-used caching of the executed experts on
    # the layers that route themselves (the product path); least-recently-used
    # caching of every layer's executed experts, no prediction; or no copies at
    # all (resident set frozen).  The plan is enqueued after the step's head flush on
    # the compute stream; the copies run on the pool's copy stream; nothing waits.
    own_layers = [l for l in range(cfg.L) if l not in prerouted]

    def step(t, prefetch="prediction"):
        binding.decode_step(dm, st, h_all[t % n_in], t)
        if pool is not None and prefetch == "prediction":
            pool.prefetch(st, t, predicted=prerouted, cached=own_layers)
        elif pool is not None and prefetch == "executed":
            pool.prefetch(st, t, cached=range(cfg.L))

    if pool is not None:
        # an empty pool fills at ~200 copies per step: 64 slots x 40 layers take
        # a dozen steps or more before the arm reaches its steady state
        args.warmup = max(args.warmup, 24)
    t = 0
    for _ in range(args.warmup):
        step(t)
        t += 1
    barrier()
    err = st.error()
    assert err == 0, f"kernel error during warm-up: {binding.status_string(err)}"

    def timed(prefetch="prediction"):
        nonlocal t
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        a.record(stream)
        for _ in range(args.steps):
            step(t, prefetch)
            t += 1
        b.record(stream)
        barrier()
        return a.elapsed_time(b)

    def arm_record(ms, s0, s1, c0, c1):
        """The arm's residency over its timed steps, from the device counters:
        cold fraction = executed (layer, expert) pairs read from host memory;
        loads = whole-expert transfers from host memory, either copies made off
        the critical path or reads inside the expert kernels."""
        ebytes = pool.gu_bytes + pool.dn_bytes
        dt = c1 - c0                                     # [L, 2]
        pre = np.array(prerouted, dtype=np.int64)
        act, cold = dt[:, 0].sum(), dt[:, 1].sum()
        copies = s1["published"] - s0["published"]
        return {
            "tokens_per_s": round(B * args.steps / (ms / 1e3), 2),
            "ms_per_step": round(ms / args.steps, 3),
            "cold_fraction": round(cold / max(act, 1), 4),
            "cold_fraction_prerouted_layers": round(dt[pre, 1].sum() / max(dt[pre, 0].sum(), 1), 4),
            "active_experts_per_step": round(act / args.steps, 1),
            "copies_per_step": round(copies / args.steps, 2),
            "copied_mb_per_step": round((s1["bytes"] - s0["bytes"]) / args.steps / 1e6, 1),
            "host_reads_per_step": round(cold / args.steps, 2),
            "host_read_mb_per_step": round(cold * ebytes / args.steps / 1e6, 1),
            "loads_per_step": round((copies + cold) / args.steps, 2),
            "mib_per_load": round(ebytes / 2 ** 20, 3),
            "failed_copies": s1["failed"] - s0["failed"],
            "plans_skipped": s1["skipped"] - s0["skipped"],
            "hit_rate": round((s1["hits"] - s0["hits"]) / max(s1["requests"] - s0["requests"], 1), 4),
        }

    if pool is not None:
        s0, c0 = pool.stats(), pool.tiers()
    with ClockSampler(dev.index) as clk:
        region_ms = timed()
    err = st.error()
    assert err == 0, f"kernel error in the timed region: {binding.status_string(err)}"
    # bytes from the routing of the last two timed steps
    ex = st.exec_ids.cpu().numpy()
    own = cfg.L - len(cfg.prerouted)
    step_bytes = statistics.mean(batched_bytes_per_step(cfg, ex[p], own) for p in (0, 1))
    arms = {}
    if pool is not None:
        arms["prediction"] = arm_record(region_ms, s0, pool.stats(), c0, pool.tiers())
        for arm in ("executed", None):
            for _ in range(args.warmup):   # the arm's steady state
                step(t, arm)
                t += 1
            barrier()
            s0, c0 = pool.stats(), pool.tiers()
            ms = timed(prefetch=arm)
            arms[arm or "frozen"] = arm_record(ms, s0, pool.stats(), c0, pool.tiers())
        assert st.error() == 0

    # end to end: pinned host input -> device, decode step, device -> host, every step
    h_host = torch.empty(args.steps, B, d, dtype=torch.float16).pin_memory()
    for i in range(args.steps):
        h_host[i].copy_(inputs.hidden(cfg, t + i, seed=args.seed))
    h = torch.empty(B, d, dtype=torch.float16, device=dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    a.record(stream)
    for i in range(args.steps):
        h.copy_(h_host[i], non_blocking=True)
        binding.decode_step(dm, st, h, t)
        if pool is not None:
            pool.prefetch(st, t, predicted=prerouted, cached=own_layers)
        h_host[i].copy_(h, non_blocking=True)
        t += 1
    b.record(stream)
    barrier()
    e2e_ms = a.elapsed_time(b)
    assert st.error() == 0

    region_ms, e2e_ms = job_times([region_ms, e2e_ms], world, dev)
    if rank != 0:
        return None
    tokens = B * args.steps * world
    value = job_throughput(tokens, region_ms)
    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (region_ms / args.steps / 1e3) / 1e9
    line = {
        "metric": f"decode tokens/s (1 GB300, {cfg.name}, {B} sequences) and achieved HBM GB/s vs roofline",
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(region_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int4xf16",
        "data": "synthetic",
        "config": {
            "workload": (f"{cfg.name}: {cfg.description}" if not args.layers else
                         f"REDUCED profiling case: {cfg.L} layers, shapes of {cfg.name}"),
            "layers": cfg.L, "d_model": d, "experts": cfg.E, "top_k": cfg.K, "batch": B, "seq_len": 1,
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (%.0f MB of weights read per step > 129 MB)" % (step_bytes / 1e6),
            "layers_per_s": round(value / B * cfg.L / world, 1),
        },
        "e2e": {"value": round(tokens / (e2e_ms / 1e3), 2), "unit": "tokens/s",
                "h2d_bytes_per_step": B * d * 2, "d2h_bytes_per_step": B * d * 2},
        # per layer: norm, dispatch, LoRA A (both matrices), gate/up, down, LoRA
        # down; + router and top-K on own-routed layers; final residual; the head
        # flush: fc1, one-hot + GELU, fc2, linear_init, one-hot, top-K, each one
        # launch over all heads; + the pool's planner and copy kernel
        "gpu_launches": args.steps * (6 * cfg.L + 2 * own + 1 + (6 if cfg.head_owners() else 0)
                                      + (2 if pool is not None else 0)),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "batched decode step (per layer: norm, routing, dispatch, gate/up, down, LoRA; "
                               "head flush), algorithmic bytes from the step's routing over the step time",
                     "algorithmic_bytes_per_step": int(step_bytes),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
        "clocks": clk.summary(),
    }
    if pool is not None:
        line["pool"] = {"slots_per_layer": pool.n_slots, "experts": cfg.E,
                        "prefetch_hit_rate": arms["prediction"]["hit_rate"],
                        "experts_copied_per_step": arms["prediction"]["copies_per_step"],
                        "prefetch_off_tokens_per_s": arms["frozen"]["tokens_per_s"],
                        "prefetch_off": "no copies: resident set frozen, misses read from host memory",
                        "arms": arms,
                        "arms_note": ("prediction: device-planned prefetch of the prerouted layers' predicted "
                                      "experts, LRU caching of the executed experts on the self-routed "
                                      "layers, copies on a second stream, nothing waits (the timed line); "
                                      "executed: the same pool caching every layer's executed experts (LRU, "
                                      "no prediction); frozen: no copies. Each arm measured over its own "
                                      "timed steps from the device counters: cold_fraction = executed "
                                      "(layer, expert) pairs read from host memory when their layer "
                                      "dispatched; a load = one expert's packed gate/up + down moved from "
                                      "host memory, by a copy off the critical path or by the expert "
                                      "kernels' own reads")}
    return line


TRACE_POINTS = {0: "start", 0x21: "y in", 2: "x", 4: "routing", 9: "b1 ready", 0x27: "gate/up MMAs",
                5: "gate/up", 7: "act out", 10: "b2 ready", 0x25: "down MMAs", 8: "y out"}


def print_trace(tr, nct, layers, sm_mhz=2070.0):
    """One traced decode step of the batch-1 kernel.  For the given layers, the
    segments between consecutive trace points of each CTA (SM cycle counter),
    mean and max over the CTAs that pass both points; the period of every layer
    (globaltimer at CTA 0's layer starts); the head flush per task (blocks
    waited for, task computed) summed over a CTA's tasks."""
    cons = tr[0]
    lines = []
    us = lambda cyc: cyc / sm_mhz
    starts = {}
    seg = {l: {} for l in layers}
    flush = []
    for c in range(nct):
        ev = {}
        for tag, tm, cy in cons[c].tolist():
            if tm != 0 and tag not in ev:
                ev[tag] = (tm, cy)
        if c == 0:
            starts = {k >> 8: v[0] for k, v in ev.items() if k < 0xF000 and (k & 0xFF) == 0}
        for l in layers:
            pts = sorted(((v[1], k & 0xFF) for k, v in ev.items() if k < 0xF000 and k >> 8 == l))
            nxt = ev.get((l + 1) << 8)
            if nxt:
                pts.append((nxt[1], 0x100))
            for (ca, ka), (cb, kb) in zip(pts, pts[1:]):
                name = f"{TRACE_POINTS.get(ka, hex(ka))} -> {TRACE_POINTS.get(kb, 'next layer') if kb != 0x100 else 'next layer'}"
                seg[l].setdefault(name, []).append(us(cb - ca))
        tasks = sorted({k & 0xFF for k in ev if 0xF100 <= k < 0xF200})
        if tasks:
            wait = sum(us(ev[0xF200 | t][1] - ev[0xF100 | t][1]) for t in tasks if 0xF200 | t in ev)
            work = sum(us(ev[0xF300 | t][1] - ev[0xF200 | t][1]) for t in tasks if 0xF300 | t in ev)
            first = ev[0xF100 | tasks[0]][0]
            last = max(ev[0xF300 | t][0] for t in tasks if 0xF300 | t in ev)
            flush.append((len(tasks), wait, work, (last - first) / 1e3))
    for l in layers:
        lines.append(f"layer {l}: " + "; ".join(
            f"{n} {statistics.mean(v):.2f}/{max(v):.2f}" for n, v in seg[l].items()) + " us (mean/max over CTAs)")
    ls = sorted(starts)
    per = [(l, (starts[l + 1] - starts[l]) / 1e3) for l in ls if l + 1 in starts]
    lines.append("layer periods (CTA 0, us): " + " ".join(f"{l}:{v:.1f}" for l, v in per))
    if flush:
        lines.append("head flush per CTA: tasks %.1f, block waits %.2f us, compute %.2f us, span %.2f us (mean)" % tuple(
            statistics.mean(f[i] for f in flush) for i in range(4)))
    sys.stderr.write("\n".join(lines) + "\n")


def _host_layers(model, n):
    """Host copy of layers [6, 6 + n) (a head owner and prerouted layers) for the
    CPU baseline sample."""
    from int4_routed_expert_prerouter_gb300 import inputs
    c = lambda trip: tuple(t.cpu() for t in trip)
    cfg = model.cfg.with_(L=n, head_owner_first=0, head_owner_last=n - 1, prerouted=tuple(range(n)),
                          ring=False)
    m = inputs.Model(cfg, model.seed)
    for l in range(6, 6 + n):
        lw = model.layers[l]
        hd = None if lw.head is None else {k: (v.cpu() if torch.is_tensor(v) else v)
                                           for k, v in lw.head.items()}
        if hd is not None:
            hd["target"] = min(l - 6 + 1, n - 1)
        m.layers.append(inputs.LayerWeights(c(lw.gate), c(lw.up), c(lw.down), c(lw.sh_gate),
                                            c(lw.sh_up), c(lw.sh_down), lw.router.cpu(),
                                            lw.gamma.cpu(), {k: v.cpu() for k, v in lw.lora.items()},
                                            None, hd, True))
    return m


def host_cpu():
    """The host's hardware threads and CPU model (for the CPU-side records)."""
    model = platform.processor() or platform.machine()
    try:
        info = open("/proc/cpuinfo").read().splitlines()
        names = [l.split(":", 1)[1].strip() for l in info if l.lower().startswith("model name")]
        if names:
            model = names[0]
        else:   # Arm: implementer and part numbers
            impl = [l.split(":", 1)[1].strip() for l in info if l.startswith("CPU implementer")]
            part = [l.split(":", 1)[1].strip() for l in info if l.startswith("CPU part")]
            known = {("0x41", "0xd4f"): "Arm Neoverse-V2", ("0x41", "0xd40"): "Arm Neoverse-V1",
                     ("0x41", "0xd0c"): "Arm Neoverse-N1"}
            if impl and part:
                model = known.get((impl[0], part[0]), f"Arm implementer {impl[0]} part {part[0]}")
    except OSError:
        pass
    return {"host_threads": os.cpu_count(), "cpu_model": f"{model} ({platform.machine()})"}


def cpu_baseline(cpu_model, args):
    """The CPU oracle (single-threaded C++, fp64) on a bounded sample: decode
    steps of `cpu_layers` 35B-shaped layers (each with a head, prerouted from
    the second step), scaled to tokens/s of the 40-layer stack."""
    import oracle
    from int4_routed_expert_prerouter_gb300 import inputs
    cfg = cpu_model.cfg
    stack = oracle.Stack(cpu_model)
    per_layer = []
    for t in range(args.cpu_steps):
        h = inputs.hidden(cfg, t, seed=args.seed)
        t0 = time.perf_counter()
        stack.step(h, t, record=False)
        per_layer.append((time.perf_counter() - t0) / cfg.L)
    sec_per_layer = statistics.mean(per_layer[1:] if len(per_layer) > 1 else per_layer)
    tok_s = 1.0 / (sec_per_layer * CFG.L)
    return {"value": round(tok_s, 5), "unit": "tokens/s", "cores": 1, "kind": "oracle", **host_cpu(),
            "sample": f"{args.cpu_steps} decode steps of {cfg.L} 35B-tier layers (layers 6..{5 + cfg.L} "
                      f"of the stack, each with its head; first step excluded), "
                      f"{sec_per_layer:.3f} s per layer, scaled to {CFG.L} layers per token"}


# ------------------------------------------------------ reference arm -----
def run_reference(args, rank):
    """The reference arm of this build: the CPU oracle as it stands, on host
    cores, each bench step one 35B-tier layer of a decode step (a bounded
    sample), reported in tokens/s of the 40-layer stack."""
    if rank != 0:
        return None
    import oracle
    from int4_routed_expert_prerouter_gb300 import inputs
    cfg = CFG.with_(L=2, head_owner_first=0, head_owner_last=0, prerouted=(1,))
    model = inputs.make_model(cfg, seed=args.seed)
    stack = oracle.Stack(model)
    h = inputs.hidden(cfg, 0, seed=args.seed)
    for t in range(args.warmup):
        stack.step(h, t, record=False, layers=[t % 2])
    times = []
    for i in range(args.steps):
        t = args.warmup + i
        t0 = time.perf_counter()
        stack.step(h, t, record=False, layers=[i % 2])
        times.append(time.perf_counter() - t0)
    sec_layer = statistics.mean(times)
    value = 1.0 / (sec_layer * CFG.L)
    sample = (f"{args.steps} steps, each one 35B-tier layer (d=2048, E=256, K=4, shared expert, "
              f"LoRA, head on the first) of a decode step on the CPU oracle, scaled to 40 layers")
    return {"metric": METRIC, "value": round(value, 5), "unit": "tokens/s", "impl": "reference",
            "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec_layer * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{CFG.name}: {CFG.description}", "batch": 1, "seq_len": 1,
                       "parallelism": "single host thread"},
            "cpu_baseline": {"value": round(value, 5), "unit": "tokens/s", "cores": 1,
                             "kind": "oracle", **host_cpu(), "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------- prefill -----
def run_prefill(args, rank):
    """The whole-layer prefill of a prompt of args.prefill tokens through the 40
    layers of the 35B-tier stack, every layer on its own router: tokens/s, with
    the roofline of the step's algorithmic bytes (every expert the prompt
    activates read once per layer, the shared expert, LoRA factors, router)
    over the measured HBM peak.  Its own JSON line (not the decode bench line)."""
    from int4_routed_expert_prerouter_gb300 import binding, inputs
    cfg = configs.CONFIGS[args.config]
    if args.layers:   # reduced case for profiler captures
        cfg = cfg.with_(L=args.layers, head_owner_last=min(cfg.head_owner_last, args.layers - 2),
                        prerouted=tuple(l for l in cfg.prerouted if l < args.layers - 1))
    T = args.prefill
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    model = inputs.make_model(cfg, seed=args.seed, device=dev, small_device=dev)
    dm = binding.DeviceModel(model, dev)
    ws = torch.empty(binding.prefill_workspace_bytes(cfg, T), dtype=torch.uint8, device=dev)
    ids = torch.zeros(cfg.L, T, cfg.K, dtype=torch.int32, device=dev)
    h0 = inputs.hidden(cfg.with_(B=T), 0, seed=args.seed, device=dev)
    stream = torch.cuda.current_stream(dev)
    flags = binding.PREFILL_TCGEN05_GATE_UP if args.prefill_tcgen05 else 0
    steps = args.steps or 5
    warm = args.warmup if args.warmup is not None else 3
    h = h0.clone()
    for _ in range(warm):
        h.copy_(h0)
        binding.prefill(dm, h, ws, ids_out=ids, flags=flags)
    torch.cuda.synchronize(dev)
    # algorithmic bytes of one prefill: the experts each layer's routing activates
    active = sum(int(torch.unique(ids[l]).numel()) for l in range(cfg.L))
    expert, shared = configs.expert_bytes(cfg.d, cfg.I), configs.expert_bytes(cfg.d, cfg.Is)
    lora = (2 * (cfg.r * cfg.d + cfg.Is * cfg.r) + (cfg.r * cfg.Is + cfg.d * cfg.r)) * 2
    router = cfg.E * cfg.d * 2
    step_bytes = active * expert + cfg.L * (shared + lora + router) + 2 * T * cfg.d * 2
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize(dev)
        for i in range(steps):
            h.copy_(h0)
            ev[i][0].record(stream)
            binding.prefill(dm, h, ws, ids_out=ids, flags=flags)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    peak, src = measured_peaks()
    achieved = step_bytes / (ms * 1e-3) / 1e9
    line = {"metric": f"prefill tokens/s (1 GB300, 35B-tier 40-layer stack, prompt of {T} tokens)",
            "value": round(T / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": steps, "warmup": warm,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int4xf16", "data": "synthetic",
            "config": {"workload": f"{cfg.name} prefill: {T} prompt tokens through {cfg.L} layers, own routing",
                       "tokens": T, "layers": cfg.L,
                       "gate_up_kernel": "tcgen05" if flags else "mma.sync", "active_experts_per_layer": round(active / cfg.L, 1),
                       "l2": "inputs larger than L2 (every prefill reads the layers' experts from HBM)"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": None,
                         "algorithmic_bytes_per_step": int(step_bytes), "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)"},
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-layers", type=int, default=4)
    ap.add_argument("--cpu-steps", type=int, default=10)
    ap.add_argument("--layers", type=int, default=0, help="reduced case for profiler captures")
    ap.add_argument("--experts", type=int, default=0, help="reduced case for profiler captures")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill", type=int, default=0,
                    help="time the whole-layer prefill of a prompt of this many tokens instead")
    ap.add_argument("--prefill-tcgen05", action="store_true", help="with --prefill: the tcgen05 gate/up kernel")
    ap.add_argument("--trace", action="store_true", help="print a per-phase split of one step")
    ap.add_argument("--trace-file", default=None, help="with --trace: save the raw per-CTA trace (.npz)")
    ap.add_argument("--config", default=CFG.name, choices=sorted(configs.CONFIGS),
                    help="workload; the batched configurations (B > 4) run the batched path")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.prefill:
        run_prefill(args, rank)
        return
    if args.impl == "reference":
        args.steps = 12 if args.steps is None else args.steps
        args.warmup = 3 if args.warmup is None else args.warmup
        line = run_reference(args, rank)
    else:
        args.steps = 512 if args.steps is None else args.steps
        args.warmup = 8 if args.warmup is None else args.warmup
        assert args.warmup >= 3
        if world > 1:
            torch.distributed.init_process_group("nccl")
        import __graft_entry__
        __graft_entry__.build()
        cfg = configs.CONFIGS[args.config]
        if cfg.B > 4:
            if args.steps == 512:
                args.steps = 16
            line = run_batched(args, rank, world, cfg)
        else:
            line = run_gpu(args, rank, world)
        if world > 1:
            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
