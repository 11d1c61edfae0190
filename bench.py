"""Benchmark of the NVFP4 MegaMoE routed-expert forward.

One step = one megamoe_forward (route -> amax -> quantise -> L1 grouped GEMM
with SiLU*up -> requantise -> L2 grouped GEMM -> combine) over one batch of
the largest single-GPU MegaMoE workload (384 experts, top-6, d 7168, I 2048,
16384 tokens with uniform routing, NVFP4 weights resident in HBM).  Prints one
JSON line; beside the headline it carries sub-records of the 4096-token
Zipf-skewed prefill and of the 8- and 1-token decode batches, each with its
own roofline and stage times.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config large]
                  [--no-sub] [--impl ours|reference]

--impl reference times the CPU oracle (the float64 reference of the method)
on a bounded sample of the same workload.  Under torchrun every rank runs its
own replica (the path has no exchange step); rank 0 prints.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "routed tokens/s and NVFP4 TFLOP/s per MoE layer fwd; % HBM / FP4 roofline"
UNIT = "routed tokens/s"
# kernels of one forward: route, amax, quant, L1 GEMM, requant, L2 GEMM,
# combine; batches of at most 262144 elements of x run route+amax as one
# kernel, and from 16384 slots on the routing is three kernels (per-block
# histograms, offsets, scatter)
PROLOGUE_MAX_ELEMS = 262144
MULTI_BLOCK_ROUTE_SLOTS = 16384


def kernels_per_step(cfg) -> int:
    if cfg.T * cfg.d <= PROLOGUE_MAX_ELEMS:
        return 6
    return 9 if cfg.T * cfg.k >= MULTI_BLOCK_ROUTE_SLOTS else 7


# kernels of one dense linear: prologue (status, offsets, amax of up to this
# many elements of x), amax of larger inputs, quantiser, GEMM, and the split-K
# finishing kernel when the call splits K
LINEAR_PROLOGUE_MAX_ELEMS = 262144


def linear_kernels_per_call(T: int, K: int, ws_bytes: int) -> int:
    """Launches of one megamoe_linear_nvfp4 call.  Whether it splits K shows in
    its workspace size: the split-K planes follow the header, codes and scales."""
    def a256(n):
        return -(-n // 256) * 256

    split = ws_bytes > 256 + a256(T * (K // 2)) + a256(T * (K // 16))
    return 3 + int(T * K > LINEAR_PROLOGUE_MAX_ELEMS) + int(split)


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        return summarize_clocks(self.lines)


def summarize_clocks(lines):
    """The `clocks` object from ClockSampler.FIELDS lines (csv, no header, no
    units): median and max SM clock, and every throttle reason seen Active."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm.append(float(parts[0]))
            mx.append(float(parts[1]))
        except ValueError:
            continue
        for n, v in zip(names, parts[4:8]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
            "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_hash() -> str:
    """sha256 (16 hex digits) of the grouped-GEMM kernel sources."""
    h = hashlib.sha256()
    for name in ("gemm.cu", "gemm_tm.cu", "gemm_common.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "nvfp4_block_scaled_topk_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profile_traffic(name: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel
    sources are unchanged since the capture (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", name)) as f:
            prof = json.load(f)
        if prof.get("source_sha256_16") != kernel_source_hash():
            return None
        return prof.get("dram_bytes_per_launch")
    except Exception:
        return None


# --------------------------------------------------------------------------
# the oracle leg (cpu_baseline and --impl reference)
# --------------------------------------------------------------------------
def oracle_sample(cfg, x, ids, w, ex, tokens: int):
    """Time the CPU oracle's forward on the first `tokens` tokens.  ``ex`` is
    an ExpertSet; the experts those tokens touch are drawn (or fetched from
    the GPU) before the clock starts, so only the oracle's own work is timed."""
    import numpy as np

    import oracle

    xs = x[:tokens].float().cpu().numpy()
    ids_s = ids[:tokens].cpu().numpy()
    ws = w[:tokens].cpu().numpy()
    for e in np.unique(ids_s[ids_s >= 0]):
        ex[int(e)]
    t0 = time.perf_counter()
    out = oracle.forward(xs, ids_s, ws, ex, pad=cfg.pad)
    dt = time.perf_counter() - t0
    assert np.all(np.isfinite(out))
    return dt


def max_over_ranks(values, world: int, device="cpu"):
    """Element-wise maximum of `values` over all ranks (identity at world 1)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    import torch

    from nvfp4_block_scaled_topk_gb300 import inputs

    rank, world, _ = _dist()
    if rank != 0:
        return
    import numpy as np

    cfg = inputs.CONFIGS[args.config]
    x = inputs.make_activations(cfg)
    ids, w = inputs.make_routing(cfg)
    flat = ids.numpy().reshape(-1)
    counts = np.bincount(flat[(flat >= 0) & (flat < cfg.E)], minlength=cfg.E)
    tokens = max(1, min(cfg.T, args.ref_tokens))
    ex = inputs.ExpertSet(cfg, None)  # experts drawn on the CPU once, on first use
    times = []
    for i in range(args.warmup + args.steps):
        dt = oracle_sample(cfg, x, ids, w, ex, tokens)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = tokens * len(times) / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(cfg, counts, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                         "sample": f"each step: the first {tokens} of {cfg.T} tokens of the "
                                   f"{cfg.name} batch, full float64 forward over the experts "
                                   "they touch; weights fetched before timing"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(cfg, counts, world):
    """The `config` object of a forward workload, the same for both arms:
    its name and sizes and the routing's per-expert row counts (`counts`, from
    the library's routing or, for the reference arm, counted on the host from
    the same seeded ids)."""
    import numpy as np

    counts = np.asarray(counts)
    active = int((counts > 0).sum())
    w_el = cfg.d * cfg.I * (0.5 + 1.0 / 16)
    return {
        "workload": f"{cfg.name}: MegaMoE routed-expert forward, E={cfg.E} top-{cfg.k} "
                    f"d={cfg.d} I={cfg.I} T={cfg.T}, NVFP4 weights resident",
        "global_batch": cfg.T * world,
        "parallelism": f"replicas x{world}",
        "l2": (f"inputs larger than L2 (~{active * 3 * w_el / 1e9:.2f} GB of expert weights "
               "read per step, L2 is 0.13 GB)") if active * 3 * w_el > 126e6 else
              (f"expert weights (~{active * 3 * w_el / 1e6:.0f} MB) smaller than L2: steps "
               "replay them from L2"),
        "active_experts": active, "valid_slots": int(counts.sum()),
        "max_expert_load": int(counts.max()), "zero_token_experts": int((counts == 0).sum()),
    }


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
#: sub-records measured beside the headline workload (its own weights each)
SUB_CONFIGS = ("prefill", "decode", "decode1")


def fp4_peak_tflops(bf16_tf: float) -> float:
    """Dense NVFP4 tensor peak: the measured bf16 peak x the nominal dense
    FP4 / BF16 ratio (13.5 / 2.25)."""
    return bf16_tf * 13.5 / 2.25


def gemm_roofline(name, bytes_, flops, ms, hbm_gbs, fp4_tf, peak_kind, traffic=None):
    """Roofline object of one grouped-GEMM launch: the binding roof is the
    larger of bytes / HBM and flops / FP4 peak; `achieved` and `frac` are
    against that roof (measured peaks), and the other roof's fraction plus
    both fractions against the datasheet figures (~8 TB/s, 13.5 PFLOP/s)
    are given beside it."""
    t = ms * 1e-3
    gbs = bytes_ / t / 1e9
    tfs = flops / t / 1e12
    t_hbm = bytes_ / (hbm_gbs * 1e9)
    t_fp4 = flops / (fp4_tf * 1e12)
    hbm_bound = t_hbm >= t_fp4
    return {
        "bound": "hbm" if hbm_bound else "tensor",
        "achieved": gbs if hbm_bound else tfs,
        "peak": hbm_gbs if hbm_bound else fp4_tf,
        "unit": "GB/s" if hbm_bound else "TFLOP/s",
        "frac": gbs / hbm_gbs if hbm_bound else tfs / fp4_tf,
        "traffic": traffic,
        "kernel": name,
        "peak_source": (f"{peak_kind} HBM copy" if hbm_bound else
                        f"{peak_kind} bf16 x 6 (nominal dense FP4/BF16 ratio)"),
        "hbm_frac": gbs / hbm_gbs, "fp4_frac": tfs / fp4_tf,
        "attainable_frac": max(t_hbm, t_fp4) / t,
        "datasheet_hbm_frac": gbs / 8000.0, "datasheet_fp4_frac": tfs / 13500.0,
        "algorithmic_bytes": bytes_, "algorithmic_flops": flops,
    }


def measure_forward(cfg, args, dev, world, rank, local, with_e2e=True, with_cpu=True):
    """Every number of one workload: the device-timed forward (inputs
    resident), the two grouped GEMMs timed alone on the forward's own
    intermediates, the roofline of the dominant one, the end-to-end loop
    through the public call with host copies, and the oracle on the host."""
    import numpy as np
    import torch

    from nvfp4_block_scaled_topk_gb300 import inputs, megamoe

    raw = inputs.make_all_experts(cfg, device=dev)
    weights = megamoe.Weights.prepare(raw)
    if not (with_cpu and rank == 0 and not args.no_cpu_baseline):
        del raw
        raw = None
    torch.cuda.empty_cache()
    # the batch is drawn on the host (the reference arm draws the same one)
    x = inputs.make_activations(cfg).to(dev)
    ids, w = (t.to(dev) for t in inputs.make_routing(cfg))
    fwd = megamoe.Forward(weights, cfg.T, cfg.k, pad=cfg.pad)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    # ---- device-timed steps (inputs resident in HBM)
    for _ in range(max(3, args.warmup)):
        fwd(x, ids, w)
    torch.cuda.synchronize()
    bits = fwd.read_status()
    if bits:
        raise RuntimeError(f"device status {bits:#x}")
    v = fwd.intermediates()
    counts = v["counts"].cpu().numpy()
    active = int((counts > 0).sum())
    valid_slots = int(counts.sum())

    # the K timed steps are recorded once into a CUDA graph and replayed by
    # one host call, so a step shorter than its host-side launch work (the
    # 1-token batch) is not bound by the host's launch rate; if the capture
    # fails the same steps run eagerly
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.steps):
                fwd(x, ids, w)
        graph.replay()  # one more untimed pass
        torch.cuda.synchronize()
    except Exception:
        graph = None
        torch.cuda.synchronize()
    device_loop = ("CUDA graph of the K steps, one replay" if graph is not None
                   else "the K steps launched eagerly")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for _ in range(args.steps):
            fwd(x, ids, w)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    del graph

    # ---- the grouped GEMMs timed alone on the forward's own intermediates,
    # CUDA events on the launching stream
    l1_out = torch.empty_like(v["h"])
    l1_amax = torch.empty(1, dtype=torch.float32, device=dev)
    expected = cfg.slots / cfg.E  # the forward's token-tile choice (tile_n 0 = auto)

    def l1():
        megamoe.grouped_gemm(v["xq_codes"], v["xq_sf"], v["gs_x"], weights.w13_codes,
                             weights.w13_scales, weights.w13_gs, v["offsets"],
                             v["padded_offsets"], megamoe.EPI_SILU_MUL, expected_tokens=expected,
                             out=l1_out, out_amax=l1_amax)

    def l2():
        megamoe.grouped_gemm(v["hq_codes"], v["hq_sf"], v["gs_h"], weights.w2_codes,
                             weights.w2_scales, weights.w2_gs.view(-1, 1), v["offsets"],
                             v["padded_offsets"], megamoe.EPI_BFP16, expected_tokens=expected,
                             out=v["y_buf"], out_amax=None)

    def timed(fn, n):
        for _ in range(3):
            fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    # a GEMM whose weights fit in L2 (decode sizes) would read them from L2
    # when replayed back to back: those are timed after a 512 MB write (the
    # median (write, GEMM) window minus the median write)
    w_el0 = cfg.d * cfg.I * (0.5 + 1.0 / 16)
    small = active * 2 * w_el0 < 2 * 126e6
    if small:
        l1_ms = _time_with_flush(l1, max(args.steps, 10), dev, stream)
        l2_ms = _time_with_flush(l2, max(args.steps, 10), dev, stream)
    else:
        l1_ms = timed(l1, max(args.steps, 10))
        l2_ms = timed(l2, max(args.steps, 10))
    clk = clocks.stop()

    # ---- end to end through the public call, host buffers, copies inside.
    # x, topk_ids and topk_weights sit in one pinned staging buffer, so each
    # step's inputs go up in a single host-to-device copy.  Two device copies
    # of the staging buffer and of the output alternate between steps: one
    # stream uploads step i+1's inputs and another downloads step i-1's output
    # while step i computes, as a serving loop would; every step still makes
    # both copies, and the timed region spans all K steps' copies and compute.
    e2e = None
    if with_e2e:
        nx, ni = x.numel() * 2, ids.numel() * 4
        stage_h = torch.empty(nx + 2 * ni, dtype=torch.uint8).pin_memory()
        stage_h[:nx].view(torch.bfloat16).copy_(x.cpu().reshape(-1))
        stage_h[nx:nx + ni].view(torch.int32).copy_(ids.cpu().reshape(-1))
        stage_h[nx + ni:].view(torch.float32).copy_(w.cpu().reshape(-1))
        stage_d = [torch.empty(stage_h.numel(), dtype=torch.uint8, device=dev) for _ in range(2)]
        views = [(sd[:nx].view(torch.bfloat16).view(cfg.T, cfg.d),
                  sd[nx:nx + ni].view(torch.int32).view(cfg.T, cfg.k),
                  sd[nx + ni:].view(torch.float32).view(cfg.T, cfg.k)) for sd in stage_d]
        out_d = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        out_h = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        up_stream = torch.cuda.Stream(device=dev)
        down_stream = torch.cuda.Stream(device=dev)

        def e2e_steps(n):
            # on the current stream (the capture stream while a graph records);
            # the copy streams fork from it and join it at the end
            comp = torch.cuda.current_stream()
            fork = torch.cuda.Event()
            fork.record(comp)
            up_stream.wait_event(fork)
            down_stream.wait_event(fork)
            computed = [None, None]
            downloaded = [None, None]
            for i in range(n):
                b = i % 2
                up = torch.cuda.Event()
                with torch.cuda.stream(up_stream):
                    if computed[b] is not None:  # step i-2 is done with buffer b
                        up_stream.wait_event(computed[b])
                    stage_d[b].copy_(stage_h, non_blocking=True)
                    up.record(up_stream)
                comp.wait_event(up)
                if downloaded[b] is not None:  # step i-2's output has left out_d[b]
                    comp.wait_event(downloaded[b])
                fwd(*views[b], out=out_d[b])
                computed[b] = torch.cuda.Event()
                computed[b].record(comp)
                with torch.cuda.stream(down_stream):
                    down_stream.wait_event(computed[b])
                    out_h[b].copy_(out_d[b], non_blocking=True)
                    downloaded[b] = torch.cuda.Event()
                    downloaded[b].record(down_stream)
            for ev in downloaded:
                if ev is not None:
                    comp.wait_event(ev)

        # the K steps are recorded once into a CUDA graph (one host call
        # replays them, so short steps are not bound by the host's launch
        # rate); if the capture fails the same steps run eagerly
        e2e_steps(3)
        barrier()
        torch.cuda.synchronize()
        graph = None
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                e2e_steps(args.steps)
            graph.replay()
            torch.cuda.synchronize()
        except Exception:
            graph = None
            torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if graph is not None:
            graph.replay()
        else:
            e2e_steps(args.steps)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a.elapsed_time(b) / args.steps
        e2e = {"ms": e2e_ms, "h2d": stage_h.numel(), "d2h": out_h[0].numel() * 2,
               "loop": ("CUDA graph of the K steps" if graph is not None else "eager") +
                       ", inputs uploaded and outputs downloaded on two copy streams, "
                       "double-buffered"}
        del graph, stage_d, out_d

    # ---- max over ranks
    vals = [ms, l1_ms, l2_ms] + ([e2e["ms"]] if e2e else [])
    vals = max_over_ranks(vals, world, dev)
    ms, l1_ms, l2_ms = vals[:3]
    if e2e:
        e2e["ms"] = vals[3]

    hbm_gbs, bf16_tf, peak_kind = _peaks()
    fp4_tf = fp4_peak_tflops(bf16_tf)
    flops = inputs.algorithmic_flops(cfg, valid_slots)
    alg_bytes = inputs.algorithmic_bytes(cfg, active)
    w_el = cfg.d * cfg.I * (0.5 + 1.0 / 16)
    a_row1 = cfg.d * (0.5 + 1 / 16)  # one quantised token row of x
    a_row2 = cfg.I * (0.5 + 1 / 16)  # one requantised row of h
    # per launch: the active experts' weights once, each routed row's
    # activations in and its output row out (L2: BFP16, 2 bytes a value and
    # one exponent byte per 16 rows x 8 columns)
    l1_bytes = active * 2 * w_el + valid_slots * (a_row1 + cfg.I * 2)
    l2_bytes = active * w_el + valid_slots * (a_row2 + cfg.d * (2 + 1 / 128))
    l1_flops = 4 * cfg.d * cfg.I * valid_slots
    l2_flops = 2 * cfg.d * cfg.I * valid_slots
    rl1 = gemm_roofline("k_grouped_gemm (L1 gate+up, SiLU*up epilogue)", l1_bytes, l1_flops,
                        l1_ms, hbm_gbs, fp4_tf, peak_kind,
                        _profile_traffic(f"l1_gemm_{cfg.name}.json"))
    rl2 = gemm_roofline("k_grouped_gemm (L2 down, BFP16 epilogue)", l2_bytes, l2_flops, l2_ms,
                        hbm_gbs, fp4_tf, peak_kind,
                        _profile_traffic(f"l2_gemm_{cfg.name}.json"))
    t_floor = max(alg_bytes / (hbm_gbs * 1e9), flops / (fp4_tf * 1e12))
    tokens_total = cfg.T * world

    cpu = None
    if raw is not None:
        tokens = max(1, min(cfg.T, args.ref_tokens))
        ex = inputs.ExpertSet(cfg, raw)
        # the same sample repeated until about 10 s of CPU work is timed
        total, reps = 0.0, 0
        while reps < 20 and (reps == 0 or total < 10.0):
            total += oracle_sample(cfg, x, ids, w, ex, tokens)
            reps += 1
        cpu = {"value": tokens * reps / total, "unit": UNIT, "cores": _cores(), "kind": "oracle",
               "sample": f"first {tokens} of {cfg.T} tokens of the {cfg.name} batch, full float64 "
                         f"forward over the experts they touch, {reps} times "
                         f"({total:.1f} s); weights fetched before timing"}
    rec = {
        "value": tokens_total / (ms * 1e-3), "ms_per_step": ms,
        "config": workload_config(cfg, counts, world),
        "tflops": flops / (ms * 1e-3) / 1e12,
        "hbm_gbs": alg_bytes / (ms * 1e-3) / 1e9,
        "hbm_frac_of_measured": alg_bytes / (ms * 1e-3) / 1e9 / hbm_gbs,
        "fp4_frac_of_measured": flops / (ms * 1e-3) / 1e12 / fp4_tf,
        "attainable_frac": t_floor / (ms * 1e-3),
        "stage_ms": {"l1_gemm": l1_ms, "l2_gemm": l2_ms},
        "device_loop": device_loop,
        "roofline": rl1 if l1_ms >= l2_ms else rl2,
        "roofline_other_gemm": rl2 if l1_ms >= l2_ms else rl1,
        "cpu_baseline": cpu,
        "e2e": None if e2e is None else {
            "value": tokens_total / (e2e["ms"] * 1e-3), "unit": UNIT,
            "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
            "loop": e2e["loop"]},
        "gpu_launches": kernels_per_step(cfg) * args.steps,
        "clocks": clk,
        "stage_timing": ("each GEMM alone after a 512 MB write (its weights fit in L2): median "
                         "(write, GEMM) window minus median write") if small else
                        "each GEMM alone, back to back (its weights exceed L2)",
    }
    del fwd, weights, raw, x, ids, w, v, l1_out
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import torch

    from nvfp4_block_scaled_topk_gb300 import build, inputs, megamoe

    rank, world, local = _dist()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    megamoe.load()

    cfg = inputs.CONFIGS[args.config]
    main = measure_forward(cfg, args, dev, world, rank, local)
    subs = {}
    if not args.no_sub:
        for name in SUB_CONFIGS:
            if name == cfg.name:
                continue
            r = measure_forward(inputs.CONFIGS[name], args, dev, world, rank, local,
                                with_e2e=True, with_cpu=False)
            subs[name] = {key: r[key] for key in (
                "value", "ms_per_step", "tflops", "hbm_gbs",
                "hbm_frac_of_measured", "fp4_frac_of_measured", "attainable_frac", "stage_ms",
                "stage_timing", "device_loop", "roofline", "roofline_other_gemm", "e2e",
                "clocks")}
            subs[name].update({key: r["config"][key] for key in (
                "workload", "active_experts", "valid_slots", "max_expert_load",
                "zero_token_experts")})
    if rank == 0:
        line = {
            "metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4 (e2m1 x e4m3 scales, fp32 acc)", "data": "synthetic",
            "config": main["config"],
            "tflops": main["tflops"], "hbm_gbs": main["hbm_gbs"],
            "hbm_frac_of_measured": main["hbm_frac_of_measured"],
            "fp4_frac_of_measured": main["fp4_frac_of_measured"],
            "attainable_frac": main["attainable_frac"],
            "stage_ms": main["stage_ms"],
            "stage_timing": main["stage_timing"],
            "device_loop": main["device_loop"],
            "roofline": main["roofline"],
            "roofline_other_gemm": main["roofline_other_gemm"],
            "cpu_baseline": main["cpu_baseline"],
            "e2e": main["e2e"],
            "gpu_launches": main["gpu_launches"],
            "clocks": main["clocks"],
            "sub_records": subs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def _time_with_flush(step, steps, dev, stream):
    """Device time of one `step` whose inputs fit in L2: windows of (write a
    512 MB buffer, then the step) and windows of the write alone, interleaved,
    each between two CUDA events on the launching stream; the median pair
    minus the median write.  The step follows the write back to back as it
    would follow other work (queued while the write runs, so the host's launch
    latency stays hidden), the events' own cost cancels, and the medians keep
    a stray slow window (a power-capped clock) out of the difference."""
    import torch

    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    n = max(steps, 9)
    for _ in range(2):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    pairs = [(ev(), ev()) for _ in range(n)]
    alone = [(ev(), ev()) for _ in range(n)]
    for (a, b), (c, e) in zip(pairs, alone):
        a.record(stream)
        flush.fill_(1)
        step()
        b.record(stream)
        c.record(stream)
        flush.fill_(1)
        e.record(stream)
    torch.cuda.synchronize()
    med = lambda xs: sorted(xs)[len(xs) // 2]
    t_pair = med([a.elapsed_time(b) for a, b in pairs])
    t_write = med([c.elapsed_time(e) for c, e in alone])
    return max(t_pair - t_write, 1e-6)


def run_linear(args):
    """The dense NVFP4 linear (measured-amax activation scale) on one GPU:
    tokens/s through megamoe_linear_nvfp4 with inputs resident, against the
    roofline max(bytes / HBM, flops / FP4 tensor peak)."""
    import torch

    from nvfp4_block_scaled_topk_gb300 import inputs, megamoe

    megamoe.load()
    cfg = inputs.LINEAR_CONFIGS[args.config]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    x, c, s, gs = inputs.make_linear(cfg, device=dev)
    w = megamoe.LinearWeights.prepare(c, s, gs)
    out = torch.empty(cfg.T, cfg.N, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(256, megamoe.linear_workspace_size(cfg.T, cfg.K, cfg.N)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        megamoe.linear_nvfp4(x, w, out=out, ws=ws)
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    # weights and x are smaller than L2 for the decode shape: each step timed
    # after a 512 MB write, the write's median time subtracted (_time_with_flush)
    ms = _time_with_flush(lambda: megamoe.linear_nvfp4(x, w, out=out, ws=ws), args.steps, dev,
                          stream)
    clk = clocks.stop()
    hbm_gbs, bf16_tf, peak_kind = _peaks()
    fp4_tf = bf16_tf * 13.5 / 2.25  # measured bf16 x the nominal dense FP4 / BF16 ratio
    w_bytes = cfg.N * cfg.K * (0.5 + 1.0 / 16)
    alg_bytes = w_bytes + cfg.T * cfg.K * 2 + cfg.T * cfg.N * 2
    flops = 2.0 * cfg.T * cfg.N * cfg.K
    t_hbm, t_fp4 = alg_bytes / (hbm_gbs * 1e9), flops / (fp4_tf * 1e12)
    bound = "hbm" if t_hbm >= t_fp4 else "tensor"
    achieved = (alg_bytes / (ms * 1e-3) / 1e9) if bound == "hbm" else flops / (ms * 1e-3) / 1e12
    peak = hbm_gbs if bound == "hbm" else fp4_tf
    line = {
        "op": "linear", "metric": "tokens/s and NVFP4 TFLOP/s, dense NVFP4 linear "
                                  "(measured-amax activation scale)",
        "value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "dtype": "nvfp4 (e2m1 x e4m3 scales, fp32 acc), bf16 out", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: x [{cfg.T}, {cfg.K}] bf16 @ W [{cfg.N}, {cfg.K}] "
                               "NVFP4", "l2": "512 MB written before every step; median "
                                              "(write, step) minus median write"},
        "tflops": flops / (ms * 1e-3) / 1e12,
        "hbm_gbs": alg_bytes / (ms * 1e-3) / 1e9,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak,
                     "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": achieved / peak,
                     "traffic": None, "kernel": "whole call (prologue, quantiser, GEMM)",
                     "peak_source": peak_kind if bound == "hbm" else
                     f"{peak_kind} bf16 x 6 (nominal FP4/BF16 ratio)"},
        "gpu_launches": linear_kernels_per_call(
            cfg.T, cfg.K, megamoe.linear_workspace_size(cfg.T, cfg.K, cfg.N)) * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


# --op gemm_sweep: the grouped GEMM alone, the same tiles at several K
SWEEP_CFGS = {
    "l2_bfp16_128": ("weights-on-M, 128-token tiles, BFP16 out (the L2 GEMM's tile)", "EPI_BFP16", 128),
    "l1_tm_silu": ("token-major 128 tokens x 256 weight rows, SiLU*up (the L1 GEMM's tile at "
                   "prefill sizes)", "EPI_SILU_MUL", 256),
    "f32_128": ("weights-on-M, 128-token tiles, fp32 out", "EPI_F32", 128),
    "bf16_128": ("weights-on-M, 128-token tiles, bf16 out (staged stores)", "EPI_BF16", 128),
    "bfp16_64": ("weights-on-M, 64-token tiles, BFP16 out", "EPI_BFP16", 64),
    "silu_64": ("weights-on-M, 64-token tiles, SiLU*up", "EPI_SILU_MUL", 64),
}


def sweep_tiles(silu: bool, bfp16: bool, tile_n: int, E: int, rows_per_expert: int, N: int) -> int:
    """Tiles of one grouped-GEMM launch with E experts of rows_per_expert rows
    each (a multiple of the token tile) and N weight rows per expert.
    Token-major tiles (tile_n 256; BFP16 runs those as 128-token tiles) are
    128 tokens x 256 weight rows; weights-on-M tiles are tile_n tokens x 128
    output features (for SiLU*up the gate and up rows of 128 features)."""
    if tile_n == 256 and bfp16:
        tile_n = 128
    if tile_n == 256:
        return E * (rows_per_expert // 128) * (N // 256)
    return E * (rows_per_expert // tile_n) * (N // 256 if silu else N // 128)


def run_gemm_sweep(args):
    """The grouped GEMM alone on synthetic NVFP4 operands: 128 experts of 256
    token rows, N = 4096 weight rows per expert, uniform random E2M1 code bytes
    and E4M3 block scales 0x30-0x47, weights above L2 at every K.  The same
    tiles are timed at each K (CUDA events, median over --steps launches);
    the time per wave of tiles fits a + b * (K / 256): a is what a tile costs
    beyond its K steps, b what one K step costs."""
    import math

    import numpy as np
    import torch

    from nvfp4_block_scaled_topk_gb300 import megamoe

    megamoe.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    E, rpe, N = 128, 256, 4096
    ks = [int(v) for v in args.sweep_k.split(",")]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    gen = torch.Generator(device=dev).manual_seed(2024)
    rows = E * rpe
    offs = torch.arange(0, E + 1, dtype=torch.int32, device=dev) * rpe
    one = torch.ones(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(0)
    clocks.start()
    result = {}
    for name in args.sweep_cfg.split(","):
        desc, epi_name, tile_n = SWEEP_CFGS[name]
        epi = getattr(megamoe, epi_name)
        silu, bfp16 = epi == megamoe.EPI_SILU_MUL, epi == megamoe.EPI_BFP16
        pts = []
        for K in ks:
            def codes(n):
                return torch.randint(0, 256, (n, K // 2), dtype=torch.uint8, device=dev, generator=gen)

            def scales(n):
                return torch.randint(0x30, 0x48, (n, K // 16), dtype=torch.uint8, device=dev,
                                     generator=gen)

            ac, asf = codes(rows), scales(rows)
            wc = megamoe.pack_weight_codes(codes(E * N), N // 2 if silu else 0).view(E, N, K // 2)
            wsc = megamoe.swizzle_scales(scales(E * N))
            wgs = torch.ones(E, 2 if silu else 1, device=dev)
            amax = torch.empty(1, dtype=torch.float32, device=dev) if silu else None
            if bfp16:
                out = torch.empty(megamoe.bfp16_bytes(rows, N), dtype=torch.uint8, device=dev)
            else:
                dt = torch.float32 if epi == megamoe.EPI_F32 else torch.bfloat16
                out = torch.empty(rows, N // 2 if silu else N, dtype=dt, device=dev)

            def step():
                megamoe.grouped_gemm(ac, asf, one, wc, wsc, wgs, offs, offs, epi, tile_n=tile_n,
                                     out=out, out_amax=amax)

            for _ in range(max(3, args.warmup)):
                step()
            torch.cuda.synchronize()
            times = []
            for _ in range(args.steps):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                step()
                b.record(stream)
                torch.cuda.synchronize()
                times.append(a.elapsed_time(b))
            ms = float(np.median(times))
            waves = math.ceil(sweep_tiles(silu, bfp16, tile_n, E, rpe, N) / sms)
            pts.append([K // 256, ms, ms * 1e3 / waves])
            del ac, asf, wc, wsc, out
            torch.cuda.empty_cache()
        rec = {"tile": desc, "tiles": sweep_tiles(silu, bfp16, tile_n, E, rpe, N),
               "points": [{"k_steps": kt, "ms": ms, "us_per_wave": us} for kt, ms, us in pts]}
        if len(pts) >= 2:
            slope, icept = np.polyfit([p[0] for p in pts], [p[2] for p in pts], 1)
            rec.update(per_tile_us=float(icept), per_k_step_us=float(slope))
        result[name] = rec
    line = {"op": "gemm_sweep", "metric": "grouped GEMM time per wave of tiles against K",
            "unit": "us", "data": "synthetic", "steps": args.steps, "warmup": args.warmup,
            "config": {"workload": f"{E} experts x {rpe} token rows, N = {N}, K in {ks}",
                       "fit": "us per wave = per_tile_us + per_k_step_us * K / 256"},
            "configs": result, "clocks": clocks.stop()}
    print(json.dumps(line), flush=True)


def run_layer(args, router_only=False):
    """The MoE layer from router logits on one GPU: megamoe_router_topk (k
    routed experts + the shared expert as expert E) then megamoe_forward over
    E + 1 experts (router_only: the router alone)."""
    import torch

    from nvfp4_block_scaled_topk_gb300 import inputs, megamoe

    megamoe.load()
    base = inputs.CONFIGS[args.config]
    cfg = inputs.with_shared_expert(base)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    logits, bias = inputs.make_router_logits(base, device=dev)
    stream = torch.cuda.current_stream()
    if router_only:
        fwd = None

        def step():
            megamoe.router_topk(logits, base.k, bias, shared_expert=base.E)
    else:
        raw = inputs.make_all_experts(cfg, device=dev)
        weights = megamoe.Weights.prepare(raw)
        del raw
        torch.cuda.empty_cache()
        x = inputs.make_activations(base, device=dev)
        fwd = megamoe.Forward(weights, base.T, cfg.k, pad=base.pad)

        def step():  # router fused ahead of the routing (megamoe_forward_from_logits)
            fwd.from_logits(x, logits, base.k, bias, shared_expert=base.E)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    if router_only:
        # the router's inputs are small: a 512 MB write before every step,
        # the write's median time subtracted
        ms = _time_with_flush(step, args.steps, dev, stream)
    else:
        # the layer reads more expert weights per step than L2 holds: steps
        # back to back between two events
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
    clk = clocks.stop()
    hbm_gbs, _, peak_kind = _peaks()
    k_out = base.k + 1
    if router_only:
        alg_bytes = base.T * base.E * 4 + base.E * 4 + base.T * k_out * 8
        kernel, launches = "k_router", 1
    else:
        ids, _ = megamoe.router_topk(logits, base.k, bias, shared_expert=base.E)
        active = int(torch.unique(ids[:, :base.k]).numel()) + 1
        alg_bytes = (inputs.algorithmic_bytes(cfg, active) + base.T * base.E * 4)
        kernel = "whole step (megamoe_forward_from_logits)"
        launches = kernels_per_step(cfg) + (0 if cfg.T * cfg.d <= 262144 else 1)
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    line = {
        "op": "router" if router_only else "layer",
        "metric": ("tokens/s, router top-k + softmax" if router_only else
                   "tokens/s, MoE layer from router logits (routed top-k + shared expert)"),
        "value": base.T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "dtype": "fp32 router; nvfp4 experts", "data": "synthetic",
        "config": {"workload": f"{base.name}: logits [{base.T}, {base.E}] fp32, top-{base.k} "
                               "+ 1 shared expert" + ("" if router_only else
                                                      f", d={base.d} I={base.I}"),
                   "l2": ("512 MB written before every step; median (write, step) minus "
                          "median write") if router_only else
                         "expert weights read per step larger than L2"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": achieved / hbm_gbs, "traffic": None, "kernel": kernel,
                     "peak_source": peak_kind},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="large",
                    help="headline workload (default: large, the largest single-GPU one)")
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the prefill / decode / decode1 sub-records")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="forward",
                    choices=["forward", "linear", "router", "layer", "gemm_sweep"],
                    help="forward: the routed-expert forward (default); linear: the dense "
                         "NVFP4 linear (--config one of the linear_* workloads); router: the "
                         "router top-k alone; layer: router + forward with a shared expert; "
                         "gemm_sweep: the grouped GEMM alone at several K (--sweep-k, "
                         "--sweep-cfg)")
    ap.add_argument("--sweep-k", default="1024,2048,3584,7168")
    ap.add_argument("--sweep-cfg", default="l2_bfp16_128,l1_tm_silu",
                    help="comma-separated: " + ", ".join(SWEEP_CFGS))
    args = ap.parse_args()
    if args.op == "gemm_sweep":
        run_gemm_sweep(args)
    elif args.op == "linear":
        if args.config == "large":
            args.config = "linear_qa_decode"
        run_linear(args)
    elif args.op in ("router", "layer"):
        if args.config == "large" and args.op == "router":
            args.config = "decode"
        run_layer(args, router_only=args.op == "router")
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
