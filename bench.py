"""Benchmark of the MoE expert-FFN forward (align -> gate/up GEMM + SiLU*up ->
down GEMM x routing weight -> combine) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME]

One step is one pass of the whole path over one synthetic batch.  The default
workload is the Mixtral-8x7B-shaped prefill layer (T=4096, H=4096, I=14336,
E=8, top-2, bf16).  Under torchrun each rank runs its own replica on its own
GPU with its own batch (weak scaling; no data-path collective).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(the plain fp64 definition) on the host cores instead, on a bounded sample of
tokens of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import dataclasses
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_grouped_02_gb300 import inputs as gen  # noqa: E402

METRIC = "MoE layer tokens/sec and TFLOP/s (prefill); HBM GB/s (decode) vs GB300 peak"
# per-launch DRAM bytes of the dominant kernels from ncu captures, with the
# hash of the kernel sources they were taken on
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "mixture_experts_grouped_02_gb300", "csrc")
# each GEMM's own sources (the shared headers also serve the other kernels,
# whose edits do not change this one)
KERNEL_SOURCES = {"wpair": ("gemm_wpair.cu", "sched.cuh"), "mx": ("gemm_mx.cu", "sched.cuh")}
# nominal dense GB300 figures (context beside the measured ones): HBM3e
# 8 TB/s, bf16 tensor 2.25 PFLOP/s, fp8 4.5 PFLOP/s
NOMINAL = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0, "fp8_tflops": 4500.0}
# the workloads timed besides the default one, each graded on its own bound
# (ordered so that workloads sharing a weight shape run one after another;
# ":fused" runs the workload with the combine fused into the down GEMM)
WORKLOADS = ([f"mixtral_decode_T{t}" for t in gen.DECODE_T] +
             ["dsv3_prefill", "dsv3_prefill:fused"] +
             [f"dsv3_decode_T{t}" for t in gen.DECODE_T] + ["lowp", "lowp_oai"])


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="mixtral_prefill")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--fused-combine", action="store_true",
                    help="combine fused into GEMM2 (fp32 atomics into a (T, H) accumulator)")
    ap.add_argument("--block-m", type=int, default=0,
                    help="align block (token tile) of the GEMMs; 0 picks it from the problem")
    ap.add_argument("--shrink", type=int, default=1,
                    help="divide the workload's tokens and experts by this factor (same tokens "
                         "per expert; for profiling captures that must stay small)")
    ap.add_argument("--sweep", action="store_true",
                    help="the 48-point batch sweep of one expert shard of the GPT-OSS-shaped "
                         "layer (lowp_oai), one JSON line with a 'sweep' list")
    ap.add_argument("--ep-shards", type=int, default=8,
                    help="expert shards of the layer in the sweep (one is timed)")
    ap.add_argument("--ep-rank", type=int, default=0, help="the shard the sweep times")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip timing the other workloads (the 'workloads' list)")
    ap.add_argument("--workload-steps", type=int, default=10,
                    help="timed steps per workload of the 'workloads' list (3 warm-up steps)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def max_over_ranks(v: float, ws: int, device) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_batch_seed(rank: int) -> int:
    """Every rank serves the same model (weights drawn with seed 0) and routes
    its own batch: rank 0 draws x and routing with seed 0, rank r > 0 with
    1000 + r, so that replicas do not repeat one another's work."""
    return 0 if rank == 0 else 1000 + rank


def aggregate(ms_per_step_local: float, tokens_per_rank: int, ws: int, device):
    """Whole-job throughput of ws replicas: the step time is the slowest
    rank's, the tokens are all ranks' (weak scaling)."""
    ms = max_over_ranks(ms_per_step_local, ws, device)
    return ms, tokens_per_rank * ws / (ms * 1e-3)


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        burst = d.get("bf16_tflops", 1900.0)
        return (d.get("hbm_gbs", 6800.0), burst, d.get("bf16_tflops_sustained", burst),
                "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_hash(family: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str, mx: bool):
    """Per-launch DRAM bytes (read + write) of `kernel` on `workload` from the
    committed ncu figures, or None when there are none or the kernel's
    sources changed since they were taken."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        table = json.load(f)
    rec = table.get(workload, {}).get(kernel)
    if not rec or rec.get("kernel_source_sha256") != kernel_source_hash("mx" if mx else "wpair"):
        return None
    return int(rec["traffic_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = list(csv.reader(io.StringIO(out)))
        samples = []
        for r in rows:
            if len(r) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                samples.append(dict(ts=ts, sm=float(r[2]), smax=float(r[3]),
                                    hw=r[6].strip(), hwt=r[7].strip(), swt=r[8].strip(),
                                    pcap=r[9].strip()))
            except (ValueError, IndexError):
                continue
        if not samples:
            return None
        inside = [s for s in samples if t0 - 1.0 <= s["ts"] <= t1 + 1.0] or samples
        reasons = set()
        for s in inside:
            if s["hw"] == "Active":
                reasons.add("hw_slowdown")
            if s["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if s["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if s["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(s["sm"] for s in inside),
                "sm_max_mhz": max(s["smax"] for s in inside), "reasons": sorted(reasons),
                "samples": len(inside)}


def bytes_algorithmic(cfg, inp):
    """Weights of experts with at least one token + x once + out once + ids
    and weights."""
    active = int((torch.bincount(inp.topk_ids.flatten().long(), minlength=cfg.E) > 0).sum())
    esz = inp.x.element_size()
    w_per_expert = (inp.w13[0].numel() * inp.w13.element_size() +
                    inp.w2[0].numel() * inp.w2.element_size())
    if inp.w13_scale is not None:
        w_per_expert += inp.w13_scale[0].numel() + inp.w2_scale[0].numel()
    return active * w_per_expert + 2 * cfg.T * cfg.H * esz + 8 * cfg.T * cfg.K, active


def kernel_rooflines(cfg, inp, active, gemm1_ms, gemm2_ms, hbm_gbs, bf16_tflops):
    """Algorithmic FLOPs and bytes of the two GEMM launches and both roofline
    fractions.  Bytes: weights of the active experts, the activation rows read
    once, the intermediate written once (h for gate/up, y for down)."""
    na, H, I = cfg.T * cfg.K, cfg.H, cfg.I
    mx = cfg.dtype == "mxfp4"
    esz = 1 if mx else inp.x.element_size()  # the GEMMs read e4m3 x and h on the mx path
    w13_e = inp.w13[0].numel() * inp.w13.element_size()
    w2_e = inp.w2[0].numel() * inp.w2.element_size()
    if mx:  # the e8m0 scales travel with the e2m1 values
        w13_e += inp.w13_scale[0].numel()
        w2_e += inp.w2_scale[0].numel()
    out = {}
    for name, ms, flops, nbytes in (
            ("gemm_gate_up", gemm1_ms, 4 * na * H * I,
             active * w13_e + cfg.T * H * esz + na * I * esz),
            ("gemm_down", gemm2_ms, 2 * na * H * I,
             active * w2_e + na * I * esz + na * H * 4)):
        tf = flops / (ms * 1e-3) / 1e12
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "flops": flops, "bytes": nbytes, "tflops": tf, "gbs": gbs,
                     "tensor_frac": tf / bf16_tflops, "hbm_frac": gbs / hbm_gbs}
    return out


def cpu_oracle_rate(cfg, inp_cpu, seconds):
    """Time the oracle (as it stands) on a bounded sample of tokens; returns
    (tokens/s, sample description, threads)."""
    import oracle
    threads = len(os.sched_getaffinity(0))
    oracle.lib()
    mx = cfg.dtype == "mxfp4"
    act = {}
    if cfg.activation == "swiglu_oai":
        act = dict(activation=oracle.ACT_SWIGLU_CLAMP, swiglu_alpha=inp_cpu.swiglu_alpha,
                   swiglu_limit=inp_cpu.swiglu_limit, gate_up_interleaved=True,
                   w13_bias=inp_cpu.w13_bias.numpy(), w2_bias=inp_cpu.w2_bias.numpy())
    P = oracle.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, gen.to_numpy_storage(inp_cpu.x[:1]),
                            gen.to_numpy_storage(inp_cpu.w13[:1]), quantize_x=mx, h_e4m3=mx,
                            h_scale=inp_cpu.h_scale, **act)
    args = (gen.to_numpy_storage(inp_cpu.x), inp_cpu.topk_ids.numpy(),
            inp_cpu.topk_weights.numpy(), gen.to_numpy_storage(inp_cpu.w13),
            gen.to_numpy_storage(inp_cpu.w2))
    scales = dict(w13_scale=gen.to_numpy_storage(inp_cpu.w13_scale),
                  w2_scale=gen.to_numpy_storage(inp_cpu.w2_scale))
    probe = np.arange(min(cfg.T, threads), dtype=np.int32)
    t = time.perf_counter()
    oracle.forward(P, *args, tokens=probe, **scales)
    dt = time.perf_counter() - t
    n = int(min(cfg.T, max(len(probe), len(probe) * seconds / max(dt, 1e-3))))
    n = max(threads, n // threads * threads) if n >= threads else n
    toks = np.arange(n, dtype=np.int32)
    t = time.perf_counter()
    oracle.forward(P, *args, tokens=toks, **scales)
    dt = time.perf_counter() - t
    return n / dt, f"first {n} of {cfg.T} tokens ({n * cfg.K} assignments), fp64, {dt:.1f} s", \
        threads


def run_reference(args, ws, rank):
    if rank != 0:
        return
    cfg = gen.config(args.config)
    inp = gen.generate(cfg, seed=0, device="cpu")
    per_step = args.cpu_seconds / max(1, args.steps + args.warmup)
    rates = []
    sample = ""
    threads = 1
    for i in range(args.warmup + args.steps):
        r, sample, threads = cpu_oracle_rate(cfg, inp, max(1.0, per_step))
        if i >= args.warmup:
            rates.append(r)
    value = statistics.median(rates)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * cfg.T / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E,
                       "top_k": cfg.K, "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def build_stages(moe, _abi, cfg, inp, dev, block_m=0, shard=None, fused=False):
    """Problem, workspace, packed weights and the exact launches moe_forward
    makes, one C-ABI call per stage.  shard = (expert_base, local_experts):
    inp's weights hold those experts only.  fused: the combine fused into
    GEMM2 (an fp32 accumulator the gather step zeroes, then one rounding
    pass)."""
    mx = cfg.dtype == "mxfp4"
    act = {}
    if cfg.activation == "swiglu_oai":  # GPT-OSS expert FFN
        act = dict(activation=moe.MOE_ACT_SWIGLU_CLAMP, swiglu_alpha=inp.swiglu_alpha,
                   swiglu_limit=inp.swiglu_limit, gate_up_interleaved=True,
                   w13_bias=inp.w13_bias, w2_bias=inp.w2_bias)
    base, L = shard if shard is not None else (0, 0)
    p = moe.make_problem(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, "bf16" if mx else cfg.dtype,
                         "mxfp4" if mx else None, block_m=block_m, h_scale=inp.h_scale,
                         expert_base=base, local_experts=L, fused_combine=fused, **act)
    wsp = moe.Workspace(p, dev)
    part = lambda i, dt=torch.int32: wsp.part(i, dt)
    st = wsp.status
    counts, offs, poffs = part(_abi.MOE_WS_COUNTS), part(_abi.MOE_WS_OFFSETS), \
        part(_abi.MOE_WS_PADDED_OFFSETS)
    sorted_ids, inv = part(_abi.MOE_WS_SORTED_IDS), part(_abi.MOE_WS_INV_PERM)
    binfo, nblk = part(_abi.MOE_WS_BLOCK_INFO), part(_abi.MOE_WS_NUM_BLOCKS)
    scratch = part(_abi.MOE_WS_ALIGN)  # empty below 16384 assignments: one-CTA align
    h = part(_abi.MOE_WS_H, torch.uint8)
    y = part(_abi.MOE_WS_Y, torch.float32)  # or, fused, the (T, H) accumulator
    acc = y if fused else None
    xq = part(_abi.MOE_WS_XQ, torch.uint8) if mx else None
    xs = part(_abi.MOE_WS_X_SCALE, torch.float32) if mx else None
    # model weights as the kernels read them (mxfp4: packed once, at load time)
    w13, s13, w2, s2 = inp.w13, None, inp.w2, None
    if mx:
        w13, s13 = moe.pack_mx(inp.w13, inp.w13_scale, 2, interleaved=inp.interleaved)
        w2, s2 = moe.pack_mx(inp.w2, inp.w2_scale, 1)
    splits = moe.moe_gemm2_default_splits(p)
    bm = moe.moe_resolve_block_m(p)  # the align block the GEMMs of this problem tile by
    cap = moe.moe_align_capacity(cfg.T, cfg.K, L if L else cfg.E, bm)
    out = torch.empty((cfg.T, cfg.H), dtype=inp.x.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    st.zero_()

    # exactly the launches moe_forward makes, one C-ABI call per stage
    stages = []
    stages.append(("align", lambda: moe.moe_align_local(
        inp.topk_ids, cfg.T, cfg.K, cfg.E, base, L if L else cfg.E, bm, counts, offs, poffs,
        sorted_ids, inv, binfo, nblk, st, stream, scratch)))
    if mx:
        stages.append(("quantize_gather_x", lambda: moe.moe_quantize_gather_x_fp8(
            inp.x, _abi.MOE_BF16, cfg.T, cfg.H, cfg.K, inv, xq, xs, st, stream, acc)))
    else:  # token rows to their sorted slots
        x_sorted = part(_abi.MOE_WS_XQ, inp.x.dtype)
        stages.append(("gather", lambda: moe.moe_gather_rows(
            inp.x, p.act, cfg.T, cfg.H, cfg.K, inv, x_sorted, st, stream, acc)))
    a_rows = xq if mx else x_sorted
    stages.append(("gemm_gate_up", lambda: moe.moe_gemm1_silu(
        p, a_rows, xs, w13, s13, sorted_ids, binfo, nblk, h, st, stream)))
    stages.append(("gemm_down", lambda: moe.moe_gemm2_weighted(
        p, h, w2, s2, inp.topk_weights, sorted_ids, binfo, nblk, y, splits, st, stream)))
    if fused:
        stages.append(("combine", lambda: moe.moe_combine_finish(
            y, cfg.T, cfg.H, p.act, out, st, stream)))
    else:
        stages.append(("combine", lambda: moe.moe_combine(
            y, splits, cap, inv, cfg.T, cfg.K, cfg.H, p.act, out, st, stream)))
    return stages, p, wsp, (w13, s13, w2, s2), out, bm, stream


def time_stage_loop(stages, stream, dev, warmup, steps):
    """Run `warmup` untimed steps, then `steps` timed ones with an event
    before the first stage and after every stage of every step; returns
    (mean ms per step, {stage: mean ms})."""
    for _ in range(warmup):
        for _, f in stages:
            f()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
          for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for i in range(steps):
        ev[i][0].record(stream)
        for j, (_, f) in enumerate(stages):
            f()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    total = statistics.mean(ev[i][0].elapsed_time(ev[i][-1]) for i in range(steps))
    stage_ms = {n: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps))
                for j, (n, _) in enumerate(stages)}
    return total, stage_ms


def graded_roofline(cfg, kern, ms_step, bytes_alg, hbm_gbs, bf16_tflops):
    """The workload's grade: prefill on the tensor cores (bf16 dense), decode
    and the low-precision layer on HBM bandwidth, taken for the dominant GEMM
    and for the whole step (roofline time max(FLOPs / tensor peak, bytes /
    HBM peak) over the step time), against the measured and nominal peaks."""
    dom = max(kern, key=lambda k: kern[k]["ms"])
    d = kern[dom]
    tensor = "prefill" in cfg.name
    out = {"kernel": dom, "kernel_ms": d["ms"], "bound": "tensor" if tensor else "hbm"}
    if tensor:
        out.update(achieved=d["tflops"], unit="TFLOP/s", peak=bf16_tflops,
                   frac=d["tflops"] / bf16_tflops, peak_nominal=NOMINAL["bf16_tflops"],
                   frac_nominal=d["tflops"] / NOMINAL["bf16_tflops"],
                   other_bound_frac={"hbm": d["gbs"] / hbm_gbs})
    else:
        out.update(achieved=d["gbs"], unit="GB/s", peak=hbm_gbs, frac=d["gbs"] / hbm_gbs,
                   peak_nominal=NOMINAL["hbm_gbs"], frac_nominal=d["gbs"] / NOMINAL["hbm_gbs"],
                   other_bound_frac={"tensor": d["tflops"] / bf16_tflops})
    mx = cfg.dtype == "mxfp4"
    # the block-scaled MMAs run at the fp8 rate: twice the bf16 one
    tc = bf16_tflops * (2 if mx else 1)
    t_roof = max(cfg.flops / (tc * 1e12), bytes_alg / (hbm_gbs * 1e9)) * 1e3
    out["step_roofline_ms"] = t_roof
    out["step_frac"] = t_roof / ms_step
    return out


def run_workloads(moe, _abi, args, dev, main_cfg, main_inp):
    """Time every other workload at full size (device-drawn inputs, weights
    drawn once per weight shape and shared by the workloads of that shape),
    `args.workload_steps` steps each after 3 warm-up steps, with events
    around every stage.  Returns one record per workload."""
    hbm_gbs, bf16_burst, _, _ = peaks()
    sampler = ClockSampler(dev.index)
    sampler.start()
    t0 = time.time()
    records = []
    weights = {}
    for entry in WORKLOADS:
        name, _, mode = entry.partition(":")
        fused = mode == "fused"
        cfg = gen.config(name)
        key = (cfg.H, cfg.I, cfg.E, cfg.dtype)
        if key == (main_cfg.H, main_cfg.I, main_cfg.E, main_cfg.dtype):
            weights[key] = (main_inp.w13, main_inp.w2, main_inp.w13_scale, main_inp.w2_scale)
        if key not in weights:
            weights.clear()  # one weight shape resident at a time
            torch.cuda.empty_cache()
            weights[key] = gen.draw_weights(cfg, seed=0, device=dev)
        w13, w2, s13, s2 = weights[key]
        ids, w = gen.route(gen.router_logits(cfg, 0, dev), cfg.K)
        inp = gen.MoEInputs(cfg, gen.draw_x(cfg, 0, dev), w13, w2, ids, w, s13, s2)
        if cfg.activation == "swiglu_oai":
            gen.draw_swiglu_oai(inp, seed=0, device=dev)
        stages, p, wsp, _, _, bm, stream = build_stages(moe, _abi, cfg, inp, dev, 0, fused=fused)
        ms_step, stage_ms = time_stage_loop(stages, stream, dev, 3, args.workload_steps)
        status = moe.moe_get_device_status(wsp.status, stream)
        if status != 0:
            raise RuntimeError(f"{name}: device status {status}")
        bytes_alg, active = bytes_algorithmic(cfg, inp)
        kern = kernel_rooflines(cfg, inp, active, stage_ms["gemm_gate_up"],
                                stage_ms["gemm_down"], hbm_gbs, bf16_burst)
        roof = graded_roofline(cfg, kern, ms_step, bytes_alg, hbm_gbs, bf16_burst)
        roof["traffic"] = profiled_traffic(name, roof["kernel"], cfg.dtype == "mxfp4")
        records.append({
            "workload": entry, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "top_k": cfg.K,
            "combine": "fused into GEMM2 (fp32 atomics)" if fused else "separate, deterministic",
            "dtype": cfg.dtype, "block_m": bm, "k_splits": moe.moe_gemm2_default_splits(p),
            "steps": args.workload_steps, "ms_per_step": ms_step,
            "tokens_per_s": cfg.T / (ms_step * 1e-3),
            "tflops": cfg.flops / (ms_step * 1e-3) / 1e12,
            "hbm_gbs_algorithmic": bytes_alg / (ms_step * 1e-3) / 1e9,
            "algorithmic_bytes": bytes_alg, "flops": cfg.flops, "active_experts": active,
            "stage_ms": stage_ms, "kernels": kern, "roofline": roof})
        del stages, p, wsp, inp
    weights.clear()
    torch.cuda.empty_cache()
    clocks = sampler.stop(t0, time.time())
    return records, clocks


def cuda_graph_ms(moe, p, buf, weights, wsp, dev, reps):
    """Capture moe_forward on its own stream into a CUDA graph (after one
    eager call on that stream) and time `reps` back-to-back replays."""
    w13, s13, w2, s2 = weights
    s = torch.cuda.Stream(dev)

    def fwd():
        moe.moe_forward(p, buf["x"], buf["ids"], buf["w"], w13, s13, w2, s2, buf["out"],
                        wsp.buffer, wsp.nbytes, s)

    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        fwd()
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
        fwd()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps


def run_ours(args, ws, rank, local):
    import mixture_experts_grouped_02_gb300 as moe
    from mixture_experts_grouped_02_gb300 import _abi

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe._abi.lib()
    cfg = gen.config(args.config)
    if args.shrink > 1:
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}/{args.shrink}",
                                  T=max(1, cfg.T // args.shrink), E=max(1, cfg.E // args.shrink))
    # weights are the same model on every rank; each rank routes its own batch
    inp = gen.generate(cfg, seed=0, device=dev)
    if rank > 0:
        seed = rank_batch_seed(rank)
        inp.x = gen.draw_x(cfg, seed=seed, device=dev)
        inp.topk_ids, inp.topk_weights = gen.route(gen.router_logits(cfg, seed, dev), cfg.K)
    stages, p, wsp, (w13, s13, w2, s2), out, bm, stream = build_stages(
        moe, _abi, cfg, inp, dev, args.block_m, fused=args.fused_combine)
    st = wsp.status
    mx = cfg.dtype == "mxfp4"
    splits = moe.moe_gemm2_default_splits(p)
    names = [n for n, _ in stages]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        for i, (_, f) in enumerate(stages):
            f()
            if ev is not None:
                ev[i + 1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    status = moe.moe_get_device_status(st, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    # the timed region: K steps back to back, one event pair around them.
    # Every 4th step also records an event between stages for the per-kernel
    # breakdown; the others run without (an event between two kernels keeps
    # the next one from launching while the previous one drains).
    t_beg, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    probe = [i for i in range(args.steps) if i % 4 == 3] or [args.steps - 1]
    evs = {i: [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
           for i in probe}
    barrier(ws)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    t_beg.record(stream)
    for i in range(args.steps):
        step(evs.get(i))
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier(ws)
    total_ms = float(t_beg.elapsed_time(t_end))
    clocks = sampler.stop(t0, t1)
    status = moe.moe_get_device_status(st, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")

    stage = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(len(stages))]
                      for i in probe])  # ms
    stage_ms = {n: float(stage[:, j].mean()) for j, n in enumerate(names)}
    ms_step, value = aggregate(total_ms / args.steps, cfg.T, ws, dev)
    tokens_all = cfg.T * ws
    flops = cfg.flops
    tflops = flops * ws / (ms_step * 1e-3) / 1e12
    bytes_alg, active = bytes_algorithmic(cfg, inp)
    gemm1_ms = stage_ms["gemm_gate_up"]
    gemm2_ms = stage_ms["gemm_down"]
    hbm_gbs, bf16_burst, bf16_sustained, peak_kind = peaks()
    # the burst GEMM figure for a run that stayed below the power cap, the
    # sustained one (a seconds-long loop under the cap) once the cap was hit
    capped = "sw_power_cap" in clocks.get("reasons", [])
    bf16_tflops = bf16_sustained if capped else bf16_burst
    kern = kernel_rooflines(cfg, inp, active, gemm1_ms, gemm2_ms, hbm_gbs, bf16_tflops)
    dom = max(kern, key=lambda k: kern[k]["ms"])
    d = kern[dom]
    # the bound of the dominant kernel: its algorithmic intensity against the ridge
    tensor_bound = d["flops"] / d["bytes"] > bf16_tflops * 1e12 / (hbm_gbs * 1e9)
    traffic = profiled_traffic(cfg.name, dom, mx)
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": d["tflops"], "peak": bf16_tflops,
                "unit": "TFLOP/s", "frac": d["tflops"] / bf16_tflops,
                "peak_source": f"{peak_kind} bf16 dense "
                               + ("(sustained: sw_power_cap seen in the timed region)" if capped
                                  else "(burst)"),
                "frac_of_burst": d["tflops"] / bf16_burst,
                "frac_of_sustained": d["tflops"] / bf16_sustained,
                "peak_nominal": NOMINAL["bf16_tflops"],
                "frac_nominal": d["tflops"] / NOMINAL["bf16_tflops"]}
    else:
        roof = {"bound": "hbm", "achieved": d["gbs"], "peak": hbm_gbs, "unit": "GB/s",
                "frac": d["gbs"] / hbm_gbs, "peak_source": f"{peak_kind} HBM copy",
                "peak_nominal": NOMINAL["hbm_gbs"], "frac_nominal": d["gbs"] / NOMINAL["hbm_gbs"]}
    roof.update({"kernel": dom, "traffic": traffic, "flops_per_launch": d["flops"],
                 "algorithmic_bytes_per_launch": d["bytes"]})

    # end to end through the public API: pinned host inputs in, result out
    x_h = inp.x.cpu().pin_memory()
    ids_h = inp.topk_ids.cpu().pin_memory()
    w_h = inp.topk_weights.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e2e_steps = min(args.steps, 50)
    # A serving loop: every step copies its inputs in and its output out, on
    # two copy streams, into double-buffered device tensors, so that step
    # i+1's host-to-device copy and step i-1's device-to-host copy run while
    # step i computes.
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = [dict(x=torch.empty_like(inp.x), ids=torch.empty_like(inp.topk_ids),
                 w=torch.empty_like(inp.topk_weights), out=torch.empty_like(out))
            for _ in range(2)]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, fwd_done, out_read = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def e2e_step(i):
        b = i & 1
        d = bufs[b]
        with torch.cuda.stream(h2d_s):
            if used[b]:
                h2d_s.wait_event(fwd_done[b])  # the forward two steps back has read buffer b
            d["x"].copy_(x_h, non_blocking=True)
            d["ids"].copy_(ids_h, non_blocking=True)
            d["w"].copy_(w_h, non_blocking=True)
            in_ready[b].record(h2d_s)
        stream.wait_event(in_ready[b])
        if used[b]:
            stream.wait_event(out_read[b])  # its output two steps back has been read out
        moe.moe_forward(p, d["x"], d["ids"], d["w"], w13, s13, w2, s2, d["out"], wsp.buffer,
                        wsp.nbytes, stream)
        fwd_done[b].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(fwd_done[b])
            out_h.copy_(d["out"], non_blocking=True)
            out_read[b].record(d2h_s)
        used[b] = True

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(h2d_s)
    for i in range(e2e_steps):
        e2e_step(3 + i)
    e1.record(d2h_s)  # after the last step's output copy, which follows all its work
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, ws, dev)
    if moe.moe_get_device_status(st, stream) != 0:
        raise RuntimeError("device status after the end-to-end loop")
    h2d = x_h.numel() * x_h.element_size() + ids_h.numel() * 4 + w_h.numel() * 4
    d2h = out_h.numel() * out_h.element_size()

    # the same forward captured once in a CUDA graph and replayed (device-
    # resident inputs): what a serving loop pays when it replays the layer
    graph_ms = cuda_graph_ms(moe, p, bufs[0], (w13, s13, w2, s2), wsp, dev, min(args.steps, 50))
    graph_ms = max_over_ranks(graph_ms, ws, dev)
    if moe.moe_get_device_status(st, stream) != 0:
        raise RuntimeError("device status after the graph replays")

    workloads, workloads_clocks = None, None
    if rank == 0 and ws == 1 and not args.no_workloads and args.shrink == 1 and \
            cfg.name == "mixtral_prefill":
        workloads, workloads_clocks = run_workloads(moe, _abi, args, dev, cfg, inp)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        inp_cpu = inp.to("cpu")
        rate, sample, threads = cpu_oracle_rate(cfg, inp_cpu, args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {"bf16": "bf16", "f32": "f32 (tf32 MMA)",
                      "mxfp4": "e4m3 x mxfp4 (fp32 acc)"}[cfg.dtype], "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E,
                       "top_k": cfg.K, "global_batch_tokens": tokens_all, "block_m": bm,
                       "combine": "fused into GEMM2 (fp32 atomics)" if args.fused_combine
                                  else "separate, deterministic",
                       "parallelism": f"replicas{ws}",
                       "l2": "inputs larger than L2 (expert weights %.2f GB)" %
                             (bytes_alg / 1e9)},
            "tflops": tflops,
            "hbm_gbs_algorithmic": bytes_alg * ws / (ms_step * 1e-3) / 1e9,
            "stage_ms": stage_ms,
            "stage_ms_source": "CUDA events between stages on every 4th timed step",
            "roofline": roof,
            "kernels": kern,
            "active_experts": active,
            "graph": {"value": tokens_all / (graph_ms * 1e-3), "unit": "tokens/s",
                      "ms_per_step": graph_ms,
                      "what": "moe_forward captured in one CUDA graph, replayed back to back"},
            "e2e": {"value": tokens_all / (e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms,
                    "copies": "pinned host buffers; each step's inputs in and output out on "
                              "two copy streams, overlapping the neighbouring steps' compute"},
            # one kernel per stage, the align three when it runs over many CTAs
            "gpu_launches": (len(stages) + (2 if wsp.sizes[_abi.MOE_WS_ALIGN] else 0)) *
                            args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        if workloads is not None:
            line["workloads"] = workloads
            line["workloads_clocks"] = workloads_clocks
            line["workloads_note"] = (
                "every other workload at full size, device-drawn inputs, 3 warm-up and "
                f"{args.workload_steps} timed steps each, stage-by-stage C-ABI calls with CUDA "
                "events around every stage; roofline.frac against the measured peaks "
                "(bf16 burst, HBM copy), frac_nominal against 2.25 PFLOP/s and 8 TB/s")
        print(json.dumps(line), flush=True)


def sweep_batch_sizes(E: int, K: int):
    """The batch sizes of the "MOE Bmm1 Fused Gather" benchmark
    (get_batch_sizes): 48 rows-per-expert counts from 4 to 992 in steps that
    widen with the size, times E / K."""
    bpe = [b for k in range(8) for b in range(2 ** (2 + k), 2 ** (3 + k), min(2 ** k, 32))]
    return [b * E // K for b in bpe]


def run_sweep(args, rank, local):
    """One expert shard (E / ep_shards local experts) of the GPT-OSS-shaped
    layer over the 48 batch sizes: the whole path per batch (tokens routed
    to other shards are skipped), timed like the main benchmark."""
    import mixture_experts_grouped_02_gb300 as moe
    from mixture_experts_grouped_02_gb300 import _abi

    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe._abi.lib()
    cfg0 = gen.config("lowp_oai")
    L = cfg0.E // args.ep_shards
    base = args.ep_rank * L
    experts = range(base, base + L)
    w13, w2, s13, s2 = gen.draw_weights(cfg0, seed=0, device=dev, experts=experts)
    full = gen.MoEInputs(cfg0, None, None, None, None, None)  # biases and scalars only
    gen.draw_swiglu_oai(full, seed=0, device=dev)
    hbm_gbs, _, _, peak_kind = peaks()
    points = []
    for T in sweep_batch_sizes(cfg0.E, cfg0.K):
        cfg = cfg0.with_tokens(T)
        ids, w = gen.route(gen.router_logits(cfg, 0, dev), cfg.K)
        inp = gen.MoEInputs(cfg, gen.draw_x(cfg, 0, dev), w13, w2, ids, w, s13, s2,
                            full.w13_bias[base:base + L].contiguous(),
                            full.w2_bias[base:base + L].contiguous(), full.swiglu_alpha,
                            full.swiglu_limit, full.h_scale)
        stages, p, wsp, _, _, bm, stream = build_stages(moe, _abi, cfg, inp, dev, 0, (base, L))
        steps = max(5, min(args.steps, 50))
        for _ in range(3):
            for _, f in stages:
                f()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
              for _ in range(steps)]
        torch.cuda.synchronize(dev)
        for i in range(steps):
            ev[i][0].record(stream)
            for j, (_, f) in enumerate(stages):
                f()
                ev[i][j + 1].record(stream)
        torch.cuda.synchronize(dev)
        if moe.moe_get_device_status(wsp.status, stream) != 0:
            raise RuntimeError(f"device status at T={T}")
        names = [n for n, _ in stages]
        ms = {n: statistics.median(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps))
              for j, n in enumerate(names)}
        total = sum(ms.values())
        flat = ids.flatten().long()
        local_n = int(((flat >= base) & (flat < base + L)).sum())
        active = int((torch.bincount(flat[(flat >= base) & (flat < base + L)] - base,
                                     minlength=L) > 0).sum())
        w13_bytes = active * (inp.w13[0].numel() + inp.w13_scale[0].numel())
        g1 = ms["gemm_gate_up"] * 1e-3
        points.append({"T": T, "local_assignments": local_n, "active_local_experts": active,
                       "ms_per_step": total, "tokens_per_s": T / (total * 1e-3),
                       "gemm_gate_up_ms": ms["gemm_gate_up"],
                       "gemm_gate_up_tflops": 4 * local_n * cfg.H * cfg.I / g1 / 1e12,
                       "gemm_gate_up_weight_gbs": w13_bytes / g1 / 1e9,
                       "gemm_gate_up_weight_hbm_frac": w13_bytes / g1 / 1e9 / hbm_gbs,
                       "stage_ms": ms})
        del stages, p, wsp, inp
        torch.cuda.empty_cache()
    line = {"metric": METRIC, "unit": "tokens/s", "impl": "ours", "n_gpus": 1,
            "data": "synthetic", "dtype": "e4m3 x mxfp4 (fp32 acc)",
            "config": {"workload": "lowp_oai batch sweep", "H": cfg0.H, "I": cfg0.I,
                       "E": cfg0.E, "top_k": cfg0.K, "ep_shards": args.ep_shards,
                       "local_experts": [base, base + L], "peak": f"{peak_kind} HBM copy"},
            "sweep": points}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, local = dist_env()
    if args.sweep:
        run_sweep(args, rank, local)
        return
    if args.impl == "reference":
        run_reference(args, ws, rank)  # rank 0 alone; no process group needed
    else:
        init_dist(ws, "nccl")
        run_ours(args, ws, rank, local)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
