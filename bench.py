"""Benchmark of the DeepSeekMoE layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

One step = one pass of the whole hot path over one synthetic batch: route,
permute, expert FFNs (routed + shared), combine, then the +-gamma bias
update.  Default workload: the V3-shaped prefill layer (T=8192, d=7168,
256 routed experts, top-8, 1 shared, intermediate 2048, bf16, seed 2).
Prints one JSON line.  N > 1 (torchrun) runs independent replicas, one per
GPU, with no data-path collective; value = all ranks' tokens / max time.

--impl reference times the CPU fp64 oracle (the only reference this method
has) on a bounded sample of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
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

from moe_inputs import as_f64, generate, get_config, upstream_grad  # noqa: E402

METRIC = "MoE-layer tokens/s at V3 shape"
# DRAM bytes (read + write) of one expert-FFN call (the grouped GEMM's two
# launches) from an ncu capture of the same kernel on a smaller case of the
# same shape, scaled by the units processed (see profiles/
# grouped_gemm_pair_small_v3dims.md, grouped_gemm_fp8_tm_small_v3dims.md).
# None where no capture exists.
MEASURED_TRAFFIC = {"v3_prefill": 25.6e9, "v3_prefill_fp8": 13.6e9}
L2_NOTE = "inputs larger than L2 (22.5 GB of expert weights read per step)"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained"),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0,
            "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def layer_flops(cfg) -> float:
    A = cfg.T * cfg.top_k
    return (6.0 * A * cfg.d * cfg.d_ff + 6.0 * cfg.T * cfg.d * cfg.n_shared *
            cfg.d_ff + 2.0 * cfg.T * cfg.d * cfg.n_routed)


def ffn_flops(cfg) -> float:
    A = cfg.T * cfg.top_k
    return 6.0 * (A + cfg.T * cfg.n_shared) * cfg.d * cfg.d_ff


def ffn_bytes(cfg, counts) -> float:
    """Algorithmic bytes of the expert-FFN call: weights of the experts that
    received tokens plus the shared experts (read once), the routed and
    shared input rows, and the outputs (fp16 for bf16 and e4m3 layers, fp32
    for fp32).  e4m3: one byte per weight plus one fp32 scale per 128 x 128
    block, one byte per input element plus one fp32 scale per 128."""
    fp8 = cfg.quant == "fp8"
    es = 2 if cfg.dtype == "bf16" else 4
    ws = 1.0 + 4.0 / (128 * 128) if fp8 else es
    xs = 1.0 + 4.0 / 128 if fp8 else es
    ys = 2 if cfg.dtype == "bf16" else 4
    touched = int((np.asarray(counts) > 0).sum())
    w = 3.0 * cfg.d * cfg.d_ff * ws * (touched + cfg.n_shared)
    A = cfg.T * cfg.top_k
    act = (A + cfg.T) * cfg.d * xs + (A + cfg.T) * cfg.d * ys
    return w + act


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no-smi"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x: float, device="cpu") -> float:
    """Largest value of a per-rank float over all ranks of the initialised
    process group (the value itself without one).  The bench's timers are
    reduced this way: the job is as slow as its slowest replica."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    if dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: int, steps: int,
                   ms_max: float) -> float:
    """Units per second of the whole job: every replica processes its own
    units (weak scaling), all within the slowest replica's time."""
    return world * units_per_rank * steps / (ms_max / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def cpu_baseline(cfg, t, budget_s: float = 15.0, max_tokens: int = 512):
    """The fp64 oracle, as it stands, on a bounded sample of this workload:
    the whole routing of sampled tokens plus their routed and shared FFNs.
    Returns tokens/s and what the sample was."""
    import oracle.moe as om
    import oracle.fp8 as of
    fp8 = cfg.quant == "fp8"
    try:
        from threadpoolctl import threadpool_info
        blas = max((i.get("num_threads", 1) for i in threadpool_info()),
                   default=1)
    except Exception:
        blas = os.cpu_count()
    rng = np.random.default_rng(cfg.seed + 99)
    order = rng.permutation(cfg.T)
    E64, b64 = as_f64(t["E"]), as_f64(t["b"])
    shared = [tuple(as_f64(t[k][s]) for k in ("ws_gate", "ws_up", "ws_down"))
              for s in range(cfg.n_shared)]
    if fp8:       # weights are quantized once, outside the timed region
        shared = [of.quantize_expert(*w) for w in shared]
    host = {}

    def routed(e):
        return host[e]
    done, spent = 0, 0.0
    for tok in order[:max_tokens]:
        u64 = as_f64(t["u"][int(tok):int(tok) + 1])
        t0 = time.perf_counter()
        r = om.route(u64, E64, b64, cfg.top_k)
        spent += time.perf_counter() - t0
        for e in r["idx"][0].tolist():      # stage weights on the host (untimed)
            if e not in host:
                w = tuple(t[k][e].cpu().to(torch.float64).numpy() for k in
                          ("w_gate", "w_up", "w_down"))
                host[e] = of.quantize_expert(*w) if fp8 else w
        t0 = time.perf_counter()
        if fp8:
            r = om.route(u64, E64, b64, cfg.top_k)
            of.fp8_layer_forward(u64, r["idx"], r["gate"], routed, shared)
        else:
            om.layer_forward(u64, E64, b64, cfg.top_k, routed, shared)
        spent += time.perf_counter() - t0
        done += 1
        if spent >= budget_s:
            break
    return {"value": done / spent, "unit": "tokens/s", "cores": int(blas),
            "kind": "oracle",
            "sample": f"{done} of {cfg.T} tokens of {cfg.name} (routing + "
                      f"routed and shared FFNs, fp64"
                      f"{', e4m3 operands' if fp8 else ''}), {spent:.1f} s"}


def run_reference(args, cfg):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    torch.manual_seed(0)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = generate(cfg, dev)
    per_step = []
    per_tok = max(1, int(args.ref_tokens))
    for i in range(args.warmup + args.steps):
        c = cpu_baseline(cfg, t, budget_s=args.ref_budget, max_tokens=per_tok)
        if i >= args.warmup:
            per_step.append(c)
    value = statistics.mean(c["value"] for c in per_step)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * cfg.T / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d,
                       "n_routed": cfg.n_routed, "top_k": cfg.top_k,
                       "n_shared": cfg.n_shared, "d_ff": cfg.d_ff},
            "cpu_baseline": dict(per_step[-1], value=value),
            "e2e": {"value": value, "unit": "tokens/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_skew(args, cfg, moe, dev, ws, rank, local):
    """The skewed-load bias loop: cfg.steps steps, each with a fresh batch,
    every one followed by the +-gamma bias update.  Reports throughput and
    the max/mean expert load of every step."""
    from moe_inputs import step_tokens
    t = generate(cfg, dev)
    steps = cfg.steps
    us = [step_tokens(cfg, s, dev) for s in range(steps)]
    bias0 = t["b"].clone()
    layer = moe.MoELayer(t["E"], t["b"].clone(), t["w_gate"], t["w_up"],
                         t["w_down"], t["ws_gate"], t["ws_up"], t["ws_down"],
                         top_k=cfg.top_k, h_dtype=torch.bfloat16)
    bufs = layer.buffers(cfg.T)
    loads = torch.empty((steps, cfg.n_routed), dtype=torch.int32, device=dev)
    for s in range(max(3, args.warmup)):          # warm-up on a scratch bias
        layer(us[s % steps], update_bias=True, gamma=cfg.gamma)
    torch.cuda.synchronize()
    layer.bias.copy_(bias0)
    moe.get_device_error()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(steps):
        layer(us[s], update_bias=True, gamma=cfg.gamma)
        loads[s].copy_(bufs.counts)
    t1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    clk = clocks.stop()
    moe.get_device_error()
    ms = max_over_ranks(t0.elapsed_time(t1), dev)
    c = loads.cpu().numpy().astype(np.float64)
    mean = cfg.T * cfg.top_k / cfg.n_routed
    mm = (c.max(axis=1) / mean).tolist()
    peaks = _peaks()
    line = {"metric": METRIC, "value": whole_job_rate(ws, cfg.T, steps, ms),
            "unit": "tokens/s", "n_gpus": ws, "steps": steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d,
                       "n_routed": cfg.n_routed, "top_k": cfg.top_k,
                       "n_shared": cfg.n_shared, "d_ff": cfg.d_ff,
                       "gamma": cfg.gamma, "zipf": cfg.zipf,
                       "parallelism": f"replicas x{ws}", "l2": L2_NOTE,
                       "shared_experts_on_side_stream": side is not None},
            "layer_tflops": layer_flops(cfg) / (ms / steps / 1e3) / 1e12,
            "layer_frac_of_bf16_peak": layer_flops(cfg) / (ms / steps / 1e3) /
            1e12 / peaks["bf16_tflops"],
            "load_max_over_mean": {"first": mm[0], "last": mm[-1],
                                   "per_step": [round(x, 3) for x in mm]},
            "clocks": clk}
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_backward(args, cfg, layer, u, dev, ws, peaks):
    """The layer backward (moe_backward: Dgrad and Wgrad GEMMs, gate and
    centroid gradients) after a forward on the same batch, timed with CUDA
    events on the launching stream; and a training step (forward + backward)
    timed over the same number of steps.  Weight gradients in bf16."""
    import mixture_experts_layer_gemms_b300 as moe
    dh = upstream_grad(cfg, dev)
    stream = torch.cuda.current_stream()
    gd = torch.bfloat16
    layer.overlap_shared = False
    for _ in range(max(3, args.warmup)):
        layer(u)
        layer.backward(u, dh, grad_dtype=gd)
    torch.cuda.synchronize()
    moe.get_device_error()
    n_launch = moe.last_launch_count()
    steps = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
          for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        layer(u)
        ev[i][1].record(stream)
        layer.backward(u, dh, grad_dtype=gd)
        ev[i][2].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    moe.get_device_error()
    bw_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    train_ms = max_over_ranks(t0.elapsed_time(t1), dev) / steps
    rows = cfg.T * cfg.top_k + cfg.n_shared * cfg.T
    # algorithmic: twice the expert FFNs' forward FLOPs (Dgrad + Wgrad);
    # executed adds the recomputed gate/up GEMM
    alg = 12.0 * cfg.d * cfg.d_ff * rows
    exe = 16.0 * cfg.d * cfg.d_ff * rows
    pk = peaks["bf16_tflops"]
    ach = alg / (bw_ms / 1e3) / 1e12
    roof = {"bound": "tensor", "achieved": ach, "peak": pk,
            "unit": "TFLOP/s", "frac": ach / pk, "traffic": None,
            "kernel": "the moe_backward call (Dgrad, recompute and Wgrad "
                      "CTA-pair GEMMs are 95% of it); algorithmic FLOPs "
                      "12 d d_ff per token-expert and per shared-expert "
                      "token",
            "peak_source": f"{peaks['source']} bf16_tflops (burst)"}
    return {"ms_per_call": bw_ms, "roofline": roof,
            "train_step_tokens_per_s": ws * cfg.T / (train_ms / 1e3),
            "train_step_ms": train_ms,
            "algorithmic_tflops": alg / (bw_ms / 1e3) / 1e12,
            "executed_tflops": exe / (bw_ms / 1e3) / 1e12,
            "executed_frac_of_bf16_peak": exe / (bw_ms / 1e3) / 1e12 / pk,
            "grad_dtype": "bf16", "gpu_launches_per_call": n_launch,
            "note": "moe_backward after a forward of the same batch: "
                    "gather, Dgrad (down, gate/up), gate/up recompute with "
                    "the SwiGLU backward, Wgrad (gate/up, down), centroid "
                    "and input gradients"}


def run_ours(args, cfg):
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import mixture_experts_layer_gemms_b300 as moe

    dev = torch.device("cuda", local)
    if cfg.steps > 1:
        run_skew(args, cfg, moe, dev, ws, rank, local)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    t = generate(cfg, dev)
    layer = moe.MoELayer(t["E"], t["b"].clone(), t["w_gate"], t["w_up"],
                         t["w_down"], t["ws_gate"], t["ws_up"], t["ws_down"],
                         top_k=cfg.top_k, h_dtype=torch.bfloat16,
                         quant=cfg.quant)
    u = t["u"]
    bufs = layer.buffers(cfg.T)
    sh = layer.shape(cfg.T)
    stream = torch.cuda.current_stream()
    # --overlap-shared: the shared experts beside the permute on a side
    # stream (as MoELayer(overlap_shared=True)); no faster on the device at
    # the V3 prefill shape (the step is power-capped), so the timed C-ABI
    # step keeps one expert-FFN call
    layer.overlap_shared = args.overlap_shared
    side = layer._shared_side_stream(u)
    # events between the calls of every timed step: route | permute |
    # expert_ffn | combine | update_bias
    CALLS = ("route", "permute", "expert_ffn", "combine", "update_bias")
    # (with the shared experts on the side stream, a 7th event marks their
    # start there, and the expert-FFN span runs from it to the join)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)]
          for _ in range(args.steps)]

    def step(i=None):
        """One step through the C ABI; returns kernels launched."""
        def mark(j):
            if i is not None:
                ev[i][j].record(stream)
        n = 0
        mark(0)
        moe.route(sh, u, layer.E, layer.bias, bufs.topk_idx, bufs.topk_gate,
                  bufs.counts, bufs.workspace)
        n += moe.last_launch_count()
        mark(1)
        if side is not None:
            # shared experts on a side stream beside the permute
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                if i is not None:
                    ev[i][6].record(side)
                moe.expert_ffn_part(sh, 2, None, None, None, None, u,
                                    layer.ws_gu, layer.ws_down, None,
                                    bufs.y_shared, bufs.workspace)
                n_side = moe.last_launch_count()
        moe.permute(sh, u, bufs.topk_idx, bufs.counts, bufs.offsets,
                    bufs.perm, bufs.inv, bufs.x_perm, bufs.workspace)
        n += moe.last_launch_count()
        mark(2)
        if side is not None:
            moe.expert_ffn_part(sh, 1, bufs.x_perm, bufs.offsets, layer.w_gu,
                                layer.w_down, u, None, None, bufs.y_perm,
                                None, bufs.workspace)
            n += moe.last_launch_count() + n_side
            stream.wait_stream(side)
        else:
            moe.expert_ffn(sh, bufs.x_perm, bufs.offsets, layer.w_gu,
                           layer.w_down, u, layer.ws_gu, layer.ws_down,
                           bufs.y_perm, bufs.y_shared, bufs.workspace)
            n += moe.last_launch_count()
        mark(3)
        moe.combine(sh, u, bufs.y_perm, bufs.y_shared, bufs.inv,
                    bufs.topk_gate, bufs.h)
        n += moe.last_launch_count()
        mark(4)
        moe.update_bias(cfg.n_routed, bufs.counts, cfg.T * cfg.top_k,
                        cfg.gamma, layer.bias)
        n += moe.last_launch_count()
        mark(5)
        return n

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    moe.get_device_error()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    launches = 0
    for i in range(args.steps):
        launches += step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    moe.get_device_error()
    ms = max_over_ranks(t0.elapsed_time(t1), dev)
    call_ms = {c: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev)
               for j, c in enumerate(CALLS)}
    if side is not None:
        # both expert-FFN parts: from the shared part's start on the side
        # stream to the join after the routed part (the span also covers
        # the permute beside it, so the rate below is a lower bound)
        call_ms["expert_ffn"] = statistics.mean(e[6].elapsed_time(e[3])
                                                for e in ev)
    ffn_ms = call_ms["expert_ffn"]
    counts = bufs.counts.cpu().numpy()

    # end to end through the public API with host buffers: every step
    # uploads its tokens from pinned memory, runs the layer and reads h back
    # (MoELayer.forward_host overlaps step i's copies with the compute of
    # its neighbours)
    # (the layer runs its shared experts on a side stream here: beside the
    # copy streams that measured 3% faster end to end)
    layer.overlap_shared = True
    e_steps = max(2, min(args.steps, 10))
    u_host = [u.cpu().pin_memory() for _ in range(2)]
    h_host = [torch.empty(bufs.h.shape, dtype=bufs.h.dtype).pin_memory()
              for _ in range(2)]
    ins = [u_host[i % 2] for i in range(e_steps)]
    outs = [h_host[i % 2] for i in range(e_steps)]
    layer.forward_host(ins[:2], outs[:2], update_bias=True, gamma=cfg.gamma)
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    layer.forward_host(ins, outs, update_bias=True, gamma=cfg.gamma)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, dev)
    moe.get_device_error()

    # the same step captured once as a CUDA graph and replayed
    replay = layer.graph(u, update_bias=True, gamma=cfg.gamma)
    for _ in range(2):
        replay()
    torch.cuda.synchronize()
    barrier()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        replay()
    g1.record(stream)
    torch.cuda.synchronize()
    barrier()
    g_ms = max_over_ranks(g0.elapsed_time(g1), dev)
    moe.get_device_error()

    peaks = _peaks()
    bwd = None
    if (not args.no_backward and cfg.quant is None and cfg.dtype == "bf16"
            and cfg.d_ff % 128 == 0):
        bwd = time_backward(args, cfg, layer, u, dev, ws, peaks)
    fp8 = cfg.quant == "fp8"
    # e4m3 contractions: the measured bf16 peak times the nominal dense
    # e4m3 : bf16 ratio (4.5 : 2.25 PFLOP/s)
    tc_peak = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
    tc_src = (f"{peaks['source']} bf16_tflops (burst) x 2 (nominal e4m3:bf16)"
              if fp8 else f"{peaks['source']} bf16_tflops (burst)")
    ms_step = ms / args.steps
    value = whole_job_rate(ws, cfg.T, args.steps, ms)
    decode = cfg.T * cfg.top_k <= 48 * cfg.n_routed
    if decode:
        ach = ffn_bytes(cfg, counts) / (ffn_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                "traffic": None,
                "kernel": ("grouped_gemm_fp8_kernel<32,1,*>" if fp8 else
                           "grouped_gemm_kernel<32,10>") +
                          " (gate/up + down launches of one expert-FFN call)",
                "peak_source": f"{peaks['source']} hbm_gbs"}
    else:
        ach = ffn_flops(cfg) / (ffn_ms / 1e3) / 1e12
        sus = peaks["bf16_tflops_sustained"]
        roof = {"bound": "tensor", "achieved": ach,
                "peak": tc_peak, "unit": "TFLOP/s",
                "frac": ach / tc_peak,
                "traffic": MEASURED_TRAFFIC.get(cfg.name),
                "kernel": ("grouped_gemm_fp8_tm_kernel" if fp8 else
                           "grouped_gemm_pair_kernel") +
                          " (gate/up + down launches of one expert-FFN call)",
                "peak_source": tc_src,
                "frac_of_sustained": (ach / (sus * (2.0 if fp8 else 1.0))
                                      if sus else None)}
    roof["ms_per_launch_pair"] = ffn_ms
    # algorithmic bytes of the bandwidth calls (read + write), judged in GB/s
    A = cfg.T * cfg.top_k
    es = 2 if cfg.dtype == "bf16" else 4           # u, E, y elements
    xe = 1.0 + 4.0 / 128 if fp8 else es            # x_perm bytes / element
    hb = bufs.h.element_size()
    ys = es if cfg.n_shared else 0
    call_bytes = {
        "route": cfg.T * cfg.d * es + cfg.n_routed * cfg.d * es + A * 8 +
                 cfg.n_routed * 4,
        "permute": cfg.T * cfg.d * es + A * cfg.d * xe + A * 12,
        "combine": cfg.T * cfg.d * (es + ys + hb) + A * cfg.d * es + A * 8,
        "update_bias": cfg.n_routed * 12,
    }
    per_call = {c: {"ms": round(call_ms[c], 4)} for c in CALLS}
    for c, nbytes in call_bytes.items():
        per_call[c]["gbs"] = round(nbytes / (call_ms[c] / 1e3) / 1e9, 1)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if fp8 else "bf16",
            "data": "synthetic",
            "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d,
                       "n_routed": cfg.n_routed, "top_k": cfg.top_k,
                       "n_shared": cfg.n_shared, "d_ff": cfg.d_ff,
                       "parallelism": f"replicas x{ws}", "l2": L2_NOTE,
                       "shared_experts_on_side_stream": side is not None},
            "layer_tflops": layer_flops(cfg) / (ms_step / 1e3) / 1e12,
            ("layer_frac_of_e4m3_peak" if fp8 else "layer_frac_of_bf16_peak"):
            layer_flops(cfg) / (ms_step / 1e3) / 1e12 / tc_peak,
            "roofline": roof,
            "clocks": clk,
            "gpu_launches": launches * ws,
            "per_call": per_call,
            "graph": {"value": whole_job_rate(ws, cfg.T, args.steps, g_ms),
                      "unit": "tokens/s", "ms_per_step": g_ms / args.steps,
                      "note": "the same step replayed from one CUDA graph "
                              "(shared experts on a side stream)"},
            "e2e": {"value": ws * cfg.T / (e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": u.numel() * u.element_size(),
                    "d2h_bytes_per_step": bufs.h.numel() *
                    bufs.h.element_size(),
                    "how": "MoELayer(overlap_shared=True).forward_host: "
                           "pinned-host batches, copies on their own streams "
                           "overlapping the neighbouring steps' compute"}}
    if bwd is not None:
        line["backward"] = bwd
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, t, budget_s=args.ref_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="v3_prefill")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward-pass block of the line")
    ap.add_argument("--overlap-shared", action="store_true",
                    help="shared experts on a side stream in the timed step")
    ap.add_argument("--ref-budget", type=float, default=15.0,
                    help="seconds of oracle work per reference step")
    ap.add_argument("--ref-tokens", type=int, default=4,
                    help="tokens per reference step (upper bound)")
    ap.add_argument("--set", action="append", default=[], metavar="KEY=VAL",
                    help="override a workload field (profiling of a smaller "
                         "case of the same kernels; not a bench line)")
    args = ap.parse_args()
    cfg = get_config(args.workload)
    if args.set:
        over = {}
        for kv in args.set:
            k, v = kv.split("=", 1)
            over[k] = type(getattr(cfg, k))(v)
        cfg = cfg.with_(name=cfg.name + "+" + ",".join(args.set), **over)
    if args.impl == "reference":
        if args.ref_budget > 10.0:
            args.ref_budget = 10.0
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
