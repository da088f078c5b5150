"""Benchmark of the DeepSeekMoE layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline] [--no-extra]

One step = one pass of the whole hot path over one synthetic batch: route,
permute, expert FFNs (routed + shared), combine, then the +-gamma bias
update.  Default workload: the V3-shaped prefill layer (T=8192, d=7168,
256 routed experts, top-8, 1 shared, intermediate 2048, bf16, seed 2).
Prints one JSON line.  With the default workload the line also carries two
blocks measured in the same run, each with its own roofline, clocks and CPU
baseline:

* ``decode``: the V3-shaped decode layer (T=128, same layer dimensions,
  seed 3), bound by streaming the touched experts' weights from HBM;
* ``skew``: the skewed-load bias loop (T=16384 tokens per step, 50 steps,
  Zipf-scaled centroids, gamma=1e-3, a fresh batch every step) with the
  max/mean expert load of every step.

N > 1 (torchrun) runs independent replicas, one per GPU, with no data-path
collective; value = all ranks' tokens / max time.

--impl reference times the CPU fp64 oracle (the only reference this method
has) on a fixed seeded sample of the workload's tokens, on rank 0 only.
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

from moe_inputs import (as_f64, generate, get_config, step_tokens,  # noqa: E402
                        upstream_grad)

METRIC = "MoE-layer tokens/s at V3 shape"
# DRAM bytes (read + write) of one expert-FFN call (the grouped GEMM's two
# launches) relative to the call's algorithmic bytes, from an ncu capture of
# the same kernels on a smaller case of the same layer dimensions (fewer
# experts, so the routed weights still exceed L2).  Traffic grows with the
# units processed (touched experts' weights, rows), so the ratio carries
# over to the full size.  None where no capture of the current kernel
# exists.
TRAFFIC_RATIO = {"v3_prefill": 3.276123 / 3.246,
                 "v3_prefill_fp8": 1.677290 / 1.653926,
                 "v3_decode": 2.918043 / 2.910781, "skew": None}
L2_NOTE = "inputs larger than L2 (22.5 GB of expert weights read per step)"
CPU_TOKENS = 16     # tokens in the oracle's timed sample


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
        sm, smax, reasons, cap = [], [], set(), 0
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
                    cap += n == "sw_power_cap"
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_cap_samples": cap}


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


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        return int(max((i.get("num_threads", 1) for i in threadpool_info()),
                       default=1))
    except Exception:
        return int(os.cpu_count() or 1)


# ------------------------------------------------------------ CPU oracle --
class OracleSample:
    """The fp64 oracle, as it stands, on a fixed seeded sample of one
    workload's tokens: routing of the sampled tokens plus their routed and
    shared expert FFNs and the combine (``oracle.moe.layer_forward``).

    The same sample serves the ``cpu_baseline`` object of the GPU line and
    every step of ``--impl reference``, so both report the same rate.  The
    experts' weights are widened to fp64 on the host one expert at a time
    as the oracle asks for them; that staging is timed separately and taken
    out of the oracle's seconds (it is data movement, not the method)."""

    def __init__(self, cfg, t, n_tokens: int, u=None):
        import oracle.fp8 as of
        self.cfg = cfg
        self.fp8 = cfg.quant == "fp8"
        self.t = t
        src = t["u"] if u is None else u
        rng = np.random.default_rng(cfg.seed + 99)
        n = max(1, min(int(n_tokens), src.shape[0]))
        self.tokens = np.sort(rng.permutation(src.shape[0])[:n])
        sel = torch.from_numpy(self.tokens).to(src.device)
        self.u64 = as_f64(src[sel])
        self.E64, self.b64 = as_f64(t["E"]), as_f64(t["b"])
        self.shared = [tuple(as_f64(t[k][s]) for k in
                             ("ws_gate", "ws_up", "ws_down"))
                       for s in range(cfg.n_shared)]
        if self.fp8:      # quantized once, outside the timed region
            self.shared = [of.quantize_expert(*w) for w in self.shared]
        self._q = {}
        self.stage_s = 0.0

    def _routed(self, e: int):
        t0 = time.perf_counter()
        if self.fp8 and e in self._q:
            w = self._q[e]
        else:
            w = tuple(self.t[k][e].to(torch.float64).cpu().numpy()
                      for k in ("w_gate", "w_up", "w_down"))
            if self.fp8:
                import oracle.fp8 as of
                w = self._q.setdefault(e, of.quantize_expert(*w))
        self.stage_s += time.perf_counter() - t0
        return w

    def step(self):
        """One pass over the sample; returns (oracle seconds, wall seconds)."""
        import oracle.fp8 as of
        import oracle.moe as om
        self.stage_s = 0.0
        t0 = time.perf_counter()
        if self.fp8:
            r = om.route(self.u64, self.E64, self.b64, self.cfg.top_k)
            of.fp8_layer_forward(self.u64, r["idx"], r["gate"], self._routed,
                                 self.shared)
        else:
            om.layer_forward(self.u64, self.E64, self.b64, self.cfg.top_k,
                             self._routed, self.shared)
        wall = time.perf_counter() - t0
        return wall - self.stage_s, wall

    def describe(self, oracle_s: float, wall_s: float) -> str:
        return (f"{self.tokens.size} of {self.cfg.T} tokens (seeded) of "
                f"{self.cfg.name}: routing, routed and shared FFNs and "
                f"combine in fp64{', e4m3 operands' if self.fp8 else ''}; "
                f"{oracle_s:.2f} s "
                f"of oracle work ({wall_s:.2f} s with the host staging of "
                f"expert weights)")


def cpu_baseline(cfg, t, n_tokens: int = CPU_TOKENS, u=None):
    s = OracleSample(cfg, t, n_tokens, u)
    oracle_s, wall = s.step()
    return {"value": s.tokens.size / oracle_s, "unit": "tokens/s",
            "cores": _blas_threads(), "kind": "oracle",
            "sample": s.describe(oracle_s, wall)}


def run_reference(args, cfg):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = generate(cfg, dev)
    u = step_tokens(cfg, 0, dev) if cfg.steps > 1 else None
    s = OracleSample(cfg, t, args.cpu_tokens, u)
    t_run = time.perf_counter()
    work = []
    for i in range(args.warmup + args.steps):
        o, w = s.step()
        if i >= args.warmup:
            work.append((o, w))
    run_s = time.perf_counter() - t_run
    oracle_s = statistics.mean(o for o, _ in work)
    wall_s = statistics.mean(w for _, w in work)
    n = int(s.tokens.size)
    value = n / oracle_s
    line = {"metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * oracle_s, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "extrapolated": True, "tokens_per_step": n,
            "sampled_wall_s": round(run_s, 2),
            "note": f"each step is the oracle over the same {n}-token sample "
                    f"of the {cfg.T}-token batch; value = sampled tokens per "
                    f"second of oracle work, extrapolated to the workload "
                    f"(the layer is per-token independent)",
            "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d,
                       "n_routed": cfg.n_routed, "top_k": cfg.top_k,
                       "n_shared": cfg.n_shared, "d_ff": cfg.d_ff},
            "cpu_baseline": {"value": value, "unit": "tokens/s",
                             "cores": _blas_threads(), "kind": "oracle",
                             "sample": s.describe(oracle_s, wall_s)},
            "e2e": {"value": value, "unit": "tokens/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- the timed steps --
CALLS = ("route", "permute", "expert_ffn", "combine", "update_bias")


def make_step(moe, cfg, layer, T, side=None):
    """One layer step through the C ABI: route | permute | expert_ffn |
    combine | update_bias, with an optional CUDA event before each call (and
    after the last).  Returns the kernels launched."""
    bufs = layer.buffers(T)
    sh = layer.shape(T)
    stream = torch.cuda.current_stream()

    def step(u, ev=None):
        def mark(j):
            if ev is not None:
                ev[j].record(stream)
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
                if ev is not None:
                    ev[6].record(side)
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
        moe.update_bias(cfg.n_routed, bufs.counts, T * cfg.top_k, cfg.gamma,
                        layer.bias)
        n += moe.last_launch_count()
        mark(5)
        return n
    return step


def timed_steps(moe, step, inputs, steps, warmup, ws, local, dev,
                after_step=None, before_timing=None, side=False):
    """``warmup`` untimed steps, then ``steps`` timed steps bracketed by a
    barrier and a device synchronise on both sides, inputs[i % len]; CUDA
    events on the launching stream around the whole loop and between the
    calls of every step; nvidia-smi clocks sampled during the loop.
    Returns (ms over ranks, per-call ms, launches, clocks)."""
    stream = torch.cuda.current_stream()
    for i in range(max(3, warmup)):
        step(inputs[i % len(inputs)])
    torch.cuda.synchronize()
    moe.get_device_error()
    if before_timing is not None:
        before_timing()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)]
          for _ in range(steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    _barrier(ws)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    launches = 0
    for i in range(steps):
        launches += step(inputs[i % len(inputs)], ev[i])
        if after_step is not None:
            after_step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    clk = clocks.stop()
    moe.get_device_error()
    ms = max_over_ranks(t0.elapsed_time(t1), dev)
    call_ms = {c: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev)
               for j, c in enumerate(CALLS)}
    if side:
        # both expert-FFN parts: from the shared part's start on the side
        # stream to the join after the routed part
        call_ms["expert_ffn"] = statistics.mean(e[6].elapsed_time(e[3])
                                                for e in ev)
    return ms, call_ms, launches, clk


def call_rates(cfg, call_ms, h_bytes):
    """Per-call ms and algorithmic GB/s of the bandwidth-bound calls."""
    A = cfg.T * cfg.top_k
    fp8 = cfg.quant == "fp8"
    es = 2 if cfg.dtype == "bf16" else 4           # u, E, y elements
    xe = 1.0 + 4.0 / 128 if fp8 else es            # x_perm bytes / element
    ys = es if cfg.n_shared else 0
    call_bytes = {
        "route": cfg.T * cfg.d * es + cfg.n_routed * cfg.d * es + A * 8 +
                 cfg.n_routed * 4,
        "permute": cfg.T * cfg.d * es + A * cfg.d * xe + A * 12,
        "combine": cfg.T * cfg.d * (es + ys + h_bytes) + A * cfg.d * es +
                   A * 8,
        "update_bias": cfg.n_routed * 12,
    }
    per_call = {c: {"ms": round(call_ms[c], 4)} for c in CALLS}
    for c, nbytes in call_bytes.items():
        per_call[c]["gbs"] = round(nbytes / (call_ms[c] / 1e3) / 1e9, 1)
    return per_call


def ffn_roofline(cfg, counts, ffn_ms, peaks, traffic_key):
    """The roofline object of the expert-FFN call (the dominant kernel:
    the grouped GEMM's gate/up and down launches)."""
    fp8 = cfg.quant == "fp8"
    decode = cfg.T * cfg.top_k <= 48 * cfg.n_routed
    ratio = TRAFFIC_RATIO.get(traffic_key)
    alg_bytes = ffn_bytes(cfg, counts)
    traffic = alg_bytes * ratio if ratio else None
    if decode:
        ach = alg_bytes / (ffn_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                "traffic": traffic,
                "algorithmic_bytes": alg_bytes,
                "kernel": ("grouped_gemm_fp8_pair_kernel" if fp8 else
                           "grouped_gemm_kernel<32,10>") +
                          " (gate/up + down launches of one expert-FFN call)",
                "peak_source": f"{peaks['source']} hbm_gbs (copy)"}
    else:
        # e4m3 contractions: the measured bf16 peak times the nominal dense
        # e4m3 : bf16 ratio (4.5 : 2.25 PFLOP/s)
        tc_peak = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
        sus = peaks["bf16_tflops_sustained"]
        ach = ffn_flops(cfg) / (ffn_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": tc_peak,
                "unit": "TFLOP/s", "frac": ach / tc_peak,
                "traffic": traffic,
                "algorithmic_bytes": alg_bytes,
                "kernel": ("grouped_gemm_fp8_pair_kernel" if fp8 else
                           "grouped_gemm_pair_kernel") +
                          " (gate/up + down launches of one expert-FFN call)",
                "peak_source": (f"{peaks['source']} bf16_tflops (burst)"
                                + (" x 2 (nominal e4m3:bf16)" if fp8 else "")),
                "frac_of_sustained": (ach / (sus * (2.0 if fp8 else 1.0))
                                      if sus else None)}
    roof["ms_per_launch_pair"] = ffn_ms
    return roof


def _new_layer(moe, cfg, t, overlap=False):
    return moe.MoELayer(t["E"], t["b"].clone(), t["w_gate"], t["w_up"],
                        t["w_down"], t["ws_gate"], t["ws_up"], t["ws_down"],
                        top_k=cfg.top_k, h_dtype=torch.bfloat16,
                        quant=cfg.quant, overlap_shared=overlap)


def _free():
    import gc
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def time_backward(args, cfg, layer, u, dev, ws, peaks):
    """The layer backward (moe_backward: Dgrad and Wgrad GEMMs, gate and
    centroid gradients) after a forward on the same batch that saved its
    gate/up pre-activations, timed with CUDA events on the launching stream;
    and a training step (that forward + backward) timed over the same number
    of steps.  Weight gradients in bf16."""
    import mixture_experts_layer_gemms_b300 as moe
    dh = upstream_grad(cfg, dev)
    stream = torch.cuda.current_stream()
    gd = torch.bfloat16
    layer.overlap_shared = False
    for _ in range(max(3, args.warmup)):
        layer(u, save_for_backward=True)
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
        layer(u, save_for_backward=True)
        ev[i][1].record(stream)
        layer.backward(u, dh, grad_dtype=gd)
        ev[i][2].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    moe.get_device_error()
    bw_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    train_ms = max_over_ranks(t0.elapsed_time(t1), dev) / steps
    rows = cfg.T * cfg.top_k + cfg.n_shared * cfg.T
    # algorithmic = executed: twice the expert FFNs' forward FLOPs (Dgrad +
    # Wgrad); the gate/up pre-activations come from the forward, so no
    # GEMM is recomputed
    alg = 12.0 * cfg.d * cfg.d_ff * rows
    exe = alg
    pk = peaks["bf16_tflops"]
    ach = alg / (bw_ms / 1e3) / 1e12
    roof = {"bound": "tensor", "achieved": ach, "peak": pk,
            "unit": "TFLOP/s", "frac": ach / pk, "traffic": None,
            "kernel": "the moe_backward call (its Dgrad and Wgrad CTA-pair "
                      "GEMMs are ~95% of it); algorithmic FLOPs "
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
            "note": "moe_backward after a forward of the same batch that "
                    "saved its gate/up pre-activations (fp16): gather, Dgrad "
                    "(down, with the SwiGLU backward in its epilogue; "
                    "gate/up), Wgrad (gate/up, down), centroid and input "
                    "gradients"}


def forward_block(args, cfg, moe, dev, ws, rank, local, headline):
    """Times the layer forward of one single-batch workload; returns the
    JSON object (the whole line for the headline workload)."""
    peaks = _peaks()
    t = generate(cfg, dev)
    layer = _new_layer(moe, cfg, t)
    u = t["u"]
    bufs = layer.buffers(cfg.T)
    # --overlap-shared: the shared experts beside the permute on a side
    # stream (as MoELayer(overlap_shared=True)); no faster on the device at
    # the V3 prefill shape (the step is power-capped), so the timed C-ABI
    # step keeps one expert-FFN call by default
    layer.overlap_shared = args.overlap_shared
    side = layer._shared_side_stream(u)
    step = make_step(moe, cfg, layer, cfg.T, side)
    ms, call_ms, launches, clk = timed_steps(
        moe, step, [u], args.steps, args.warmup, ws, local, dev,
        side=side is not None)
    counts = bufs.counts.cpu().numpy()
    fp8 = cfg.quant == "fp8"
    tc_peak = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
    ms_step = ms / args.steps
    out = {"metric": METRIC,
           "value": whole_job_rate(ws, cfg.T, args.steps, ms),
           "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
           "warmup": max(3, args.warmup), "ms_per_step": ms_step,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "e4m3" if fp8 else cfg.dtype, "data": "synthetic",
           "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d,
                      "n_routed": cfg.n_routed, "top_k": cfg.top_k,
                      "n_shared": cfg.n_shared, "d_ff": cfg.d_ff,
                      "parallelism": f"replicas x{ws}", "l2": L2_NOTE,
                      "shared_experts_on_side_stream": side is not None},
           "layer_tflops": layer_flops(cfg) / (ms_step / 1e3) / 1e12,
           ("layer_frac_of_e4m3_peak" if fp8 else "layer_frac_of_bf16_peak"):
           layer_flops(cfg) / (ms_step / 1e3) / 1e12 / tc_peak,
           "roofline": ffn_roofline(cfg, counts, call_ms["expert_ffn"], peaks,
                                    cfg.name),
           "clocks": clk,
           "gpu_launches": launches * ws,
           "per_call": call_rates(cfg, call_ms, bufs.h.element_size())}

    # end to end through the public API with host buffers: every step
    # uploads its tokens from pinned memory, runs the layer and reads h back
    # (MoELayer.forward_host overlaps step i's copies with the compute of
    # its neighbours; the layer runs its shared experts on a side stream
    # there, beside the copy streams)
    layer.overlap_shared = True
    e_steps = max(2, min(args.steps, 10))
    u_host = [u.cpu().pin_memory() for _ in range(2)]
    h_host = [torch.empty(bufs.h.shape, dtype=bufs.h.dtype).pin_memory()
              for _ in range(2)]
    ins = [u_host[i % 2] for i in range(e_steps)]
    outs = [h_host[i % 2] for i in range(e_steps)]
    layer.forward_host(ins[:2], outs[:2], update_bias=True, gamma=cfg.gamma)
    torch.cuda.synchronize()
    _barrier(ws)
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    layer.forward_host(ins, outs, update_bias=True, gamma=cfg.gamma)
    e1.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, dev)
    moe.get_device_error()
    out["e2e"] = {"value": ws * cfg.T / (e_ms / 1e3), "unit": "tokens/s",
                  "h2d_bytes_per_step": u.numel() * u.element_size(),
                  "d2h_bytes_per_step": bufs.h.numel() * bufs.h.element_size(),
                  "how": "MoELayer(overlap_shared=True).forward_host: "
                         "pinned-host batches, copies on their own streams "
                         "overlapping the neighbouring steps' compute"}
    layer.overlap_shared = False

    if args.graph:
        replay = layer.graph(u, update_bias=True, gamma=cfg.gamma)
        for _ in range(2):
            replay()
        torch.cuda.synchronize()
        _barrier(ws)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            replay()
        g1.record(stream)
        torch.cuda.synchronize()
        _barrier(ws)
        g_ms = max_over_ranks(g0.elapsed_time(g1), dev)
        moe.get_device_error()
        out["graph"] = {"value": whole_job_rate(ws, cfg.T, args.steps, g_ms),
                        "unit": "tokens/s", "ms_per_step": g_ms / args.steps,
                        "note": "the same step replayed from one CUDA graph"}

    if (headline and not args.no_backward and cfg.quant is None
            and cfg.dtype == "bf16" and cfg.d_ff % 128 == 0):
        out["backward"] = time_backward(args, cfg, layer, u, dev, ws, peaks)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, t, args.cpu_tokens)
    del layer, t, u, bufs, step
    _free()
    return out


def skew_block(args, cfg, moe, dev, ws, rank, local):
    """The skewed-load bias loop: cfg.steps steps, each with a fresh batch,
    every one followed by the +-gamma bias update.  Reports throughput and
    the max/mean expert load of every step."""
    peaks = _peaks()
    t = generate(cfg, dev)
    steps = cfg.steps
    us = [step_tokens(cfg, s, dev) for s in range(steps)]
    bias0 = t["b"].clone()
    layer = _new_layer(moe, cfg, t)
    bufs = layer.buffers(cfg.T)
    loads = torch.empty((steps, cfg.n_routed), dtype=torch.int32, device=dev)
    step = make_step(moe, cfg, layer, cfg.T)

    def restart():            # the warm-up ran on a scratch bias
        layer.bias.copy_(bias0)
        torch.cuda.synchronize()

    ms, call_ms, launches, clk = timed_steps(
        moe, step, us, steps, args.warmup, ws, local, dev,
        after_step=lambda i: loads[i].copy_(bufs.counts),
        before_timing=restart)
    c = loads.cpu().numpy().astype(np.float64)
    mean = cfg.T * cfg.top_k / cfg.n_routed
    mm = (c.max(axis=1) / mean).tolist()
    ms_step = ms / steps
    out = {"metric": METRIC, "value": whole_job_rate(ws, cfg.T, steps, ms),
           "unit": "tokens/s", "n_gpus": ws, "steps": steps,
           "warmup": max(3, args.warmup), "ms_per_step": ms_step,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16", "data": "synthetic",
           "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d,
                      "n_routed": cfg.n_routed, "top_k": cfg.top_k,
                      "n_shared": cfg.n_shared, "d_ff": cfg.d_ff,
                      "gamma": cfg.gamma, "zipf": cfg.zipf,
                      "parallelism": f"replicas x{ws}", "l2": L2_NOTE},
           "layer_tflops": layer_flops(cfg) / (ms_step / 1e3) / 1e12,
           "layer_frac_of_bf16_peak": layer_flops(cfg) / (ms_step / 1e3) /
           1e12 / peaks["bf16_tflops"],
           "roofline": ffn_roofline(cfg, c[-1], call_ms["expert_ffn"], peaks,
                                    "skew"),
           "load_max_over_mean": {"first": mm[0], "last": mm[-1],
                                  "per_step": [round(x, 3) for x in mm]},
           "clocks": clk,
           "gpu_launches": launches * ws,
           "per_call": call_rates(cfg, call_ms, bufs.h.element_size())}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, t, args.cpu_tokens, u=us[0])
    del layer, t, us, bufs, loads, step
    _free()
    return out


def run_ours(args, cfg):
    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import mixture_experts_layer_gemms_b300 as moe

    dev = torch.device("cuda", local)
    if cfg.steps > 1:
        line = skew_block(args, cfg, moe, dev, ws, rank, local)
    else:
        line = forward_block(args, cfg, moe, dev, ws, rank, local,
                             headline=True)
        if cfg.name == "v3_prefill" and not args.no_extra:
            line["decode"] = forward_block(args, get_config("v3_decode"), moe,
                                           dev, ws, rank, local,
                                           headline=False)
            line["skew"] = skew_block(args, get_config("skew"), moe, dev, ws,
                                      rank, local)
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
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the decode and skew blocks of the default line")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step replayed from one CUDA graph")
    ap.add_argument("--overlap-shared", action="store_true",
                    help="shared experts on a side stream in the timed step")
    ap.add_argument("--cpu-tokens", type=int, default=CPU_TOKENS,
                    help="tokens in the oracle's timed sample")
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
        args.no_extra = True
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
