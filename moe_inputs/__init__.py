"""Seeded synthetic inputs for the DeepSeekMoE layer forward.

This module is shared by the CPU oracle (``oracle/``) and the CUDA path
(``mixture_experts_layer_gemms_b300``).  It draws random numbers and nothing
else: it holds none of the layer's arithmetic (no affinity, no selection, no
FFN, no combine, no bias rule).  Both sides consume the tensors it returns.

Workload recipes (shapes, value distributions, seeds) follow the five layer
configurations this project measures:

====  ===========  ======  =====  ====  ==  ==  =====  =====  ===========
name  dtype        T       d      N_r   K   N_s I      seed   bias
====  ===========  ======  =====  ====  ==  ==  =====  =====  ===========
tiny  fp32         64      256    16    4   1   128    0      0
mid   bf16         4096    2048   64    6   2   1408   1      U(-.01,.01)
v3_prefill bf16    8192    7168   256   8   1   2048   2      0
v3_decode  bf16    128     7168   256   8   1   2048   3      0
skew  bf16         16384   7168   256   8   1   2048   4      0 (+50 steps)
====  ===========  ======  =====  ====  ==  ==  =====  =====  ===========

v3_prefill_fp8 and v3_decode_fp8 are v3_prefill and v3_decode (same seeds,
same tensors) run with e4m3 expert GEMMs.

Distributions: u ~ N(0,1); centroids e_i ~ N(0, 1/d); gate/up weights
~ N(0, 1/d); down weights ~ N(0, 1/I).  The skew workload scales centroid i
by (i+1)^-1.1 (largest at i = 0) so that routing starts imbalanced, and
draws a fresh u for every step.

Every value is sampled in fp32 and then rounded (round-to-nearest-even) to
the workload dtype; the bias is always fp32.  Draw order from one
``torch.Generator`` seeded with the workload seed: u, E, b, then for each
routed expert e the triple (W_gate[e], W_up[e], W_down[e]), then the same
triple for each shared expert.  Per-step inputs of the skew loop come from a
second generator seeded with ``seed * 1_000_003 + step + 1``.

Layouts (row-major): u[T,d], E[N_r,d], b[N_r] fp32, w_gate/w_up[N_r,I,d],
w_down[N_r,d,I], ws_gate/ws_up[N_s,I,d], ws_down[N_s,d,I].
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, Optional

import torch

__all__ = ["MoEConfig", "CONFIGS", "get_config", "generate", "step_tokens",
           "upstream_grad",
           "torch_dtype"]


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    n_routed: int
    top_k: int
    n_shared: int
    d_ff: int
    dtype: str            # "f32" or "bf16"
    seed: int
    bias: str = "zero"    # "zero" or "uniform" (U(-0.01, 0.01))
    zipf: Optional[float] = None   # centroid i scaled by (i+1)**-zipf
    steps: int = 1
    gamma: float = 1e-3
    quant: Optional[str] = None   # "fp8": e4m3 expert GEMMs (inputs unchanged)

    @property
    def assignments(self) -> int:
        return self.T * self.top_k

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


CONFIGS: Dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", T=64, d=256, n_routed=16, top_k=4, n_shared=1,
                      d_ff=128, dtype="f32", seed=0),
    "mid": MoEConfig("mid", T=4096, d=2048, n_routed=64, top_k=6, n_shared=2,
                     d_ff=1408, dtype="bf16", seed=1, bias="uniform"),
    "v3_prefill": MoEConfig("v3_prefill", T=8192, d=7168, n_routed=256,
                            top_k=8, n_shared=1, d_ff=2048, dtype="bf16",
                            seed=2),
    "v3_decode": MoEConfig("v3_decode", T=128, d=7168, n_routed=256, top_k=8,
                           n_shared=1, d_ff=2048, dtype="bf16", seed=3),
    "skew": MoEConfig("skew", T=16384, d=7168, n_routed=256, top_k=8,
                      n_shared=1, d_ff=2048, dtype="bf16", seed=4,
                      zipf=1.1, steps=50, gamma=1e-3),
}
# The two V3 workloads with e4m3 expert GEMMs: same inputs (same seeds),
# bf16 weights quantized by the library.
for _n in ("v3_prefill", "v3_decode"):
    CONFIGS[_n + "_fp8"] = CONFIGS[_n].with_(name=_n + "_fp8", quant="fp8")


def get_config(name: str) -> MoEConfig:
    return CONFIGS[name]


def torch_dtype(cfg: MoEConfig) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[cfg.dtype]


def _normal(gen, shape, std, dtype, device):
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def generate(cfg: MoEConfig, device="cpu", experts: bool = True,
             routed_experts: Optional[bool] = None) -> Dict[str, torch.Tensor]:
    """Draw one workload's tensors on ``device`` (seeded, deterministic).

    ``experts=False`` stops after (u, E, b) -- enough for routing-only work.
    The draw order is fixed, so a partial draw is a prefix of the full one.
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed)
    dt = torch_dtype(cfg)
    T, d, N, S, I = cfg.T, cfg.d, cfg.n_routed, cfg.n_shared, cfg.d_ff
    out: Dict[str, torch.Tensor] = {}
    out["u"] = _normal(gen, (T, d), 1.0, dt, dev)
    e32 = torch.randn((N, d), generator=gen, dtype=torch.float32, device=dev)
    e32.mul_(d ** -0.5)
    if cfg.zipf is not None:
        scale = torch.arange(1, N + 1, dtype=torch.float64) ** (-cfg.zipf)
        e32.mul_(scale.to(torch.float32).to(dev)[:, None])
    out["E"] = e32.to(dt)
    if cfg.bias == "uniform":
        b = torch.rand((N,), generator=gen, dtype=torch.float32, device=dev)
        out["b"] = b.mul_(0.02).sub_(0.01)
    else:
        out["b"] = torch.zeros((N,), dtype=torch.float32, device=dev)
    if routed_experts is None:
        routed_experts = experts
    if not experts:
        return out
    if routed_experts:
        wg = torch.empty((N, I, d), dtype=dt, device=dev)
        wu = torch.empty((N, I, d), dtype=dt, device=dev)
        wd = torch.empty((N, d, I), dtype=dt, device=dev)
        for e in range(N):
            wg[e] = _normal(gen, (I, d), d ** -0.5, dt, dev)
            wu[e] = _normal(gen, (I, d), d ** -0.5, dt, dev)
            wd[e] = _normal(gen, (d, I), I ** -0.5, dt, dev)
        out["w_gate"], out["w_up"], out["w_down"] = wg, wu, wd
    else:
        # keep the generator state identical to a full draw
        for e in range(N):
            for shape, std in (((I, d), d ** -0.5), ((I, d), d ** -0.5),
                               ((d, I), I ** -0.5)):
                torch.randn(shape, generator=gen, dtype=torch.float32,
                            device=dev)
    sg = torch.empty((S, I, d), dtype=dt, device=dev)
    su = torch.empty((S, I, d), dtype=dt, device=dev)
    sd = torch.empty((S, d, I), dtype=dt, device=dev)
    for s in range(S):
        sg[s] = _normal(gen, (I, d), d ** -0.5, dt, dev)
        su[s] = _normal(gen, (I, d), d ** -0.5, dt, dev)
        sd[s] = _normal(gen, (d, I), I ** -0.5, dt, dev)
    out["ws_gate"], out["ws_up"], out["ws_down"] = sg, su, sd
    return out


def step_tokens(cfg: MoEConfig, step: int, device="cpu") -> torch.Tensor:
    """Fresh layer input u[T,d] for step ``step`` of a multi-step workload."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed * 1_000_003 + step + 1)
    return _normal(gen, (cfg.T, cfg.d), 1.0, torch_dtype(cfg), dev)


def upstream_grad(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """Synthetic upstream gradient dh[T, d] ~ N(0, 1) for the backward pass,
    in the layer's dtype, from its own seeded stream."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed * 1_000_003 + 999_983)
    return _normal(gen, (cfg.T, cfg.d), 1.0, torch_dtype(cfg), dev)


def as_f64(t: torch.Tensor):
    """Exact widening of a bf16/fp32 tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
