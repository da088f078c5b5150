"""The benchmark's own code paths at small sizes, so that no block of the
JSON line can rot unnoticed: the oracle's reference arm on the CPU, and the
forward, decode-style and skewed bias-loop blocks on the GPU."""
import argparse
import io
import json
from contextlib import redirect_stdout

import pytest
import torch

import bench
from moe_inputs import get_config


def _args(**kw):
    a = dict(gpus=1, steps=2, warmup=3, impl="ours", workload="x",
             no_cpu_baseline=False, no_backward=True, no_extra=True,
             graph=False, overlap_shared=False, cpu_tokens=4, set=[])
    a.update(kw)
    return argparse.Namespace(**a)


def test_reference_arm_is_a_timed_sample():
    """--impl reference: every step is the oracle over the same seeded
    sample; the line says so, and its steps fit the run's own wall time."""
    cfg = get_config("tiny")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(_args(impl="reference", steps=3, warmup=1), cfg)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["extrapolated"] is True
    assert line["steps"] == 3 and line["tokens_per_step"] == 4
    assert line["ms_per_step"] * line["steps"] <= \
        1000.0 * line["sampled_wall_s"] + 1.0
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["value"] == pytest.approx(4 / (line["ms_per_step"] / 1e3))


def test_oracle_sample_is_seeded():
    cfg = get_config("mid").with_(T=300)
    from moe_inputs import generate
    t = generate(cfg, "cpu", experts=False)
    t.update({k: torch.zeros((cfg.n_shared, cfg.d_ff, cfg.d))
              for k in ("ws_gate", "ws_up")})
    t["ws_down"] = torch.zeros((cfg.n_shared, cfg.d, cfg.d_ff))
    a = bench.OracleSample(cfg, t, 10)
    b = bench.OracleSample(cfg, t, 10)
    assert (a.tokens == b.tokens).all() and a.tokens.size == 10
    assert (a.u64 == b.u64).all()


@pytest.mark.gpu
def test_forward_block_small():
    import mixture_experts_layer_gemms_b300 as moe
    cfg = get_config("v3_decode").with_(name="v3_decode+small", n_routed=32)
    out = bench.forward_block(_args(), cfg, moe, torch.device("cuda", 0), 1,
                              0, 0, headline=False)
    assert out["roofline"]["bound"] == "hbm"
    assert out["value"] > 0 and out["e2e"]["value"] > 0
    assert out["gpu_launches"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.gpu
def test_skew_block_small():
    import mixture_experts_layer_gemms_b300 as moe
    cfg = get_config("skew").with_(name="skew+small", T=512, steps=3,
                                   n_routed=32)
    out = bench.skew_block(_args(), cfg, moe, torch.device("cuda", 0), 1, 0,
                           0)
    assert out["steps"] == 3
    assert len(out["load_max_over_mean"]["per_step"]) == 3
    assert out["roofline"]["unit"] in ("TFLOP/s", "GB/s")
    assert out["cpu_baseline"]["value"] > 0
