"""GPU parity of the layer backward (moe_backward) against the fp64 oracle
(oracle/backward.py), on the GPU's own selection (checked first against the
oracle's routing rules).

Tolerance.  The pages fix no bar for gradients.  The relative part of the
forward's bar carries over unchanged: relative Frobenius error <= 5e-3.  The
absolute part is scaled to the tensor: max|err| <= max(2e-2, 1e-2 *
max|ref|).  A gradient entry is a sum over an expert's tokens (all T for the
shared experts) of products of bf16-rounded operands (dY = g dh, dA, H;
unit roundoff 2^-9), so its rounding error grows with the entries' scale.
A model of this path's rounding points on the CPU
(tests/test_backward_tolerance.py) stays below 0.5% of max|ref| at these
sizes; the bar is 1% (about 2.5 bf16 ulps at the largest entry).
Requires a B300 (sm_103a)."""
import numpy as np
import pytest
import torch

import oracle.backward as ob
import oracle.moe as om
from moe_inputs import as_f64, generate, get_config, upstream_grad
from parity_utils import (GRAD_REL_FRO as REL_FRO, check_routing, errors,
                          grad_max_abs, make_inputs)

pytestmark = pytest.mark.gpu


def grad_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    e = errors(got, ref)
    lim = grad_max_abs(ref)
    assert e["rel_fro"] <= REL_FRO and e["max_abs"] <= lim, (what, e, lim)
    return e


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_gemms_b300 as m
    return m


def _layer(moe, g, cfg):
    S = cfg.n_shared
    return moe.MoELayer(g["E"], g["b"].clone(), g["w_gate"], g["w_up"],
                        g["w_down"], g["ws_gate"] if S else None,
                        g["ws_up"] if S else None, g["ws_down"] if S else None,
                        top_k=cfg.top_k, h_dtype=torch.float32)


def _run(moe, cfg, grad_dtype=torch.float32, saved=False):
    g = make_inputs(cfg)
    dh = upstream_grad(cfg, "cpu").to("cuda")
    layer = _layer(moe, g, cfg)
    layer(g["u"], save_for_backward=saved)
    gr = layer.backward(g["u"], dh, grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    moe.get_device_error()
    return g, dh, layer, gr


BASE = dict(T=64, d=256, n_routed=16, top_k=4, n_shared=1, d_ff=128,
            dtype="bf16")
CASES = {
    "tiny_bf16_T64": ("tiny", dict(BASE)),
    "ragged_T37_S2_I256": ("tiny", dict(BASE, T=37, n_shared=2, d_ff=256)),
    # d % 256 != 0: the 128-column weight-gradient tiles
    "d384_T300": ("tiny", dict(BASE, T=300, d=384)),
    "no_shared_T500": ("tiny", dict(BASE, T=500, n_shared=0, d=512,
                                    d_ff=256)),
    "single_token": ("tiny", dict(BASE, T=1)),
    "mid_dims_T700": ("mid", dict(T=700)),
    # CTA-pair kernels (d, d_ff multiples of 256) under skewed centroids:
    # experts with 185..982 tokens -> multi-chunk Dgrad / recompute items
    # and Wgrad K loops of up to 16 blocks
    "skew_pair_T2000": ("tiny", dict(BASE, T=2000, d=512, d_ff=256,
                                     zipf=1.1)),
}


@pytest.mark.parametrize("saved", [False, True], ids=["recompute", "saved"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_parity(moe, case, saved):
    """Both ways to the SwiGLU backward: a and c recomputed by a gate/up
    GEMM, or saved (bf16) by the forward and used in the dH GEMM's
    epilogue."""
    name, over = CASES[case]
    cfg = get_config(name).with_(**over)
    g, dh, layer, gr = _run(moe, cfg, saved=saved)
    b = layer.buffers(cfg.T)
    idx = b.topk_idx.cpu().numpy()
    u64, E64, b64 = as_f64(g["u"]), as_f64(g["E"]), as_f64(g["b"])
    r = om.route(u64, E64, b64, cfg.top_k)
    check_routing(r, b64, idx, b.counts.cpu().numpy(), cfg.top_k)
    S = cfg.n_shared
    routed = lambda e: tuple(as_f64(g[k][e]) for k in
                             ("w_gate", "w_up", "w_down"))
    shared = [tuple(as_f64(g[k][s]) for k in ("ws_gate", "ws_up", "ws_down"))
              for s in range(S)]
    ref = ob.layer_backward(u64, E64, b64, cfg.top_k, routed, shared,
                            as_f64(dh), idx_override=idx)
    out = {}
    out["du"] = grad_close(gr["du"].cpu().numpy(), ref["du"], "du")
    out["dE"] = grad_close(gr["dE"].cpu().numpy(), ref["dE"], "dE")
    for j, k in enumerate(("dw_gate", "dw_up", "dw_down")):
        want = np.stack([ref["dW"][e][j] for e in range(cfg.n_routed)])
        out[k] = grad_close(gr[k].float().cpu().numpy(), want, k)
    for j, k in enumerate(("dws_gate", "dws_up", "dws_down")):
        if S:
            want = np.stack([ref["dWs"][s][j] for s in range(S)])
            out[k] = grad_close(gr[k].float().cpu().numpy(), want, k)
        else:
            assert k not in gr
    print(case, saved, out)


@pytest.mark.parametrize("over", [dict(BASE, T=64),
                                  dict(BASE, T=300, d=384, n_shared=2),
                                  dict(BASE, T=300, d=512, d_ff=256)],
                         ids=["small_groups", "single_sm", "cta_pair"])
def test_forward_saves_preactivations(moe, over):
    """save_for_backward leaves the forward's outputs bit for bit unchanged
    and stores a = x W_gate^T, c = x W_up^T of every slot (and of every
    token for the shared experts) as fp16, in the packed column order
    (blocks of 64 gate then 64 up values), within fp16 rounding (2^-11
    relative) of the fp64 products of the bf16 operands, plus the fp32
    accumulation's share."""
    cfg = get_config("tiny").with_(**over)
    g = make_inputs(cfg)
    plain, saving = _layer(moe, g, cfg), _layer(moe, g, cfg)
    h0 = plain(g["u"]).clone()
    h1 = saving(g["u"], save_for_backward=True)
    torch.cuda.synchronize()
    moe.get_device_error()
    assert torch.equal(h0, h1)
    b0, b1 = plain.buffers(cfg.T), saving.buffers(cfg.T)
    assert torch.equal(b0.y_perm, b1.y_perm)
    assert b1.saved
    I, S = cfg.d_ff, cfg.n_shared

    def unpack(act, n_units):
        a = act.float().cpu().numpy().reshape(act.shape[0], n_units // 64, 2,
                                              64)
        return (a[:, :, 0, :].reshape(act.shape[0], n_units),
                a[:, :, 1, :].reshape(act.shape[0], n_units))

    u64 = as_f64(g["u"])
    offs = b1.offsets.cpu().numpy()
    perm = b1.perm.cpu().numpy()
    ga, gc = unpack(b1.act[:offs[-1]], I)
    for e in range(cfg.n_routed):
        sl = slice(offs[e], offs[e + 1])
        x = u64[perm[sl]]
        for got, w in ((ga[sl], g["w_gate"][e]), (gc[sl], g["w_up"][e])):
            ref = x @ as_f64(w).T
            assert np.all(np.abs(got - ref) <= 2.0 ** -11 * np.abs(ref) + 1e-4)
    if S:
        sa, sc = unpack(b1.act_shared, S * I)
        for s_ in range(S):
            cols = slice(s_ * I, (s_ + 1) * I)
            for got, w in ((sa[:, cols], g["ws_gate"][s_]),
                           (sc[:, cols], g["ws_up"][s_])):
                ref = u64 @ as_f64(w).T
                assert np.all(np.abs(got - ref) <=
                              2.0 ** -11 * np.abs(ref) + 1e-4)


@pytest.mark.parametrize("over", [dict(BASE, T=200),
                                  dict(BASE, T=300, d=512, d_ff=256,
                                       n_shared=2)],
                         ids=["single_sm", "cta_pair"])
def test_backward_bf16_gradients(moe, over):
    """Weight gradients stored as bf16 are the fp32 gradients rounded once
    (to nearest even); du and dE do not depend on the gradient dtype."""
    cfg = get_config("tiny").with_(**over)
    g, dh, layer, g16 = _run(moe, cfg, torch.bfloat16)
    g16 = {k: v.float().clone() for k, v in g16.items()}
    g32 = layer.backward(g["u"], dh, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    moe.get_device_error()
    for k in ("dw_gate", "dw_up", "dw_down", "dws_gate", "dws_up", "dws_down"):
        a, w = g16[k], g32[k].float()
        # the bf16 store is the fp32 result rounded once
        assert torch.equal(a, w.to(torch.bfloat16).float()), k
    assert torch.equal(g16["du"], g32["du"]) and torch.equal(g16["dE"],
                                                              g32["dE"])


def test_backward_deterministic(moe):
    cfg = get_config("tiny").with_(**dict(BASE, T=300, n_shared=2))
    g, dh, layer, gr = _run(moe, cfg)
    first = {k: v.clone() for k, v in gr.items()}
    again = layer.backward(g["u"], dh)
    torch.cuda.synchronize()
    moe.get_device_error()
    for k in first:
        assert torch.equal(first[k], again[k]), k


@pytest.mark.parametrize("saved", [False, True], ids=["recompute", "saved"])
def test_backward_empty_batch(moe, saved):
    cfg = get_config("tiny").with_(**dict(BASE, T=0))
    g = make_inputs(cfg.with_(T=4))
    layer = _layer(moe, g, cfg)
    u = g["u"][:0]
    layer(u, save_for_backward=saved)
    gr = layer.backward(u, torch.empty((0, cfg.d), dtype=torch.bfloat16,
                                       device="cuda"))
    torch.cuda.synchronize()
    moe.get_device_error()
    assert gr["du"].shape == (0, cfg.d)
    for k, v in gr.items():
        assert not torch.any(v != 0), k


def test_backward_unused_experts_zero(moe):
    """Experts no token selected get exactly zero weight and centroid
    gradients (the bias makes experts 0..3 unreachable here)."""
    cfg = get_config("tiny").with_(**dict(BASE, T=40))
    g = make_inputs(cfg)
    g["b"] = g["b"].clone()
    g["b"][:4] = -100.0
    dh = upstream_grad(cfg, "cpu").to("cuda")
    layer = _layer(moe, g, cfg)
    layer(g["u"])
    gr = layer.backward(g["u"], dh)
    torch.cuda.synchronize()
    moe.get_device_error()
    assert int(layer.buffers(cfg.T).counts[:4].sum()) == 0
    for k in ("dw_gate", "dw_up", "dw_down"):
        assert not torch.any(gr[k][:4] != 0), k
    assert not torch.any(gr["dE"][:4] != 0)
    assert torch.any(gr["dw_down"][4:] != 0)


@pytest.mark.parametrize("saved", [False, True], ids=["recompute", "saved"])
def test_backward_full_v3_prefill_sampled(moe, saved):
    """V3 prefill shapes: du of sampled tokens, every weight and centroid
    gradient of two sampled experts, and sampled intermediate rows of the
    shared expert's gradients, each against the oracle."""
    cfg = get_config("v3_prefill")
    g = generate(cfg, "cuda")
    dh = upstream_grad(cfg, "cuda")
    layer = _layer(moe, g, cfg)
    layer(g["u"], save_for_backward=saved)
    gr = layer.backward(g["u"], dh)
    torch.cuda.synchronize()
    moe.get_device_error()
    b = layer.buffers(cfg.T)
    idx = b.topk_idx.cpu().numpy()
    gate = b.topk_gate.cpu().numpy().astype(np.float64)
    u64, E64, b64, dh64 = (as_f64(g["u"]), as_f64(g["E"]), as_f64(g["b"]),
                           as_f64(dh))
    rng = np.random.default_rng(0)
    rows = rng.choice(cfg.T, 3, replace=False)
    routed = lambda e: tuple(as_f64(g[k][e]) for k in
                             ("w_gate", "w_up", "w_down"))
    shared = [tuple(as_f64(g[k][0]) for k in ("ws_gate", "ws_up", "ws_down"))]
    ref = ob.layer_backward(u64, E64, b64, cfg.top_k, routed, shared, dh64,
                            idx_override=idx, tokens=rows)
    r = om.route(u64[rows], E64, b64, cfg.top_k)
    check_routing(r, b64, idx[rows], None, cfg.top_k)
    grad_close(gr["du"][rows].cpu().numpy(), ref["du"], "du rows")
    # gate from the oracle's affinity at the GPU's selection
    counts = b.counts.cpu().numpy()
    for e in rng.choice(np.nonzero(counts > 0)[0], 2, replace=False):
        rws = np.nonzero((idx == e).any(axis=1))[0]
        s_rows = om.affinity(u64[rws], E64)
        g_ref = np.zeros_like(gate)
        g_ref[rws] = np.take_along_axis(s_rows, idx[rws], axis=1)
        out = ob.expert_backward(u64, idx, g_ref, int(e), routed(int(e)),
                                 E64[e], dh64)
        grad_close(gr["dw_gate"][e].float().cpu().numpy(), out["dW_gate"],
                   f"dW_gate[{e}]")
        grad_close(gr["dw_up"][e].float().cpu().numpy(), out["dW_up"],
                   f"dW_up[{e}]")
        grad_close(gr["dw_down"][e].float().cpu().numpy(), out["dW_down"],
                   f"dW_down[{e}]")
        grad_close(gr["dE"][e].cpu().numpy(), out["dE"], f"dE[{e}]")
    # shared expert: the gradient rows (and down-projection columns) of
    # intermediate units R depend on those units' weights alone
    R = rng.choice(cfg.d_ff, 8, replace=False)
    wg, wu, wd = shared[0]
    _, dWg, dWu, dWd, _ = ob.swiglu_ffn_backward(u64, wg[R], wu[R], wd[:, R],
                                                 dh64)
    grad_close(gr["dws_gate"][0][R].float().cpu().numpy(), dWg, "dWs_gate")
    grad_close(gr["dws_up"][0][R].float().cpu().numpy(), dWu, "dWs_up")
    grad_close(gr["dws_down"][0][:, R].float().cpu().numpy(), dWd, "dWs_down")


def test_training_step_graph(moe):
    """Forward (saving its pre-activations) + bias update + backward captured
    as one CUDA graph replay the eager step bit for bit, on new tokens and
    gradients written into the captured buffers."""
    cfg = get_config("tiny").with_(**dict(BASE, T=300, d=512, d_ff=256))
    g = make_inputs(cfg)
    mk = lambda: _layer(moe, g, cfg)
    eager, graphed = mk(), mk()
    u = g["u"].clone()
    dh = upstream_grad(cfg, "cpu").to("cuda")
    run = graphed.graph(u, update_bias=True, dh=dh, grad_dtype=torch.bfloat16)
    gen = torch.Generator(device="cuda").manual_seed(11)
    for step in range(3):
        if step:
            u.copy_(torch.randn(u.shape, generator=gen, device="cuda")
                    .to(u.dtype))
            dh.copy_(torch.randn(dh.shape, generator=gen, device="cuda")
                     .to(dh.dtype))
        want_h = eager(u, update_bias=True, save_for_backward=True).clone()
        want = {k: v.clone() for k, v in
                eager.backward(u, dh, grad_dtype=torch.bfloat16).items()}
        h, grads = run()
        torch.cuda.synchronize()
        moe.get_device_error()
        assert torch.equal(want_h, h), step
        for k in want:
            assert torch.equal(want[k], grads[k]), (step, k)
        assert torch.equal(eager.bias, graphed.bias), step


def test_backward_after_group_limited_routing(moe):
    """The backward takes the forward's selection as given: after
    group-limited routing (4 groups, best 2 kept) its gradients match the
    oracle's on that selection."""
    cfg = get_config("tiny").with_(**dict(BASE, T=300, d=512, d_ff=256))
    g = make_inputs(cfg)
    dh = upstream_grad(cfg, "cpu").to("cuda")
    S = cfg.n_shared
    layer = moe.MoELayer(g["E"], g["b"].clone(), g["w_gate"], g["w_up"],
                         g["w_down"], g["ws_gate"], g["ws_up"], g["ws_down"],
                         top_k=cfg.top_k, h_dtype=torch.float32, n_groups=4,
                         topk_groups=2)
    layer(g["u"])
    gr = layer.backward(g["u"], dh)
    torch.cuda.synchronize()
    moe.get_device_error()
    b = layer.buffers(cfg.T)
    idx = b.topk_idx.cpu().numpy()
    u64, E64, b64 = as_f64(g["u"]), as_f64(g["E"]), as_f64(g["b"])
    r = om.route(u64, E64, b64, cfg.top_k, groups=(4, 2))
    check_routing(r, b64, idx, b.counts.cpu().numpy(), cfg.top_k,
                  groups=(4, 2))
    routed = lambda e: tuple(as_f64(g[k][e]) for k in
                             ("w_gate", "w_up", "w_down"))
    shared = [tuple(as_f64(g[k][s]) for k in ("ws_gate", "ws_up", "ws_down"))
              for s in range(S)]
    ref = ob.layer_backward(u64, E64, b64, cfg.top_k, routed, shared,
                            as_f64(dh), idx_override=idx)
    grad_close(gr["du"].cpu().numpy(), ref["du"], "du")
    grad_close(gr["dE"].cpu().numpy(), ref["dE"], "dE")
    for j, k in enumerate(("dw_gate", "dw_up", "dw_down")):
        want = np.stack([ref["dW"][e][j] for e in range(cfg.n_routed)])
        grad_close(gr[k].float().cpu().numpy(), want, k)
