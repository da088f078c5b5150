"""GPU parity: every C-ABI call, and the whole layer, against the CPU fp64
oracle on the same seeded inputs.  Requires a B300 (sm_103a)."""
import numpy as np
import pytest
import torch

import oracle.moe as om
from moe_inputs import as_f64, generate, get_config, step_tokens
from parity_utils import (assert_close, check_routing, errors,
                          half_ulp_bf16, make_inputs, oracle_weights)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_gemms_b300 as m
    return m


def _shape(moe, cfg, T=None):
    return moe.make_shape(cfg.T if T is None else T, cfg.d, cfg.n_routed,
                          cfg.top_k, cfg.n_shared, cfg.d_ff, cfg.dtype)


def _ws(moe, sh):
    return torch.empty(max(moe.workspace_size(sh), 256), dtype=torch.uint8,
                       device="cuda")


def _route_gpu(moe, cfg, u, E, b, groups=None):
    T, K, N = u.shape[0], cfg.top_k, cfg.n_routed
    sh = _shape(moe, cfg, T)
    idx = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    gate = torch.empty((T, K), dtype=torch.float32, device="cuda")
    counts = torch.full((N,), -7, dtype=torch.int32, device="cuda")
    if groups is None:
        moe.route(sh, u, E, b, idx, gate, counts, _ws(moe, sh))
    else:
        moe.route_grouped(sh, groups[0], groups[1], u, E, b, idx, gate,
                          counts, _ws(moe, sh))
    moe.get_device_error()
    return idx.cpu().numpy(), gate.cpu().numpy(), counts.cpu().numpy()


# ----------------------------------------------------------------- route --
# Gate tolerance.  z = u.e is accumulated in fp32 by the tensor core over
# d/16 MMA steps split across (at least) two accumulators; with up to one
# ulp of drift per step, |dz| <= (d/16/2) * 2^-23 * |z| = 2.7e-5 |z| at
# d = 7168, and |ds| = s(1-s) |dz| <= max_z s(1-s) |z| * 2.7e-5 < 1.2e-5.
GATE_ATOL = 1.2e-5
ROUTE_CASES = {
    "tiny_f32": ("tiny", {}),
    "mid_bf16": ("mid", {}),
    "v3_ragged_T300": ("v3_prefill", {"T": 300}),
    "mid_T1": ("mid", {"T": 1}),
    "skew_T1024": ("skew", {"T": 1024}),
}


@pytest.mark.parametrize("case", sorted(ROUTE_CASES))
def test_route_parity(moe, case):
    name, over = ROUTE_CASES[case]
    cfg = get_config(name).with_(**over)
    t = generate(cfg, "cpu", experts=False)
    u, E, b = (t[k].cuda() for k in ("u", "E", "b"))
    idx, gate, counts = _route_gpu(moe, cfg, u, E, b)
    b64 = as_f64(t["b"])
    r = om.route(as_f64(t["u"]), as_f64(t["E"]), b64, cfg.top_k)
    near = check_routing(r, b64, idx, counts, cfg.top_k)
    s_at = np.take_along_axis(r["s"], idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(gate, s_at, rtol=0, atol=GATE_ATOL)
    assert near <= max(2, cfg.T // 50) or cfg.zipf is not None, near


def test_route_full_v3_prefill(moe):
    """Routing of the full 8192-token prefill batch (all tokens checked)."""
    cfg = get_config("v3_prefill")
    t = generate(cfg, "cuda", experts=False)
    idx, gate, counts = _route_gpu(moe, cfg, t["u"], t["E"], t["b"])
    b64 = as_f64(t["b"])
    r = om.route(as_f64(t["u"]), as_f64(t["E"]), b64, cfg.top_k)
    check_routing(r, b64, idx, counts, cfg.top_k)
    assert counts.sum() == cfg.T * cfg.top_k


def test_route_full_unsplit_v3_dims(moe):
    """V3 dimensions with T = 16384 (the skewed-bias loop's batch): 128
    token tiles x 2 would exceed one wave of the GPU's SMs, so the router
    runs unsplit (one CTA per tile over all of d = 7168, sigmoid in its
    first epilogue branch).  All tokens checked, as at T = 8192."""
    cfg = get_config("v3_prefill").with_(T=16384)
    t = generate(cfg, "cuda", experts=False)
    idx, gate, counts = _route_gpu(moe, cfg, t["u"], t["E"], t["b"])
    b64 = as_f64(t["b"])
    r = om.route(as_f64(t["u"]), as_f64(t["E"]), b64, cfg.top_k)
    check_routing(r, b64, idx, counts, cfg.top_k)
    assert counts.sum() == cfg.T * cfg.top_k


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_route_ties_lowest_index(moe, dtype):
    """E = 0 makes every affinity exactly 1/2: selection follows the bias,
    and equal biased scores go to the lower index."""
    cfg = get_config("tiny").with_(T=200, dtype=dtype, n_routed=32,
                                   top_k=5)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    u = torch.randn((cfg.T, cfg.d), generator=torch.Generator().manual_seed(0)
                    ).to(dt).cuda()
    E = torch.zeros((cfg.n_routed, cfg.d), dtype=dt, device="cuda")
    b = torch.zeros(cfg.n_routed, dtype=torch.float32, device="cuda")
    idx, gate, counts = _route_gpu(moe, cfg, u, E, b)
    assert (idx == np.arange(5)[None, :]).all()
    assert (gate == 0.5).all()
    bias = np.zeros(32, np.float32)
    bias[[7, 3, 20, 9]] = [0.25, 0.25, 0.125, 0.25]   # 3 and 7, 9 tie
    idx, gate, counts = _route_gpu(moe, cfg, u, E, torch.from_numpy(bias).cuda())
    assert (idx == np.array([3, 7, 9, 20, 0])[None, :]).all()
    assert (gate == 0.5).all()          # the gate is s, never s + b
    assert counts[[0, 3, 7, 9, 20]].tolist() == [200] * 5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_route_empty_batch(moe, dtype):
    cfg = get_config("tiny").with_(T=0, dtype=dtype)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    E = torch.randn((cfg.n_routed, cfg.d)).to(dt).cuda()
    b = torch.zeros(cfg.n_routed, device="cuda")
    sh = _shape(moe, cfg)
    counts = torch.full((cfg.n_routed,), 5, dtype=torch.int32, device="cuda")
    moe.route(sh, None, E, b, None, None, counts, _ws(moe, sh))
    moe.get_device_error()
    assert counts.cpu().tolist() == [0] * cfg.n_routed


# -------------------------------------------------------- grouped route --
GROUP_CASES = {
    "tiny_f32_G4_M2": ("tiny", {}, (4, 2)),
    "mid_bf16_G8_M4": ("mid", {}, (8, 4)),
    "mid_bf16_G32_M1": ("mid", {"top_k": 1}, (32, 1)),
    "v3_T300_G8_M4": ("v3_prefill", {"T": 300}, (8, 4)),
    "v3_T300_G64_M8": ("v3_prefill", {"T": 300}, (64, 8)),
    "skew_T1024_G8_M3": ("skew", {"T": 1024}, (8, 3)),
}


@pytest.mark.parametrize("case", sorted(GROUP_CASES))
def test_route_grouped_parity(moe, case):
    name, over, groups = GROUP_CASES[case]
    cfg = get_config(name).with_(**over)
    t = generate(cfg, "cpu", experts=False)
    u, E, b = (t[k].cuda() for k in ("u", "E", "b"))
    idx, gate, counts = _route_gpu(moe, cfg, u, E, b, groups)
    b64 = as_f64(t["b"])
    r = om.route(as_f64(t["u"]), as_f64(t["E"]), b64, cfg.top_k, groups)
    near = check_routing(r, b64, idx, counts, cfg.top_k, groups=groups)
    s_at = np.take_along_axis(r["s"], idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(gate, s_at, rtol=0, atol=GATE_ATOL)
    # every token's experts come from at most M groups
    per = cfg.n_routed // groups[0]
    used = [len(set((row // per).tolist())) for row in idx]
    assert max(used) <= groups[1]
    assert near <= max(2, cfg.T // 50) or cfg.zipf is not None, near


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_route_grouped_all_groups_is_plain(moe, dtype):
    """Keeping every group (M = G) is plain routing, bit for bit."""
    cfg = get_config("mid").with_(dtype=dtype, T=500)
    t = generate(cfg, "cpu", experts=False)
    u, E, b = (t[k].cuda() for k in ("u", "E", "b"))
    plain = _route_gpu(moe, cfg, u, E, b)
    for groups in ((1, 1), (8, 8)):
        got = _route_gpu(moe, cfg, u, E, b, groups)
        for x, y in zip(plain, got):
            assert x.tobytes() == y.tobytes(), groups


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_route_grouped_ties(moe, dtype):
    """E = 0 makes every affinity 1/2, so the bias alone decides.  32
    experts in 4 groups of 8; biases put groups 1 and 3 level on top."""
    cfg = get_config("tiny").with_(T=130, dtype=dtype, n_routed=32, top_k=4)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    u = torch.randn((cfg.T, cfg.d), generator=torch.Generator().manual_seed(1)
                    ).to(dt).cuda()
    E = torch.zeros((cfg.n_routed, cfg.d), dtype=dt, device="cuda")
    bias = np.zeros(32, np.float32)
    bias[[12, 30, 20]] = [0.25, 0.25, 0.125]
    bd = torch.from_numpy(bias).cuda()
    want = {(4, 2): [12, 30, 8, 9],       # groups 1, 3 kept
            (4, 1): [12, 8, 9, 10],       # tie 1 vs 3 -> group 1
            (4, 4): [12, 30, 20, 0]}      # plain routing
    for groups, exp in want.items():
        idx, gate, counts = _route_gpu(moe, cfg, u, E, bd, groups)
        assert (idx == np.array(exp)[None, :]).all(), (groups, idx[0])
        assert (gate == 0.5).all()
        assert counts[exp].tolist() == [cfg.T] * 4
        r = om.route(np.zeros((1, cfg.d)), np.zeros((32, cfg.d)),
                     bias.astype(np.float64), 4, groups)
        assert r["idx"][0].tolist() == exp


def test_route_grouped_full_v3_prefill(moe):
    """8192 tokens, 256 experts in 8 groups, 4 kept, top-8."""
    cfg = get_config("v3_prefill")
    t = generate(cfg, "cuda", experts=False)
    idx, gate, counts = _route_gpu(moe, cfg, t["u"], t["E"], t["b"], (8, 4))
    b64 = as_f64(t["b"])
    r = om.route(as_f64(t["u"]), as_f64(t["E"]), b64, cfg.top_k, (8, 4))
    check_routing(r, b64, idx, counts, cfg.top_k, groups=(8, 4))
    assert counts.sum() == cfg.T * cfg.top_k


@pytest.mark.parametrize("name,over,groups", [
    ("mid", {}, (8, 2)),
    ("v3_prefill", {"T": 200, "n_routed": 64}, (8, 4)),
])
def test_layer_grouped_parity(moe, name, over, groups):
    cfg = get_config(name).with_(**over)
    t, g = _layer_inputs(cfg)
    e, near, _ = _layer_check(moe, cfg, t, g, groups=groups)
    print(name, groups, e, "near-ties", near)


# ----------------------------------------------------------- update_bias --
def test_update_bias_bit_exact(moe):
    rng = np.random.default_rng(3)
    N, TK = 256, 8192 * 8
    b = rng.uniform(-0.05, 0.05, N).astype(np.float32)
    counts = rng.multinomial(TK, np.ones(N) / N).astype(np.int32)
    counts[:4] = TK // N            # exactly balanced: unchanged
    bd = torch.from_numpy(b).cuda()
    for gamma in (1e-3, 2.0 ** -10, 0.0):
        want = om.update_bias(bd.cpu().numpy(), counts, TK, gamma)
        moe.update_bias(N, torch.from_numpy(counts).cuda(), TK, gamma, bd)
        got = bd.cpu().numpy()
        assert got.tobytes() == want.tobytes(), gamma


def test_update_bias_golden(moe):
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "bias_update_worked_example.json")))
    c = g["cases"]["from_one"]
    b = np.array([int(x, 16) for x in c["b_hex"]], np.uint32).view(np.float32)
    bd = torch.from_numpy(b.copy()).cuda()
    moe.update_bias(g["N"], torch.tensor(g["counts"], dtype=torch.int32,
                                         device="cuda"),
                    g["total_assign"], c["gamma"], bd)
    got = [f"0x{v:08X}" for v in bd.cpu().numpy().view(np.uint32).tolist()]
    assert got == c["expected_hex"]


# --------------------------------------------------------------- permute --
@pytest.mark.parametrize("T,N,K,dtype", [(64, 16, 4, "f32"), (300, 64, 6, "bf16"),
                                         (1000, 256, 8, "bf16"),
                                         (129, 16, 16, "bf16")])
def test_permute_exact(moe, T, N, K, dtype):
    rng = np.random.default_rng(T)
    idx = np.stack([rng.permutation(N)[:K] for _ in range(T)]).astype(np.int32)
    counts = np.bincount(idx.ravel(), minlength=N).astype(np.int32)
    off, perm, inv = om.permute(idx, counts)
    cfg = get_config("tiny").with_(T=T, n_routed=N, top_k=K, dtype=dtype,
                                   d=256)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    u = torch.randn((T, cfg.d)).to(dt).cuda()
    sh = _shape(moe, cfg)
    A = T * K
    o_d = torch.empty(N + 1, dtype=torch.int32, device="cuda")
    p_d = torch.empty(A, dtype=torch.int32, device="cuda")
    i_d = torch.empty((T, K), dtype=torch.int32, device="cuda")
    x_d = torch.empty((A, cfg.d), dtype=dt, device="cuda")
    moe.permute(sh, u, torch.from_numpy(idx).cuda(),
                torch.from_numpy(counts).cuda(), o_d, p_d, i_d, x_d,
                _ws(moe, sh))
    moe.get_device_error()
    np.testing.assert_array_equal(o_d.cpu().numpy(), off)
    np.testing.assert_array_equal(p_d.cpu().numpy(), perm)
    np.testing.assert_array_equal(i_d.cpu().numpy(), inv)
    assert torch.equal(x_d.cpu(), u.cpu()[torch.from_numpy(perm)])


# ------------------------------------------------------------ expert_ffn --
FFN_CASES = {
    "tiny_f32": ("tiny", {}),
    "mid_bf16_T1024": ("mid", {"T": 1024}),
    "v3dims_T96": ("v3_prefill", {"T": 96, "n_routed": 32}),
    "no_shared_bf16": ("mid", {"T": 256, "n_shared": 0}),
}


def _layer_inputs(cfg):
    g = make_inputs(cfg)      # device tensors; the oracle widens copies
    return g, g


@pytest.mark.parametrize("case", sorted(FFN_CASES))
def test_expert_ffn_parity(moe, case):
    name, over = FFN_CASES[case]
    cfg = get_config(name).with_(**over)
    t, g = _layer_inputs(cfg)
    T, K, N, d = cfg.T, cfg.top_k, cfg.n_routed, cfg.d
    u64 = as_f64(t["u"])
    r = om.route(u64, as_f64(t["E"]), as_f64(t["b"]), K)
    off, perm, inv = om.permute(r["idx"], r["counts"])
    routed, shared = oracle_weights(t)
    y_ref, ys_ref = om.expert_ffn(u64[perm], off, routed, u64, shared)
    layer = moe.MoELayer(g["E"], g["b"], g["w_gate"], g["w_up"], g["w_down"],
                         g["ws_gate"] if cfg.n_shared else None,
                         g["ws_up"] if cfg.n_shared else None,
                         g["ws_down"] if cfg.n_shared else None, top_k=K)
    sh = layer.shape(T)
    b = layer.buffers(T)
    x_perm = g["u"][torch.from_numpy(perm).cuda()].contiguous()
    moe.expert_ffn(sh, x_perm, torch.from_numpy(off.astype(np.int32)).cuda(),
                   layer.w_gu, layer.w_down, g["u"], layer.ws_gu,
                   layer.ws_down, b.y_perm, b.y_shared, b.workspace)
    moe.get_device_error()
    assert_close(b.y_perm[:T * K].float().cpu().numpy(), y_ref,
                 what="y_perm")
    if cfg.n_shared:
        assert_close(b.y_shared.float().cpu().numpy(), ys_ref, what="y_shared")


def test_expert_ffn_rejects_bad_offsets(moe):
    """A device-side check: offsets past the buffer are refused without any
    out-of-range access, and reported as MOE_ERR_DEVICE_CHECK."""
    cfg = get_config("mid").with_(T=64, n_shared=0)
    t, g = _layer_inputs(cfg)
    layer = moe.MoELayer(g["E"], g["b"], g["w_gate"], g["w_up"], g["w_down"],
                         top_k=cfg.top_k)
    sh = layer.shape(cfg.T)
    b = layer.buffers(cfg.T)
    off = torch.arange(cfg.n_routed + 1, dtype=torch.int32,
                       device="cuda") * 1000
    moe.expert_ffn(sh, b.x_perm, off, layer.w_gu, layer.w_down, None, None,
                   None, b.y_perm, None, b.workspace)
    with pytest.raises(moe.MoEError) as ei:
        moe.get_device_error()
    assert ei.value.status == 6
    moe.get_device_error()   # cleared


# --------------------------------------------------------------- combine --
@pytest.mark.parametrize("dtype,hdt", [("f32", torch.float32),
                                       ("bf16", torch.float32),
                                       ("bf16", torch.bfloat16)])
def test_combine_parity(moe, dtype, hdt):
    T, N, K, d, S = 333, 64, 6, 1024, 1
    rng = np.random.default_rng(9)
    idx = np.stack([rng.permutation(N)[:K] for _ in range(T)])
    counts = np.bincount(idx.ravel(), minlength=N)
    off, perm, inv = om.permute(idx, counts)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    gen = torch.Generator().manual_seed(1)
    ydt = torch.float16 if dtype == "bf16" else torch.float32
    u = torch.randn((T, d), generator=gen).to(dt)
    y = torch.randn((T * K, d), generator=gen).to(ydt)
    ys = torch.randn((T, d), generator=gen).to(ydt)
    gate = torch.rand((T, K), generator=gen)
    ref = om.combine(as_f64(u), as_f64(y), as_f64(ys), inv, as_f64(gate))
    cfg = get_config("tiny").with_(T=T, n_routed=N, top_k=K, d=d, n_shared=S,
                                   dtype=dtype)
    h = torch.empty((T, d), dtype=hdt, device="cuda")
    moe.combine(_shape(moe, cfg), u.cuda(), y.cuda(), ys.cuda(),
                torch.from_numpy(inv.astype(np.int32)).cuda(), gate.cuda(), h)
    moe.get_device_error()
    got = h.float().cpu().numpy()
    if hdt == torch.float32:
        e = errors(got, ref)
        assert e["max_abs"] <= 1e-5 * max(1.0, np.abs(ref).max()), e
    else:   # one rounding of the fp32 sum to bf16: at most half an ulp
        assert np.all(np.abs(got - ref) <= half_ulp_bf16(ref) * 1.001 + 1e-5)


# ------------------------------------------------------- the whole layer --
def _layer_check(moe, cfg, t, g, tokens=None, h_dtype=torch.float32,
                 groups=None):
    G, M = (1, 1) if groups is None else groups
    layer = moe.MoELayer(g["E"], g["b"].clone(), g["w_gate"], g["w_up"],
                         g["w_down"],
                         g["ws_gate"] if cfg.n_shared else None,
                         g["ws_up"] if cfg.n_shared else None,
                         g["ws_down"] if cfg.n_shared else None,
                         top_k=cfg.top_k, h_dtype=h_dtype, n_groups=G,
                         topk_groups=M)
    h = layer(g["u"])
    torch.cuda.synchronize()
    moe.get_device_error()
    b = layer.buffers(cfg.T)
    idx = b.topk_idx.cpu().numpy()
    counts = b.counts.cpu().numpy()
    routed, shared = oracle_weights(t)
    b64 = as_f64(t["b"])
    sel = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    u64 = as_f64(t["u"][torch.from_numpy(sel).to(t["u"].device)])
    r = om.route(u64, as_f64(t["E"]), b64, cfg.top_k, groups)
    near = check_routing(r, b64, idx[sel], None, cfg.top_k, groups=groups)
    assert counts.sum() == cfg.T * cfg.top_k
    np.testing.assert_array_equal(
        counts, np.bincount(idx.ravel(), minlength=cfg.n_routed))
    # h against the definition, on the GPU's selection (identical to the
    # oracle's except on near-tied tokens)
    h_ref, _ = om.layer_forward(u64, as_f64(t["E"]), b64, cfg.top_k, routed,
                                shared, idx_override=idx[sel])
    got = h.float().cpu().numpy()[sel]
    if h_dtype == torch.bfloat16:
        # bf16 output: the bar is 2e-2 plus the half ulp of the final rounding
        bound = 2e-2 + half_ulp_bf16(h_ref)
        assert np.all(np.abs(got - h_ref) <= bound), \
            np.abs(got - h_ref).max()
        e = errors(got, h_ref, base=u64)
    else:
        e = assert_close(got, h_ref, base=u64, what=cfg.name)
    return e, near, layer


LAYER_CASES = {
    "tiny_f32": ("tiny", {}),
    "mid_bf16": ("mid", {}),
    "dense_K_eq_N": ("mid", {"T": 100, "n_routed": 16, "top_k": 16, "d": 256,
                             "d_ff": 128}),
    "v3dims_T200_N64": ("v3_prefill", {"T": 200, "n_routed": 64}),
    "ragged_T37": ("mid", {"T": 37}),
    # d % 256 != 0 and I % 128 != 0: the single-SM grouped GEMM
    "single_sm_d384_I192": ("mid", {"T": 400, "d": 384, "d_ff": 192,
                                    "n_routed": 16, "top_k": 4}),
}


@pytest.mark.parametrize("case", sorted(LAYER_CASES))
def test_layer_parity(moe, case):
    name, over = LAYER_CASES[case]
    cfg = get_config(name).with_(**over)
    t, g = _layer_inputs(cfg)
    e, near, _ = _layer_check(moe, cfg, t, g)
    print(case, e, "near-ties", near)


def test_layer_skewed_multi_chunk(moe):
    """A bias that sends every token to the same K experts: groups of T rows
    span several 256-token chunks (and the rest of the experts are empty)."""
    cfg = get_config("mid").with_(T=600, n_shared=1)
    t, g = _layer_inputs(cfg)
    b = torch.zeros(cfg.n_routed)
    b[[5, 17, 33, 40, 41, 63]] = 2.0
    g["b"] = b.cuda()
    e, near, layer = _layer_check(moe, cfg, t, g)
    counts = layer.buffers(cfg.T).counts.cpu().numpy()
    assert sorted(np.nonzero(counts)[0].tolist()) == [5, 17, 33, 40, 41, 63]


def test_layer_small_groups_path(moe):
    """Average group below 48 tokens selects the 32-token chunk kernel; a
    skewed bias gives one expert many chunks of it."""
    cfg = get_config("mid").with_(T=300, n_routed=64, top_k=2, n_shared=1)
    t, g = _layer_inputs(cfg)
    b = torch.zeros(cfg.n_routed)
    b[11] = 2.0
    g["b"] = b.cuda()
    e, near, layer = _layer_check(moe, cfg, t, g)
    assert layer.buffers(cfg.T).counts.cpu().numpy()[11] == cfg.T


def test_layer_bf16_output(moe):
    cfg = get_config("mid").with_(T=256)
    t, g = _layer_inputs(cfg)
    _layer_check(moe, cfg, t, g, h_dtype=torch.bfloat16)


def test_layer_empty_batch(moe):
    cfg = get_config("mid").with_(T=0)
    t, g = _layer_inputs(cfg)
    layer = moe.MoELayer(g["E"], g["b"], g["w_gate"], g["w_up"], g["w_down"],
                         g["ws_gate"], g["ws_up"], g["ws_down"],
                         top_k=cfg.top_k)
    h = layer(g["u"])
    torch.cuda.synchronize()
    moe.get_device_error()
    assert h.shape == (0, cfg.d)
    assert layer.buffers(0).offsets.cpu().tolist() == [0] * (cfg.n_routed + 1)


def test_layer_deterministic(moe):
    cfg = get_config("mid").with_(T=512)
    t, g = _layer_inputs(cfg)
    layer = moe.MoELayer(g["E"], g["b"], g["w_gate"], g["w_up"], g["w_down"],
                         g["ws_gate"], g["ws_up"], g["ws_down"],
                         top_k=cfg.top_k)
    h1 = layer(g["u"]).clone()
    h2 = layer(g["u"]).clone()
    assert torch.equal(h1, h2)


# ------------------------------------------- full sizes, sampled outputs --
def _full_layer(moe, cfg, g, h_dtype=torch.float32):
    layer = moe.MoELayer(g["E"], g["b"].clone(), g["w_gate"], g["w_up"],
                         g["w_down"], g["ws_gate"], g["ws_up"], g["ws_down"],
                         top_k=cfg.top_k, h_dtype=h_dtype)
    h = layer(g["u"])
    torch.cuda.synchronize()
    moe.get_device_error()
    return layer, h


def _check_h_rows(cfg, g, idx, h, rows):
    """h on the given token rows against the definition, on the GPU's
    selection (identical to the oracle's away from near-ties)."""
    routed, shared = oracle_weights(g)
    b64 = as_f64(g["b"])
    sel = torch.from_numpy(np.asarray(rows)).to(g["u"].device)
    u64 = as_f64(g["u"][sel])
    h_ref, _ = om.layer_forward(u64, as_f64(g["E"]), b64, cfg.top_k, routed,
                                shared, idx_override=idx[rows])
    got = h[sel].float().cpu().numpy()
    return assert_close(got, h_ref, base=u64, what=cfg.name)


def test_layer_full_v3_prefill(moe):
    """The full V3 prefill layer (T = 8192) in the benchmark's launch
    configuration (CTA-pair grouped GEMM, d = 7168, d_ff = 2048).

    * routing of every token against the oracle;
    * h on >= 200 tokens: for every expert a seeded token of its LAST
      token chunk and the token in its last slot (so the last chunk of every
      expert's items, ragged tails included, reaches the check), plus a
      seeded sample and the batch's last token;
    * y_perm element by element on every row of the four most loaded
      experts (each over 256 tokens, so split into several chunks)."""
    cfg = get_config("v3_prefill")
    g = generate(cfg, "cuda")
    layer, h = _full_layer(moe, cfg, g)
    b = layer.buffers(cfg.T)
    idx = b.topk_idx.cpu().numpy()
    counts = b.counts.cpu().numpy()
    off = b.offsets.cpu().numpy().astype(np.int64)
    perm = b.perm.cpu().numpy().astype(np.int64)
    b64 = as_f64(g["b"])
    r = om.route(as_f64(g["u"]), as_f64(g["E"]), b64, cfg.top_k)
    near = check_routing(r, b64, idx, counts, cfg.top_k)
    # the permutation is the oracle's on the GPU's own selection
    o_off, o_perm, _ = om.permute(idx, counts)
    np.testing.assert_array_equal(off, o_off)
    np.testing.assert_array_equal(perm, o_perm)
    # the grouped GEMM splits an expert's m rows into ceil(m / 256) chunks of
    # equal size (rounded up to 16); take a seeded row of every expert's
    # last chunk, and the expert's very last row (the ragged tail)
    rng = np.random.default_rng(cfg.seed)
    pick = []
    for e in range(cfg.n_routed):
        m = int(counts[e])
        if m == 0:
            continue
        ce = -(-m // 256)
        sz = (-(-m // ce) + 15) // 16 * 16
        lo = int(off[e]) + (ce - 1) * sz
        pick += [perm[rng.integers(lo, int(off[e + 1]))], perm[off[e + 1] - 1]]
    rows = np.unique(np.concatenate([pick, rng.choice(cfg.T, 32, False),
                                     [cfg.T - 1]]))
    assert rows.size >= 200, rows.size
    e_h = _check_h_rows(cfg, g, idx, h, rows)
    # y_perm of multi-chunk experts, every row
    big = np.argsort(-counts, kind="stable")[:4]
    assert counts[big].min() > 256, counts[big]
    y = b.y_perm
    errs = []
    for e in big.tolist():
        lo, hi = int(off[e]), int(off[e + 1])
        x = as_f64(g["u"][torch.from_numpy(perm[lo:hi]).cuda()])
        w = tuple(as_f64(g[k][e]) for k in ("w_gate", "w_up", "w_down"))
        ref = om.swiglu_ffn(x, *w)
        errs.append(assert_close(y[lo:hi].float().cpu().numpy(), ref,
                                 what=f"y_perm expert {e} ({hi - lo} rows)"))
    print("v3_prefill h", rows.size, "tokens", e_h, "near-ties", near,
          "y_perm", errs)
    del layer, g, h
    torch.cuda.empty_cache()


def test_layer_full_v3_decode(moe):
    """The full V3 decode layer (T = 128, the weight-streaming kernel):
    routing and h of every token against the oracle."""
    cfg = get_config("v3_decode")
    g = generate(cfg, "cuda")
    layer, h = _full_layer(moe, cfg, g)
    b = layer.buffers(cfg.T)
    idx = b.topk_idx.cpu().numpy()
    b64 = as_f64(g["b"])
    r = om.route(as_f64(g["u"]), as_f64(g["E"]), b64, cfg.top_k)
    near = check_routing(r, b64, idx, b.counts.cpu().numpy(), cfg.top_k)
    e = _check_h_rows(cfg, g, idx, h, np.arange(cfg.T))
    print("v3_decode", e, "near-ties", near)
    del layer, g, h
    torch.cuda.empty_cache()


def test_bias_loop_full_size_teacher_forced(moe):
    """The skewed-load bias loop at its full size, as the benchmark runs it:
    T = 16384 tokens per step, 50 steps, V3 dimensions, Zipf-scaled
    centroids, gamma = 1e-3, the whole layer every step (bf16 h) followed by
    the bias update.  At T = 16384 the router runs one CTA per 128-token
    tile (the unsplit path: 128 tiles already fill most of the SMs).

    Teacher-forced: every step's routing is compared on every token with
    the oracle given the GPU's incoming bias, and the bias after the step
    bit for bit with the oracle's update applied to the GPU's counts (so one
    near-tied token cannot fork the trajectory).  h is compared with the
    definition on sampled tokens of the first and the last step."""
    cfg = get_config("skew")
    g = generate(cfg, "cuda")
    layer = moe.MoELayer(g["E"], g["b"].clone(), g["w_gate"], g["w_up"],
                         g["w_down"], g["ws_gate"], g["ws_up"], g["ws_down"],
                         top_k=cfg.top_k, h_dtype=torch.bfloat16)
    b = layer.buffers(cfg.T)
    E64 = as_f64(g["E"])
    TK = cfg.T * cfg.top_k
    rng = np.random.default_rng(cfg.seed)
    mm, nears = [], []
    for step in range(cfg.steps):
        u = step_tokens(cfg, step, "cuda")
        b_in = layer.bias.cpu().numpy().copy()
        h = layer(u, update_bias=True, gamma=cfg.gamma)
        torch.cuda.synchronize()
        moe.get_device_error()
        idx = b.topk_idx.cpu().numpy()
        c = b.counts.cpu().numpy()
        r = om.route(as_f64(u), E64, b_in.astype(np.float64), cfg.top_k)
        nears.append(check_routing(r, b_in.astype(np.float64), idx, c,
                                   cfg.top_k))
        want = om.update_bias(b_in, c, TK, cfg.gamma)
        assert layer.bias.cpu().numpy().tobytes() == want.tobytes(), step
        mm.append(c.max() / (TK / cfg.n_routed))
        if step in (0, cfg.steps - 1):
            rows = np.sort(rng.choice(cfg.T, 4, replace=False))
            sel = torch.from_numpy(rows).cuda()
            routed, shared = oracle_weights(g)
            u64 = as_f64(u[sel])
            h_ref, _ = om.layer_forward(u64, E64, b_in.astype(np.float64),
                                        cfg.top_k, routed, shared,
                                        idx_override=idx[rows])
            got = h[sel].float().cpu().numpy()
            assert np.all(np.abs(got - h_ref) <= 2e-2 + half_ulp_bf16(h_ref))
    # the loop moves the load towards balance
    assert mm[-1] < mm[0], (mm[0], mm[-1])
    print("skew max/mean load", round(mm[0], 3), "->", round(mm[-1], 3),
          "near-ties per step", nears)
    del layer, g
    torch.cuda.empty_cache()


def test_bias_loop_teacher_forced(moe):
    """Skewed routing with the +-gamma update after every step (V3 dims,
    fewer tokens and steps): each step's bias is bit-exact against the
    oracle's update applied to the GPU's counts, and the GPU's routing
    matches the oracle given the GPU's incoming bias."""
    cfg = get_config("skew").with_(T=512, steps=6)
    t = generate(cfg, "cpu", experts=False)
    E = t["E"].cuda()
    bias = torch.zeros(cfg.n_routed, device="cuda")
    sh = _shape(moe, cfg)
    ws = _ws(moe, sh)
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    gate = torch.empty((cfg.T, cfg.top_k), device="cuda")
    counts = torch.empty(cfg.n_routed, dtype=torch.int32, device="cuda")
    E64 = as_f64(t["E"])
    for step in range(cfg.steps):
        u = step_tokens(cfg, step)
        b_in = bias.cpu().numpy().copy()
        moe.route(sh, u.cuda(), E, bias, idx, gate, counts, ws)
        moe.update_bias(cfg.n_routed, counts, cfg.T * cfg.top_k, cfg.gamma,
                        bias)
        moe.get_device_error()
        c = counts.cpu().numpy()
        r = om.route(as_f64(u), E64, b_in.astype(np.float64), cfg.top_k)
        check_routing(r, b_in.astype(np.float64), idx.cpu().numpy(), c,
                      cfg.top_k)
        want = om.update_bias(b_in, c, cfg.T * cfg.top_k, cfg.gamma)
        assert bias.cpu().numpy().tobytes() == want.tobytes(), step


def test_bias_loop_resume_bit_exact(moe, tmp_path):
    """Checkpoint/resume of the bias loop: 3 steps, save, a fresh bias
    tensor restored from the file, 3 more steps == 6 uninterrupted steps."""
    from mixture_experts_layer_gemms_b300.checkpoint import load_bias, save_bias
    cfg = get_config("skew").with_(T=384, steps=6)
    t = generate(cfg, "cpu", experts=False)
    E = t["E"].cuda()
    sh = _shape(moe, cfg)
    ws = _ws(moe, sh)
    idx = torch.empty((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    gate = torch.empty((cfg.T, cfg.top_k), device="cuda")
    counts = torch.empty(cfg.n_routed, dtype=torch.int32, device="cuda")
    us = [step_tokens(cfg, s).cuda() for s in range(cfg.steps)]

    def run(bias, steps):
        for s in steps:
            moe.route(sh, us[s], E, bias, idx, gate, counts, ws)
            moe.update_bias(cfg.n_routed, counts, cfg.T * cfg.top_k,
                            cfg.gamma, bias)
        torch.cuda.synchronize()
        moe.get_device_error()
    b_full = torch.zeros(cfg.n_routed, device="cuda")
    run(b_full, range(6))
    b_half = torch.zeros(cfg.n_routed, device="cuda")
    run(b_half, range(3))
    path = str(tmp_path / "bias.ckpt")
    save_bias(path, b_half, 3)
    b_loaded, step = load_bias(path)
    assert step == 3
    b_resumed = torch.from_numpy(b_loaded.copy()).cuda()
    run(b_resumed, range(step, 6))
    assert b_resumed.cpu().numpy().tobytes() == b_full.cpu().numpy().tobytes()
    assert (b_full.cpu().numpy() != 0).any()


def test_wait_timeout_is_reported_and_context_survives(moe):
    """A bounded device wait that nothing satisfies gives up, is reported as
    MOE_ERR_TIMEOUT, and the next calls on the same context still work."""
    moe.get_device_error()                      # start clean
    moe.selftest_wait_timeout(20000)            # 20 ms limit
    with pytest.raises(moe.MoEError) as ei:
        moe.get_device_error()
    assert ei.value.status == 5
    moe.get_device_error()                      # cleared
    cfg = get_config("mid").with_(T=256)
    t = generate(cfg, "cpu", experts=False)
    idx, gate, counts = _route_gpu(moe, cfg, t["u"].cuda(), t["E"].cuda(),
                                   t["b"].cuda())
    assert counts.sum() == cfg.T * cfg.top_k


@pytest.mark.parametrize("name,quant", [("mid", None), ("mid", "fp8")])
def test_layer_cuda_graph_replay(moe, name, quant):
    """One captured step replays bit-identically to the eager step, and
    follows new tokens written into its input buffer."""
    cfg = get_config(name).with_(T=512)
    g = make_inputs(cfg)
    mk = lambda: moe.MoELayer(g["E"], g["b"].clone(), g["w_gate"], g["w_up"],
                              g["w_down"], g["ws_gate"], g["ws_up"],
                              g["ws_down"], top_k=cfg.top_k, quant=quant)
    eager, graphed = mk(), mk()
    u = g["u"].clone()
    run = graphed.graph(u)
    for seed in (0, 1):
        if seed:
            u.copy_(torch.randn(u.shape, generator=torch.Generator(
                device="cuda").manual_seed(7), device="cuda").to(u.dtype))
        want = eager(u).clone()
        got = run().clone()
        torch.cuda.synchronize()
        moe.get_device_error()
        assert torch.equal(want, got), seed


def test_forward_host_pipeline(moe):
    """Host batches through the copy/compute pipeline give the same h as
    device-side forwards, in batch order (with the bias moving per batch)."""
    cfg = get_config("mid").with_(T=256)
    g = make_inputs(cfg)
    mk = lambda: moe.MoELayer(g["E"], g["b"].clone(), g["w_gate"], g["w_up"],
                              g["w_down"], g["ws_gate"], g["ws_up"],
                              g["ws_down"], top_k=cfg.top_k,
                              h_dtype=torch.bfloat16)
    gen = torch.Generator(device="cuda").manual_seed(3)
    us = [torch.randn((cfg.T, cfg.d), generator=gen, device="cuda")
          .to(torch.bfloat16) for _ in range(5)]
    ref_layer = mk()
    want = [ref_layer(x, update_bias=True).cpu() for x in us]
    layer = mk()
    ins = [x.cpu().pin_memory() for x in us]
    outs = [torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16).pin_memory()
            for _ in us]
    layer.forward_host(ins, outs, update_bias=True)
    torch.cuda.synchronize()
    moe.get_device_error()
    for i, (a, b) in enumerate(zip(want, outs)):
        assert torch.equal(a, b), i
    assert torch.equal(layer.bias, ref_layer.bias)


@pytest.mark.parametrize("name,T", [("mid", 1024), ("mid", 3000),
                                    ("v3_prefill", 2048)])
def test_shared_overlap_matches(moe, name, T):
    """The shared experts on a side stream (beside the permute and the
    routed experts) give the same h, bit for bit, as the single call, eager
    and replayed from a CUDA graph."""
    cfg = get_config(name).with_(T=T)
    g = make_inputs(cfg) if name != "v3_prefill" else generate(cfg, "cuda")
    mk = lambda ov: moe.MoELayer(g["E"], g["b"].clone(), g["w_gate"],
                                 g["w_up"], g["w_down"], g["ws_gate"],
                                 g["ws_up"], g["ws_down"], top_k=cfg.top_k,
                                 h_dtype=torch.bfloat16, overlap_shared=ov)
    plain, side = mk(False), mk(True)
    u = g["u"].clone()
    assert side._shared_side_stream(u) is not None
    want = plain(u, update_bias=True).clone()
    got = side(u, update_bias=True).clone()
    torch.cuda.synchronize()
    moe.get_device_error()
    assert torch.equal(want, got)
    assert torch.equal(plain.bias, side.bias)
    run = side.graph(u)
    want = plain(u).clone()
    got = run().clone()
    torch.cuda.synchronize()
    moe.get_device_error()
    assert torch.equal(want, got)
