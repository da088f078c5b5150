"""GPU parity of the e4m3 (MOE_FP8) expert path against the fp64 oracle of
the same quantized arithmetic (oracle/fp8.py).

* weight and activation codes and their block scales: bit-exact (both sides
  scale by a power of two, which is exact, and round to nearest even);
* expert outputs and the layer output: the bf16 bar (max-abs 2e-2,
  relative Frobenius 5e-3) against the quantized oracle.  The GPU forms
  SwiGLU from fp32 sums and the oracle from exact ones, so a requantized
  H element can land one e4m3 step apart where its value sits on a rounding
  boundary; each such step moves y by at most 2^-4 |h| |W_down| -- far
  inside the bar.
Requires a B300 (sm_103a)."""
import numpy as np
import pytest
import torch

import oracle.fp8 as of
import oracle.moe as om
from moe_inputs import as_f64, generate, get_config
from parity_utils import assert_close, check_routing, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_layer_gemms_b300 as m
    return m


def _layer(moe, g, cfg, h_dtype=torch.float32):
    S = cfg.n_shared
    return moe.MoELayer(g["E"], g["b"].clone(), g["w_gate"], g["w_up"],
                        g["w_down"], g["ws_gate"] if S else None,
                        g["ws_up"] if S else None, g["ws_down"] if S else None,
                        top_k=cfg.top_k, h_dtype=h_dtype, quant="fp8")


def _codes_scales(buf, rows, cols):
    """Split a packed buffer into codes [rows, cols] and scales."""
    b = buf.cpu().numpy()
    nc = (rows * cols + 255) // 256 * 256
    codes = b[:rows * cols].reshape(rows, cols)
    sc = b[nc:nc + (rows // 128) * (cols // 128) * 4].view(np.float32)
    return codes, sc.reshape(rows // 128, cols // 128)


def _ue8(buf, rows, cols, weights):
    """The UE8M0 scale table after the codes and fp32 scales: [R][P] bytes,
    R = rows / 128 for weights, rows for activations; P = cols / 128 rounded
    up to 16."""
    b = buf.cpu().numpy()
    r256 = lambda x: (x + 255) // 256 * 256      # noqa: E731
    R = rows // 128 if weights else rows
    off = r256(rows * cols) + r256(R * (cols // 128) * 4)
    P = ((cols // 128) + 15) // 16 * 16
    return b[off:off + R * P].reshape(R, P)


def _expect_ue8(e, P):
    """127 + e for every block, 127 (2^0) in the padding."""
    t = np.full((e.shape[0], P), 127, dtype=np.uint8)
    t[:, :e.shape[1]] = (127 + e).astype(np.uint8)
    return t


def _expect(q, e):
    return of.e4m3_encode(q), np.exp2(e).astype(np.float32)


SMALL = dict(T=64, d=256, n_routed=16, top_k=4, n_shared=1, d_ff=128,
             dtype="bf16")


def test_fp8_pack_bit_exact(moe):
    cfg = get_config("tiny").with_(**dict(SMALL, n_shared=2, d_ff=256))
    g = make_inputs(cfg)
    layer = _layer(moe, g, cfg)
    torch.cuda.synchronize()
    moe.get_device_error()
    N, d, I, S = cfg.n_routed, cfg.d, cfg.d_ff, cfg.n_shared
    # routed gate/up: 128-row blocks alternate gate / up of the same rows
    codes, sc = _codes_scales(layer.w_gu, 2 * N * I, d)
    for e in range(N):
        qg, eg = of.quantize_blocks(as_f64(g["w_gate"][e]))
        qu, eu = of.quantize_blocks(as_f64(g["w_up"][e]))
        for j in range(I // 128):
            r0 = e * 2 * I + j * 256
            for part, (q, ex) in enumerate(((qg, eg), (qu, eu))):
                wc, ws = _expect(q[j * 128:(j + 1) * 128], ex[j:j + 1])
                assert np.array_equal(codes[r0 + 128 * part:
                                            r0 + 128 * part + 128], wc)
                assert np.array_equal(sc[r0 // 128 + part], ws[0])
    # the UE8M0 table of the same scales (rows = packed row blocks)
    ue = _ue8(layer.w_gu, 2 * N * I, d, True)
    exps = []
    for e in range(N):
        _, eg = of.quantize_blocks(as_f64(g["w_gate"][e]))
        _, eu = of.quantize_blocks(as_f64(g["w_up"][e]))
        for j in range(I // 128):
            exps += [eg[j], eu[j]]
    assert np.array_equal(ue, _expect_ue8(np.array(exps), ue.shape[1]))
    # routed down: [N*d, I]
    codes, sc = _codes_scales(layer.w_down, N * d, I)
    for e in range(N):
        q, ex = of.quantize_blocks(as_f64(g["w_down"][e]))
        wc, ws = _expect(q, ex)
        assert np.array_equal(codes[e * d:(e + 1) * d], wc)
        assert np.array_equal(sc[e * d // 128:(e + 1) * d // 128], ws)
    # shared down: the S matrices side by side along the reduction
    codes, sc = _codes_scales(layer.ws_down, d, S * I)
    for s in range(S):
        q, ex = of.quantize_blocks(as_f64(g["ws_down"][s]))
        wc, ws = _expect(q, ex)
        assert np.array_equal(codes[:, s * I:(s + 1) * I], wc)
        assert np.array_equal(sc[:, s * I // 128:(s + 1) * I // 128], ws)


def test_fp8_permute_bit_exact(moe):
    cfg = get_config("tiny").with_(**dict(SMALL, T=300))
    g = make_inputs(cfg)
    layer = _layer(moe, g, cfg)
    layer(g["u"])
    torch.cuda.synchronize()
    moe.get_device_error()
    b = layer.buffers(cfg.T)
    A, d = cfg.T * cfg.top_k, cfg.d
    perm = b.perm.cpu().numpy()
    codes, _ = _codes_scales(b.x_perm, A, d)
    raw = b.x_perm.cpu().numpy()
    nc = (A * d + 255) // 256 * 256
    sx = raw[nc:nc + (d // 128) * A * 4].view(np.float32).reshape(d // 128, A)
    q, e = of.quantize_rows(as_f64(g["u"])[perm])
    assert np.array_equal(codes, of.e4m3_encode(q))
    assert np.array_equal(sx, np.exp2(e).T.astype(np.float32))
    ue = _ue8(b.x_perm, A, d, False)
    assert np.array_equal(ue, _expect_ue8(e, ue.shape[1]))


def _fp8_oracle_h(g, cfg, idx, rows=None):
    u = as_f64(g["u"])
    sel = np.arange(cfg.T) if rows is None else np.asarray(rows)
    r = om.route(u[sel], as_f64(g["E"]), as_f64(g["b"]), cfg.top_k)
    gate = np.take_along_axis(r["s"], idx[sel].astype(np.int64), axis=1)
    cache = {}

    def routed(e):
        if e not in cache:
            cache[e] = of.quantize_expert(*(as_f64(g[k][e]) for k in
                                            ("w_gate", "w_up", "w_down")))
        return cache[e]
    shared = [of.quantize_expert(*(as_f64(g[k][s]) for k in
                                   ("ws_gate", "ws_up", "ws_down")))
              for s in range(cfg.n_shared)]
    h = of.fp8_layer_forward(u[sel], idx[sel], gate, routed, shared)
    return h, r, u[sel]


FP8_CASES = {
    # 32-token chunks (average group <= 48 tokens)
    "small_T64": ("tiny", dict(SMALL)),
    "small_ragged_T37_S2": ("tiny", dict(SMALL, T=37, n_shared=2,
                                         d_ff=256)),
    # 128-token chunks, gate/up pair tiles, groups of several chunks
    "chunked_T1000_d512": ("tiny", dict(SMALL, T=1000, d=512, d_ff=256,
                                        n_shared=2)),
    "mid_dims_T700": ("mid", dict(T=700)),
    # the block-scaled CTA-pair kernel with reductions of 6 and 3 128-blocks
    # (scale groups of four stages, the last one partly used)
    "pair_d768_I384_T1200": ("tiny", dict(SMALL, T=1200, d=768, d_ff=384)),
    # d % 256 != 0: the single-SM kernels, prefill- and decode-sized groups
    "fallback_d384_T1200": ("tiny", dict(SMALL, T=1200, d=384, d_ff=256)),
    "fallback_small_d384_T64": ("tiny", dict(SMALL, d=384, d_ff=256)),
    "no_shared_T1": ("tiny", dict(SMALL, T=1, n_shared=0)),
    "no_shared_T900": ("tiny", dict(SMALL, T=900, n_shared=0, d=512)),
}


@pytest.mark.parametrize("case", sorted(FP8_CASES))
def test_fp8_layer_parity(moe, case):
    name, over = FP8_CASES[case]
    cfg = get_config(name).with_(**over)
    g = make_inputs(cfg)
    layer = _layer(moe, g, cfg)
    h = layer(g["u"])
    torch.cuda.synchronize()
    moe.get_device_error()
    b = layer.buffers(cfg.T)
    idx = b.topk_idx.cpu().numpy()
    h_ref, r, u64 = _fp8_oracle_h(g, cfg, idx)
    check_routing(r, as_f64(g["b"]), idx, b.counts.cpu().numpy(), cfg.top_k)
    e = assert_close(h.float().cpu().numpy(), h_ref, base=u64, what=case)
    print(case, e)


def test_fp8_skewed_multi_chunk(moe):
    """A bias that sends every token to the same K experts: on the e4m3
    CTA-pair kernel each of them splits into chunks of at most 192 tokens
    (4 chunks of 150, rounded up to 160 MMA columns, here), and the other
    experts are empty."""
    cfg = get_config("mid").with_(T=600)
    g = make_inputs(cfg)
    b = torch.zeros(cfg.n_routed)
    b[[5, 17, 33, 40, 41, 63]] = 2.0
    g["b"] = b.cuda()
    layer = _layer(moe, g, cfg)
    h = layer(g["u"])
    torch.cuda.synchronize()
    moe.get_device_error()
    buf = layer.buffers(cfg.T)
    counts = buf.counts.cpu().numpy()
    assert sorted(np.nonzero(counts)[0].tolist()) == [5, 17, 33, 40, 41, 63]
    idx = buf.topk_idx.cpu().numpy()
    h_ref, r, u64 = _fp8_oracle_h(g, cfg, idx)
    e = assert_close(h.float().cpu().numpy(), h_ref, base=u64, what="skew")
    print("fp8 skewed", e)


def test_fp8_close_to_bf16_layer(moe):
    """The e4m3 layer stays within the quantization error of the bf16 one."""
    cfg = get_config("tiny").with_(**dict(SMALL, T=256))
    g = make_inputs(cfg)
    h8 = _layer(moe, g, cfg)(g["u"]).float().clone()
    S = cfg.n_shared
    h16 = moe.MoELayer(g["E"], g["b"].clone(), g["w_gate"], g["w_up"],
                       g["w_down"], g["ws_gate"], g["ws_up"], g["ws_down"],
                       top_k=cfg.top_k)(g["u"]).float()
    torch.cuda.synchronize()
    moe.get_device_error()
    u = g["u"].float()
    rel = (torch.linalg.norm(h8 - h16) / torch.linalg.norm(h16 - u)).item()
    assert rel < 0.1, rel


@pytest.mark.parametrize("name,n_sample", [("v3_decode", 6),
                                           ("v3_prefill", 4)])
def test_fp8_full_size_sampled(moe, name, n_sample):
    """V3 shapes through the e4m3 path; sampled tokens against the oracle
    (each sampled token needs its experts quantized on the CPU)."""
    cfg = get_config(name)
    g = generate(cfg, "cuda")
    layer = _layer(moe, g, cfg)
    h = layer(g["u"])
    torch.cuda.synchronize()
    moe.get_device_error()
    idx = layer.buffers(cfg.T).topk_idx.cpu().numpy()
    rows = np.random.default_rng(0).choice(cfg.T, n_sample, replace=False)
    h_ref, r, u64 = _fp8_oracle_h(g, cfg, idx, rows)
    got = h.float().cpu().numpy()[rows]
    assert_close(got, h_ref, base=u64, what=name)


def test_fp8_empty_batch(moe):
    cfg = get_config("tiny").with_(**dict(SMALL, T=0))
    g = make_inputs(cfg.with_(T=4))
    layer = _layer(moe, g, cfg)
    h = layer(g["u"][:0])
    torch.cuda.synchronize()
    moe.get_device_error()
    assert h.shape == (0, cfg.d)
