"""Pins of the FP8 (e4m3, block-scaled) oracle against things other than
itself: the bit-field definition of e4m3, torch's float8_e4m3fn cast (a
library routine), brute-force nearest-value search, closed forms of the
scale rule, and a scalar-loop FFN on tiny sizes."""
import itertools

import numpy as np
import pytest
import torch

import oracle.fp8 as of
import oracle.moe as om


def _finite_values():
    codes = np.arange(256, dtype=np.uint8)
    v = of.e4m3_decode(codes)
    keep = ~np.isnan(v)
    return codes[keep], v[keep]


def _nearest_brute(x, table):
    """Nearest table value by exhaustive search; ties to the even code."""
    codes, vals = table
    out = np.empty_like(x)
    for i, xi in enumerate(x):
        if abs(xi) > 448:
            out[i] = np.copysign(448.0, xi)
            continue
        d = np.abs(vals - xi)
        best = np.nonzero(d == d.min())[0]
        if len(best) > 1:
            best = [b for b in best if codes[b] % 2 == 0] or best
        out[i] = vals[best[0]]
    return out


def test_e4m3_decode_table():
    codes, vals = _finite_values()
    assert len(vals) == 254                        # 2 NaN patterns
    assert np.nanmax(vals) == 448.0 and np.nanmin(vals) == -448.0
    assert of.e4m3_decode(0x01) == 2.0 ** -9       # smallest subnormal
    assert of.e4m3_decode(0x08) == 2.0 ** -6       # smallest normal
    assert of.e4m3_decode(0x38) == 1.0
    assert of.e4m3_decode(0x7E) == 448.0
    assert np.isnan(of.e4m3_decode(0x7F))


def test_e4m3_round_fixes_every_code():
    codes, vals = _finite_values()
    assert np.array_equal(of.e4m3_round(vals), vals)
    assert np.array_equal(of.e4m3_encode(vals), codes)


def test_e4m3_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 40,
                        rng.standard_normal(20000) * 2.0 ** -7,
                        rng.uniform(-448, 448, 20000)])
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64)
    assert np.array_equal(of.e4m3_round(x), want.numpy())


def test_e4m3_round_brute_force_and_ties():
    table = _finite_values()
    pos = np.sort(table[1][table[1] > 0])
    mids = (pos[:-1] + pos[1:]) / 2              # every tie between codes
    rng = np.random.default_rng(1)
    x = np.concatenate([mids, -mids, rng.uniform(-460, 460, 3000),
                        [0.0, 449.0, 470.0, -1000.0]])
    assert np.array_equal(of.e4m3_round(x), _nearest_brute(x, table))


def test_scale_exponent_closed_form():
    rng = np.random.default_rng(2)
    a = np.abs(rng.standard_normal(5000)) * np.exp2(rng.integers(-20, 20, 5000))
    e = of.scale_exponent(a)
    assert np.all(a <= 448 * np.exp2(e))
    assert np.all(a > 448 * np.exp2(e - 1))
    assert of.scale_exponent([448.0, 0.0, 224.0]).tolist() == [0, 0, -1]


def test_quantize_rows_blocks():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 384)) * np.exp2(rng.integers(-4, 4, (5, 1)))
    q, e = of.quantize_rows(x)
    assert e.shape == (5, 3)
    for r, b in itertools.product(range(5), range(3)):
        blk = slice(128 * b, 128 * b + 128)
        qs = q[r, blk]
        assert np.abs(qs).max() <= 448 and np.abs(qs).max() > 224 - 16
        back = qs * 2.0 ** e[r, b]
        # round to nearest: error <= half the spacing 2^(E-3) of each value
        err = np.abs(back - x[r, blk])
        assert np.all(err <= np.maximum(np.abs(x[r, blk]), 2.0 ** (e[r, b] - 6))
                      * 2.0 ** -4 + 1e-300)
    w = rng.standard_normal((256, 256))
    qw, ew = of.quantize_blocks(w)
    assert ew.shape == (2, 2)
    assert np.abs(of.dequant_blocks(qw, ew) - w).max() <= np.abs(w).max() / 16


def test_qgemm_is_matmul_of_dequantized():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((7, 256))
    w = rng.standard_normal((128, 256)) / 16
    qx, ex = of.quantize_rows(x)
    qw, ew = of.quantize_blocks(w)
    got = of.qgemm(qx, ex, qw, ew)
    want = of.dequant_rows(qx, ex) @ of.dequant_blocks(qw, ew).T
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def _scalar_fp8_ffn(x, wg, wu, wd):
    """Scalar loops: quantize by brute-force nearest value, dot products."""
    table = _finite_values()

    def qrow(v):
        out, ex = [], []
        for b in range(0, len(v), 128):
            blk = v[b:b + 128]
            a = max(abs(t) for t in blk)
            e = 0
            if a > 0:
                e = -200
                while a > 448 * 2.0 ** e:
                    e += 1
            ex.append(e)
            out += list(_nearest_brute(np.array(blk) * 2.0 ** -e, table)
                        * 2.0 ** e)
        return out

    def qmat(W):
        W = np.asarray(W)
        out = np.zeros_like(W)
        for r0 in range(0, W.shape[0], 128):
            for c0 in range(0, W.shape[1], 128):
                blk = W[r0:r0 + 128, c0:c0 + 128]
                a = np.abs(blk).max()
                e = 0
                if a > 0:
                    e = -200
                    while a > 448 * 2.0 ** e:
                        e += 1
                out[r0:r0 + 128, c0:c0 + 128] = _nearest_brute(
                    (blk * 2.0 ** -e).ravel(), table).reshape(blk.shape) \
                    * 2.0 ** e
        return out

    G, U, D = qmat(wg), qmat(wu), qmat(wd)
    ys = []
    for row in x:
        xq = qrow(list(row))
        g = [sum(a * b for a, b in zip(G[i], xq)) for i in range(len(G))]
        u = [sum(a * b for a, b in zip(U[i], xq)) for i in range(len(U))]
        h = [gi / (1 + np.exp(-gi)) * ui for gi, ui in zip(g, u)]
        hq = qrow(h)
        ys.append([sum(a * b for a, b in zip(D[j], hq)) for j in range(len(D))])
    return np.array(ys)


def test_fp8_ffn_scalar_loops():
    rng = np.random.default_rng(5)
    d, I = 256, 128
    x = rng.standard_normal((3, d))
    wg = rng.standard_normal((I, d)) / np.sqrt(d)
    wu = rng.standard_normal((I, d)) / np.sqrt(d)
    wd = rng.standard_normal((d, I)) / np.sqrt(I)
    got = of.fp8_swiglu_ffn(x, of.quantize_expert(wg, wu, wd))
    want = _scalar_fp8_ffn(x, wg, wu, wd)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_fp8_ffn_near_full_precision():
    """Quantization error of the whole FFN.  e4m3 keeps 3 mantissa bits, so
    each quantized operand carries ~3.6% rms relative error; four quantized
    operands on the path (x, W_gate/W_up, H, W_down) give ~7% rms."""
    rng = np.random.default_rng(6)
    d, I = 512, 256
    x = rng.standard_normal((64, d))
    wg = rng.standard_normal((I, d)) / np.sqrt(d)
    wu = rng.standard_normal((I, d)) / np.sqrt(d)
    wd = rng.standard_normal((d, I)) / np.sqrt(I)
    y8 = of.fp8_swiglu_ffn(x, of.quantize_expert(wg, wu, wd))
    y = om.swiglu_ffn(x, wg, wu, wd)
    rel = np.linalg.norm(y8 - y) / np.linalg.norm(y)
    assert 0.03 < rel < 0.1, rel


def test_mutant_truncating_round_caught(monkeypatch):
    def trunc(x):
        x = np.asarray(x, dtype=np.float64)
        ax = np.abs(x)
        _, ex = np.frexp(ax)
        sp = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)
        return np.copysign(np.minimum(np.floor(ax / sp) * sp, 448.0), x)
    monkeypatch.setattr(of, "e4m3_round", trunc)
    x = np.random.default_rng(7).uniform(-400, 400, 5000)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64)
    assert not np.array_equal(of.e4m3_round(x), want.numpy())


def test_mutant_scale_off_by_one_caught(monkeypatch):
    real = of.scale_exponent
    monkeypatch.setattr(of, "scale_exponent", lambda a: real(a) + 1)
    a = np.array([3.0, 500.0, 0.01])
    e = of.scale_exponent(a)
    assert not np.all(a > 448 * np.exp2(e - 1))
