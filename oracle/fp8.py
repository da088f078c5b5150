"""FP8 (e4m3) expert FFN of the DeepSeekMoE layer -- fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU
baseline call this; the product path never does.

Source (cited by page and section):

* [report-commentary] DeepSeek-V3 technical-report commentary
  (cooktownmusic.com), FP8 training-framework part with Fig. 6 and Fig. 7:
  most GEMMs run with FP8 inputs; activations and weights are grouped into
  blocks and each block is scaled on its own (fine-grained quantization,
  Fig. 7a) so that outliers stay local; partial sums of the tensor cores are
  promoted to FP32 on the CUDA cores at an interval of N_C = 128 elements of
  the reduction (Fig. 7b).
* [V3-features] "DeepSeek V3特點與技術" (techduker.com), highlight list: the
  MoE gating stays in high precision -- so the router is not quantized.

Readings where the pages are silent (listed with reasons in the project's
design notes):

* element format: e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
  bits; no infinities; largest finite 448; subnormals 2^-9 .. 7 * 2^-9),
  round to nearest, ties to even, saturating at +-448;
* block shapes: activations 1 x 128 (one token, 128 consecutive channels of
  the reduction dimension), weights 128 x 128 (128 output rows, 128
  reduction channels) -- the tile shapes are not on the pages; 128 matches
  the promotion interval N_C;
* scales: powers of two, s = 2^e with e the smallest integer such that the
  block's largest magnitude is <= 448 * 2^e (e = 0 for an all-zero block), so
  that scaling and rescaling are exact;
* FFN: x and every weight matrix are quantized; SwiGLU is computed at full
  precision on the dequantized GEMM results; H = SiLU(G) * U is quantized
  again (1 x 128 blocks along the intermediate dimension) before the down
  projection; the projection outputs are not quantized.

The oracle computes each quantized GEMM as
    D[r, c] = sum_kb 2^(e_w[r/128, kb] + e_x[c, kb]) * sum_{k in kb} q_w q_x
in float64 (products of two e4m3 values and their 128-term sums are exact in
float64), i.e. the definition with no blocking beyond the quantization's.
Library primitives used as single steps: numpy frexp, ldexp, rint, matmul.
"""
from __future__ import annotations

from typing import Callable, Sequence, Tuple

import numpy as np

from .moe import silu

E4M3_MAX = 448.0
BLOCK = 128


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# --- the element format ----------------------------------------------------

def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value (ties to even mantissa), saturating at +-448.

    A normal e4m3 number with unbiased exponent E (-6 <= E <= 8) has spacing
    2^(E-3); below 2^-6 the subnormal spacing is 2^-9.  Rounding is done on
    x / spacing with round-half-even, which is exact in float64.  NaN stays
    NaN.
    """
    x = _f64(x)
    ax = np.abs(x)
    _, ex = np.frexp(ax)                 # ax = m * 2^ex, m in [0.5, 1)
    E = np.maximum(ex - 1, -6)           # exponent of the binade
    spacing = np.ldexp(1.0, E - 3)
    q = np.rint(ax / spacing) * spacing
    q = np.minimum(q, E4M3_MAX)
    q = np.where(ax == 0, 0.0, q)
    return np.where(np.isnan(x), np.nan, np.copysign(q, x))


def e4m3_decode(code) -> np.ndarray:
    """Value of an e4m3 bit pattern (uint8): sign, 4-bit exponent field with
    bias 7, 3-bit mantissa; field 0 is subnormal; S.1111.111 is NaN."""
    c = np.asarray(code, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, ef - 7)
    sub = np.ldexp(m / 8.0, -6)
    v = np.where(ef == 0, sub, normal)
    v = np.where((ef == 15) & (m == 7), np.nan, v)
    return s * v


def e4m3_encode(v) -> np.ndarray:
    """Bit pattern (uint8) of values that are already e4m3 numbers."""
    v = _f64(v)
    sign = np.signbit(v).astype(np.int64) << 7
    av = np.abs(v)
    _, ex = np.frexp(av)
    E = ex - 1
    normal = E >= -6
    ef = np.where(normal, E + 7, 0)
    m = np.where(normal, np.ldexp(av, -E) - 1.0, np.ldexp(av, 6)) * 8.0
    m = np.where(av == 0, 0.0, m)
    ef = np.where(av == 0, 0, ef)
    if not np.all(m == np.rint(m)):
        raise ValueError("not an e4m3 value")
    return (sign | (ef << 3) | m.astype(np.int64)).astype(np.uint8)


# --- block scales ----------------------------------------------------------

def scale_exponent(amax) -> np.ndarray:
    """Smallest integer e with amax <= 448 * 2^e (0 where amax == 0).

    With amax = m * 2^ex (m in [0.5, 1)) and 448 = 0.875 * 2^9 the condition
    is m * 2^ex <= 0.875 * 2^(9+e): e = ex - 9 when m <= 0.875, else ex - 8.
    """
    a = _f64(amax)
    m, ex = np.frexp(a)
    e = np.where(m <= 0.875, ex - 9, ex - 8)
    return np.where(a == 0, 0, e).astype(np.int64)


def quantize_rows(x, block: int = BLOCK):
    """1 x `block` quantization along the last axis of x [R, K].

    Returns (q [R, K] e4m3 values as float64, e [R, K/block] int64)."""
    x = _f64(x)
    R, K = x.shape
    if K % block:
        raise ValueError("K must be a multiple of the block")
    xb = x.reshape(R, K // block, block)
    e = scale_exponent(np.abs(xb).max(axis=2))
    q = e4m3_round(np.ldexp(xb, -e[:, :, None]))
    return q.reshape(R, K), e


def quantize_blocks(w, block: int = BLOCK):
    """`block` x `block` quantization of a weight matrix w [rows, K].

    Returns (q [rows, K] e4m3 values as float64, e [rows/block, K/block])."""
    w = _f64(w)
    R, K = w.shape
    if R % block or K % block:
        raise ValueError("both dimensions must be multiples of the block")
    wb = w.reshape(R // block, block, K // block, block)
    e = scale_exponent(np.abs(wb).max(axis=(1, 3)))
    q = e4m3_round(np.ldexp(wb, -e[:, None, :, None]))
    return q.reshape(R, K), e


def dequant_rows(q, e, block: int = BLOCK) -> np.ndarray:
    return _f64(q) * np.ldexp(1.0, np.repeat(e, block, axis=1))


def dequant_blocks(q, e, block: int = BLOCK) -> np.ndarray:
    return _f64(q) * np.ldexp(1.0, np.repeat(np.repeat(e, block, axis=0),
                                             block, axis=1))


# --- quantized GEMM and FFN ------------------------------------------------

def qgemm(qx, ex, qw, ew, block: int = BLOCK) -> np.ndarray:
    """D = x_q . w_q^T with per-block scales: for every reduction block kb,
    the exact sum of e4m3 products times 2^(e_w + e_x), summed over kb
    ([report-commentary], Fig. 7b: partial sums promoted every N_C = 128)."""
    qx, qw = _f64(qx), _f64(qw)
    R, K = qx.shape
    out = np.zeros((R, qw.shape[0]))
    for kb in range(K // block):
        sl = slice(kb * block, (kb + 1) * block)
        part = qx[:, sl] @ qw[:, sl].T
        sc = np.ldexp(1.0, ex[:, kb][:, None] +
                      np.repeat(ew[:, kb], block)[None, :])
        out += sc * part
    return out


QWeights = Tuple[Tuple[np.ndarray, np.ndarray], Tuple[np.ndarray, np.ndarray],
                 Tuple[np.ndarray, np.ndarray]]


def quantize_expert(w_gate, w_up, w_down) -> QWeights:
    """Each of the three matrices in 128 x 128 blocks."""
    return (quantize_blocks(w_gate), quantize_blocks(w_up),
            quantize_blocks(w_down))


def fp8_swiglu_ffn(x, qweights: QWeights) -> np.ndarray:
    """y = W_down(SiLU(W_gate x) * W_up x) with x, the weights and H in e4m3
    (readings in the module docstring).  x [R, d] -> y [R, d]."""
    (qg, eg), (qu, eu), (qd, ed) = qweights
    qx, ex = quantize_rows(x)
    g = qgemm(qx, ex, qg, eg)
    u = qgemm(qx, ex, qu, eu)
    h = silu(g) * u
    qh, eh = quantize_rows(h)
    return qgemm(qh, eh, qd, ed)


def fp8_layer_forward(u, idx, gate, routed_q: Callable[[int], QWeights],
                      shared_q: Sequence[QWeights] = ()) -> np.ndarray:
    """h = u + sum_s FFN8^(s)(u) + sum_k g_k FFN8^(r)_{idx_k}(u) on a given
    routing (idx, gate); the router itself is not quantized."""
    u = _f64(u)
    h = u.copy()
    for w in shared_q:
        h += fp8_swiglu_ffn(u, w)
    idx = np.asarray(idx)
    gate = _f64(gate)
    for e in np.unique(idx):
        rows, ks = np.nonzero(idx == e)
        h[rows] += gate[rows, ks][:, None] * fp8_swiglu_ffn(u[rows],
                                                             routed_q(int(e)))
    return h
