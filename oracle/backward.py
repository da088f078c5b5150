"""Plain fp64 CPU oracle of the DeepSeekMoE layer BACKWARD pass.

TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU
baseline call this; the product path never does.

Source: "AI新顶流-DeepSeek 技术大揭秘" (blog.csdn.net), section
"FP8混合精度训练框架": each linear operator of training runs three GEMMs,
Fprop (the forward), Dgrad (the gradient of the activations) and Wgrad (the
gradient of the weights).  The layer whose gradients are taken is the
forward of ``oracle/moe.py`` ("【推理llm論文精讀】DeepSeek V3技術論文",
section 2.2, FFN-output equation h = u + sum_s FFN^(s)(u) +
sum_i g_i FFN^(r)_i(u) with g_i = s_i = Sigmoid(u . e_i) at the selected
experts).  The pages print no derivative; everything below is the chain
rule applied to that forward, written out:

* the selection (top-K of s + b) is piecewise constant: it passes no
  gradient, and the bias b gets none;
* per selected expert e of token t, with x = u_t, g = s_{t,e} and the
  upstream gradient dh_t:
      a = W_g x,  c = W_u x,  H = SiLU(a) * c,  y = W_d H
      dy = g dh_t                       (the gated output's gradient)
      dW_d += dy H^T
      dH = W_d^T dy
      da = dH * c * SiLU'(a),  SiLU'(a) = sig(a) (1 + a (1 - sig(a)))
      dc = dH * SiLU(a)
      dW_g += da x^T,  dW_u += dc x^T
      du_t += W_g^T da + W_u^T dc       (through the expert's input)
      dg = dh_t . y
      dz = dg * g (1 - g)               (through the sigmoid of the gate)
      du_t += dz e_e,  dE_e += dz u_t   (z = u_t . e_e)
* shared experts: the same with g = 1 and no gate term;
* the residual: du_t += dh_t.

Library primitives used as single steps: numpy matmul, exp.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

from .moe import route, sigmoid, silu

Weights = Tuple[np.ndarray, np.ndarray, np.ndarray]   # (W_gate, W_up, W_down)


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def silu_grad(a):
    """d SiLU(a) / da = sig(a) (1 + a (1 - sig(a))), fp64."""
    a = _f64(a)
    sg = sigmoid(a)
    return sg * (1.0 + a * (1.0 - sg))


def swiglu_ffn_backward(x, w_gate, w_up, w_down, dy):
    """Gradients of y = W_down (SiLU(W_gate x) * (W_up x)) for rows
    x [M, d] given dy [M, d].

    Returns (dx [M, d], dW_gate [I, d], dW_up [I, d], dW_down [d, I],
    y [M, d]), fp64.
    """
    x, dy = _f64(x), _f64(dy)
    wg, wu, wd = _f64(w_gate), _f64(w_up), _f64(w_down)
    a = x @ wg.T                        # [M, I]
    c = x @ wu.T                        # [M, I]
    H = silu(a) * c
    y = H @ wd.T                        # [M, d]
    dWd = dy.T @ H                      # [d, I]
    dH = dy @ wd                        # [M, I]
    da = dH * c * silu_grad(a)
    dc = dH * silu(a)
    dWg = da.T @ x                      # [I, d]
    dWu = dc.T @ x
    dx = da @ wg + dc @ wu              # [M, d]
    return dx, dWg, dWu, dWd, y


def gate_backward(dh_rows, y, g):
    """dz = (dh . y) * g (1 - g): the gradient reaching z = u . e through
    the gate g = Sigmoid(z) of one expert, for rows of tokens."""
    dg = np.sum(_f64(dh_rows) * _f64(y), axis=1)
    g = _f64(g)
    return dg * g * (1.0 - g)


def expert_backward(u, idx, gate, e: int, weights: Weights, E_e, dh):
    """Everything expert e contributes to the gradients, over the tokens
    that selected it (idx [T, K], gate [T, K]).

    Returns dict(rows, dx_rows (through the FFN input), du_rows (dx plus
    the gate term dz e_e), dW_gate, dW_up, dW_down, dE (the centroid's
    gradient, [d]), dz).
    """
    u, dh = _f64(u), _f64(dh)
    rows, ks = np.nonzero(np.asarray(idx) == e)
    g = _f64(gate)[rows, ks]
    x = u[rows]
    dy = g[:, None] * dh[rows]
    dx, dWg, dWu, dWd, y = swiglu_ffn_backward(x, *weights, dy)
    dz = gate_backward(dh[rows], y, g)
    E_e = _f64(E_e)
    return dict(rows=rows, dx_rows=dx, du_rows=dx + dz[:, None] * E_e,
                dW_gate=dWg, dW_up=dWu, dW_down=dWd, dE=dz @ x, dz=dz)


def layer_backward(u, E, b, K: int, routed: Callable[[int], Weights],
                   shared: Sequence[Weights], dh,
                   idx_override: Optional[np.ndarray] = None,
                   groups=None, tokens: Optional[np.ndarray] = None):
    """Gradients of the layer forward for the upstream gradient dh [T, d].

    Routing is recomputed by the forward's rule (``route`` in
    ``oracle/moe.py``), or taken from ``idx_override``; the gate is s at the
    selected experts.  ``tokens`` restricts the computation to those rows
    (du of those rows is exact; dE and the weight gradients then cover only
    their contributions).

    Returns dict(du [T', d], dE [N, d], dW {e: (dW_gate, dW_up, dW_down)}
    for every expert (zeros for unselected ones), dWs [(dW_gate, dW_up,
    dW_down)] per shared expert, idx, gate).
    """
    u, dh, E = _f64(u), _f64(dh), _f64(E)
    if tokens is not None:
        tokens = np.asarray(tokens)
        u, dh = u[tokens], dh[tokens]
        if idx_override is not None:
            idx_override = np.asarray(idx_override)[tokens]
    r = route(u, E, b, K, groups)
    idx = r["idx"] if idx_override is None else np.asarray(idx_override)
    gate = np.take_along_axis(r["s"], idx, axis=1)
    du = dh.copy()                                  # the residual
    dWs: List[Tuple[np.ndarray, np.ndarray, np.ndarray]] = []
    for w in shared:
        dx, dWg, dWu, dWd, _ = swiglu_ffn_backward(u, *w, dh)
        du += dx
        dWs.append((dWg, dWu, dWd))
    N, d = E.shape
    dE = np.zeros((N, d))
    dW: Dict[int, Tuple[np.ndarray, np.ndarray, np.ndarray]] = {}
    for e in range(N):
        wg, wu, wd = routed(e)
        if not np.any(idx == e):
            dW[e] = (np.zeros(np.shape(wg)), np.zeros(np.shape(wu)),
                     np.zeros(np.shape(wd)))
            continue
        out = expert_backward(u, idx, gate, e, (wg, wu, wd), E[e], dh)
        du[out["rows"]] += out["du_rows"]   # a token selects e at most once
        dE[e] = out["dE"]
        dW[e] = (out["dW_gate"], out["dW_up"], out["dW_down"])
    return dict(du=du, dE=dE, dW=dW, dWs=dWs, idx=idx, gate=gate)
