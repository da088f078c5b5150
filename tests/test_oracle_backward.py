"""Pins for the fp64 oracle of the layer backward (``oracle/backward.py``),
no GPU.

The backward oracle is the chain rule written out by hand.  It is trusted
only because it agrees with three things that share none of its formulas:

* central finite differences of the forward oracle (L = sum dh * h) on a
  tiny layer, for every input and weight element;
* torch.autograd (fp64, CPU) differentiating a plain torch restatement of
  the forward with the same selection;
* sympy's symbolic derivative of a one-token layer, evaluated exactly.

``test_mutant_*`` plant plausible mistakes in the oracle (monkeypatch, on
the CPU) and check that the finite-difference pin catches each one.
"""
import numpy as np
import pytest
import sympy
import torch

import oracle.backward as ob
import oracle.moe as om


def _tiny(seed=0, T=4, d=6, N=5, K=2, S=1, I=3):
    rng = np.random.default_rng(seed)
    u = rng.normal(size=(T, d))
    E = rng.normal(size=(N, d)) / np.sqrt(d)
    b = rng.uniform(-0.05, 0.05, size=N)
    routed = [(rng.normal(size=(I, d)) / np.sqrt(d),
               rng.normal(size=(I, d)) / np.sqrt(d),
               rng.normal(size=(d, I)) / np.sqrt(I)) for _ in range(N)]
    shared = [(rng.normal(size=(I, d)) / np.sqrt(d),
               rng.normal(size=(I, d)) / np.sqrt(d),
               rng.normal(size=(d, I)) / np.sqrt(I)) for _ in range(S)]
    dh = rng.normal(size=(T, d))
    return u, E, b, K, routed, shared, dh


def _loss(u, E, b, K, routed, shared, dh, idx_ref):
    h, r = om.layer_forward(u, E, b, K, lambda e: routed[e], shared)
    assert np.array_equal(r["idx"], idx_ref), "selection moved under eps"
    return float(np.sum(dh * h))


def _fd_check(seed=0, eps=1e-6, tol=1e-6):
    """Max relative deviation of the oracle's gradients from central
    differences, over every element of u, E and all weights."""
    u, E, b, K, routed, shared, dh = _tiny(seed)
    g = ob.layer_backward(u, E, b, K, lambda e: routed[e], shared, dh)
    idx = g["idx"]
    # the selection must not move within +-eps: margins far above eps
    s = om.affinity(u, E) + b
    srt = -np.sort(-s, axis=1)
    assert np.min(srt[:, K - 1] - srt[:, K]) > 1e3 * eps

    worst = 0.0

    def compare(arr, grad, name):
        nonlocal worst
        it = np.nditer(arr, flags=["multi_index"], op_flags=["readwrite"])
        for _ in it:
            i = it.multi_index
            v = arr[i]
            arr[i] = v + eps
            lp = _loss(u, E, b, K, routed, shared, dh, idx)
            arr[i] = v - eps
            lm = _loss(u, E, b, K, routed, shared, dh, idx)
            arr[i] = v
            fd = (lp - lm) / (2 * eps)
            err = abs(fd - grad[i]) / max(1.0, abs(fd))
            worst = max(worst, err)
            if err > tol:
                return f"{name}{i}: fd {fd} oracle {grad[i]}"
        return None

    msgs = [compare(u, g["du"], "du"), compare(E, g["dE"], "dE")]
    for e in range(len(routed)):
        for j, nm in enumerate(("dW_gate", "dW_up", "dW_down")):
            msgs.append(compare(routed[e][j], g["dW"][e][j], f"{nm}[{e}]"))
    for s_ in range(len(shared)):
        for j, nm in enumerate(("dWs_gate", "dWs_up", "dWs_down")):
            msgs.append(compare(shared[s_][j], g["dWs"][s_][j],
                                f"{nm}[{s_}]"))
    msgs = [m for m in msgs if m]
    return (not msgs), (msgs[0] if msgs else ""), worst


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_matches_finite_differences(seed):
    ok, msg, worst = _fd_check(seed)
    assert ok, msg
    assert worst < 1e-6


def _torch_forward(u, E, routed, shared, idx):
    """The layer forward restated with torch ops (fp64), selection fixed."""
    s = torch.sigmoid(u @ E.T)
    h = u.clone()
    for wg, wu, wd in shared:
        h = h + (torch.nn.functional.silu(u @ wg.T) * (u @ wu.T)) @ wd.T
    T, K = idx.shape
    for t in range(T):
        for k in range(K):
            e = int(idx[t, k])
            wg, wu, wd = routed[e]
            x = u[t:t + 1]
            y = (torch.nn.functional.silu(x @ wg.T) * (x @ wu.T)) @ wd.T
            h = h + torch.nn.functional.pad(
                s[t, e] * y, (0, 0, t, T - t - 1))
    return h


def test_backward_matches_torch_autograd():
    u, E, b, K, routed, shared, dh = _tiny(seed=5, T=24, d=16, N=8, K=3,
                                           S=2, I=8)
    g = ob.layer_backward(u, E, b, K, lambda e: routed[e], shared, dh)
    tt = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    ut, Et = tt(u), tt(E)
    rt = [tuple(tt(w) for w in ws) for ws in routed]
    st = [tuple(tt(w) for w in ws) for ws in shared]
    h = _torch_forward(ut, Et, rt, st, g["idx"])
    (h * torch.tensor(dh)).sum().backward()
    np.testing.assert_allclose(g["du"], ut.grad.numpy(), rtol=1e-10,
                               atol=1e-12)
    np.testing.assert_allclose(g["dE"], Et.grad.numpy(), rtol=1e-10,
                               atol=1e-12)
    for e in range(len(routed)):
        for j in range(3):
            got = g["dW"][e][j]
            want = rt[e][j].grad
            want = np.zeros_like(got) if want is None else want.numpy()
            np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)
    for s_ in range(len(shared)):
        for j in range(3):
            np.testing.assert_allclose(g["dWs"][s_][j], st[s_][j].grad.numpy(),
                                       rtol=1e-10, atol=1e-12)


def test_backward_matches_sympy_one_token():
    """One token, d = 2, two experts (top-1), one shared expert with I = 1:
    sympy differentiates the written-out h and is evaluated at rationals."""
    R = sympy.Rational
    u = sympy.symbols("u0 u1")
    e = [sympy.symbols(f"e{i}0 e{i}1") for i in range(2)]
    wg = [sympy.symbols(f"g{i}0 g{i}1") for i in range(3)]   # expert 2 = shared
    wu = [sympy.symbols(f"p{i}0 p{i}1") for i in range(3)]
    wd = [sympy.symbols(f"q{i}0 q{i}1") for i in range(3)]
    sig = lambda z: 1 / (1 + sympy.exp(-z))
    dot = lambda a, c: a[0] * c[0] + a[1] * c[1]

    def ffn(i):   # I = 1: W_gate, W_up are 1 x 2, W_down is 2 x 1
        a, c = dot(wg[i], u), dot(wu[i], u)
        hid = a * sig(a) * c
        return [wd[i][0] * hid, wd[i][1] * hid]

    vals = {u[0]: R(3, 5), u[1]: R(-2, 7),
            e[0][0]: R(1, 2), e[0][1]: R(1, 3), e[1][0]: R(-1, 4),
            e[1][1]: R(1, 5)}
    rng = np.random.default_rng(3)
    for i in range(3):
        for sym in (*wg[i], *wu[i], *wd[i]):
            vals[sym] = R(int(rng.integers(-9, 10)), 10)
    # expert 0 wins (s + b with b = 0): z0 = 0.3 - 2/21 > z1 = -0.15 - 2/35
    dh = (R(7, 10), R(-3, 10))
    y0, ys = ffn(0), ffn(2)
    h = [u[j] + ys[j] + sig(dot(u, e[0])) * y0[j] for j in range(2)]
    L = dh[0] * h[0] + dh[1] * h[1]

    num = {k: float(v) for k, v in vals.items()}
    u_np = np.array([[num[u[0]], num[u[1]]]])
    E_np = np.array([[num[s] for s in e[i]] for i in range(2)])
    W = [(np.array([[num[s] for s in wg[i]]]), np.array([[num[s] for s in wu[i]]]),
          np.array([[num[wd[i][0]]], [num[wd[i][1]]]])) for i in range(3)]
    g = ob.layer_backward(u_np, E_np, np.zeros(2), 1, lambda i: W[i], [W[2]],
                          np.array([[float(dh[0]), float(dh[1])]]))
    assert g["idx"].tolist() == [[0]]

    def sym_grad(sym):
        return float(sympy.N(sympy.diff(L, sym).subs(vals), 30))

    for j in range(2):
        assert abs(sym_grad(u[j]) - g["du"][0, j]) < 1e-13
        assert abs(sym_grad(e[0][j]) - g["dE"][0, j]) < 1e-13
        assert g["dE"][1, j] == 0.0
        assert abs(sym_grad(wg[0][j]) - g["dW"][0][0][0, j]) < 1e-13
        assert abs(sym_grad(wu[0][j]) - g["dW"][0][1][0, j]) < 1e-13
        assert abs(sym_grad(wd[0][j]) - g["dW"][0][2][j, 0]) < 1e-13
        assert abs(sym_grad(wg[2][j]) - g["dWs"][0][0][0, j]) < 1e-13
        assert abs(sym_grad(wu[2][j]) - g["dWs"][0][1][0, j]) < 1e-13
        assert abs(sym_grad(wd[2][j]) - g["dWs"][0][2][j, 0]) < 1e-13
    assert not any(np.any(w) for w in g["dW"][1])


def test_backward_zero_and_linear_in_dh():
    u, E, b, K, routed, shared, dh = _tiny(seed=2)
    run = lambda d_: ob.layer_backward(u, E, b, K, lambda e: routed[e],
                                       shared, d_)
    z = run(np.zeros_like(dh))
    assert not np.any(z["du"]) and not np.any(z["dE"])
    g1, g2, g3 = run(dh), run(2.0 * dh), run(dh + dh[::-1])
    g4 = run(dh[::-1].copy())
    np.testing.assert_allclose(g2["du"], 2 * g1["du"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g3["dE"], g1["dE"] + g4["dE"], rtol=1e-12,
                               atol=1e-14)
    for e in range(len(routed)):
        for j in range(3):
            np.testing.assert_allclose(g3["dW"][e][j],
                                       g1["dW"][e][j] + g4["dW"][e][j],
                                       rtol=1e-12, atol=1e-14)


# --- mutants: each plausible mistake must fail the finite-difference pin --

def _bad_silu_grad(a):
    sg = om.sigmoid(a)
    return sg                                   # dropped 1 + a (1 - sig)


def _bad_gate_backward(dh_rows, y, g):
    return np.sum(dh_rows * y, axis=1)          # dropped g (1 - g)


def test_mutant_silu_grad(monkeypatch):
    monkeypatch.setattr(ob, "silu_grad", _bad_silu_grad)
    assert not _fd_check(0)[0]


def test_mutant_gate_grad(monkeypatch):
    monkeypatch.setattr(ob, "gate_backward", _bad_gate_backward)
    assert not _fd_check(0)[0]


def test_mutant_misscaled_dy(monkeypatch):
    real = ob.swiglu_ffn_backward

    def misscaled(x, wg, wu, wd, dy):
        # mistake: the FFN sees its output gradient off by a factor (the
        # gate applied twice, or not at all, scales dy the same way)
        return real(x, wg, wu, wd, dy * 1.7)
    monkeypatch.setattr(ob, "swiglu_ffn_backward", misscaled)
    assert not _fd_check(0)[0]


def test_mutant_transposed_down_grad(monkeypatch):
    real = ob.swiglu_ffn_backward

    def swapped(x, wg, wu, wd, dy):
        dx, dWg, dWu, dWd, y = real(x, wg, wu, wd, dy)
        return dx, dWu, dWg, dWd, y             # gate and up swapped
    monkeypatch.setattr(ob, "swiglu_ffn_backward", swapped)
    assert not _fd_check(0)[0]
