"""Pins for the CPU fp64 oracle (no GPU).

The oracle is only trusted once it agrees with things other than itself:
hand-worked examples (``tests/golden``), library routines that compute the
same special case (scipy's expit, torch's silu / linear), brute force on tiny
inputs, closed forms and invariants.  The ``test_mutant_*`` tests plant
plausible mistakes in the oracle (on the CPU, via monkeypatch) and check that
a pin catches each one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle
import oracle.micro as micro
import oracle.moe as om
from moe_inputs import as_f64, generate, get_config

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _num(v, env):
    return float(eval(v, {"__builtins__": {}}, env)) if isinstance(v, str) \
        else float(v)


def _env():
    L = math.log(3.0)
    return {"L": L, "sig1": 1.0 / (1.0 + math.exp(-1.0)), "exp": math.exp}


# --- pin checks (return (ok, message)) -----------------------------------

def check_golden_routing():
    g = _load("routing_worked_example.json")
    env = _env()
    u = np.array([[_num(v, env) for v in row] for row in g["u"]])
    E = np.array(g["E"])
    s = om.affinity(u, E)
    if not np.allclose(s, np.array(g["s"]), rtol=0, atol=1e-15):
        return False, f"affinity {s}"
    for name, c in g["cases"].items():
        r = om.route(u, E, np.array(c["b"]), g["K"])
        if r["idx"].tolist() != c["idx"]:
            return False, f"{name}: idx {r['idx'].tolist()} != {c['idx']}"
        if not np.allclose(r["gate"], np.array(c["gate"]), rtol=0,
                           atol=1e-15):
            return False, f"{name}: gate {r['gate'].tolist()}"
        if r["counts"].tolist() != c["counts"]:
            return False, f"{name}: counts {r['counts'].tolist()}"
    return True, ""


def _golden_layer_inputs():
    g = _load("layer_worked_example.json")
    env = _env()
    u = np.array([[_num(v, env) for v in row] for row in g["u"]])
    E = np.array(g["E"])
    b = np.array(g["b"])
    routed = [tuple(np.array(w[k]) for k in ("w_gate", "w_up", "w_down"))
              for w in g["routed"]]
    shared = [tuple(np.array(w[k]) for k in ("w_gate", "w_up", "w_down"))
              for w in g["shared"]]
    h_exp = np.array([[_num(v, env) for v in row] for row in g["expected_h"]])
    return g, u, E, b, routed, shared, h_exp


def check_golden_layer():
    g, u, E, b, routed, shared, h_exp = _golden_layer_inputs()
    h, r = om.layer_forward(u, E, b, g["K"], lambda e: routed[e], shared)
    if r["idx"].tolist() != g["expected_idx"]:
        return False, f"idx {r['idx'].tolist()}"
    if not np.allclose(r["gate"], np.array(g["expected_gate"]), atol=1e-15,
                       rtol=0):
        return False, f"gate {r['gate'].tolist()}"
    if not np.allclose(h, h_exp, rtol=0, atol=1e-13):
        return False, f"h {h.tolist()} != {h_exp.tolist()}"
    # the same example through the step-by-step decomposition
    rr = om.route(u, E, b, g["K"])
    off, perm, inv = om.permute(rr["idx"], rr["counts"])
    y, ys = om.expert_ffn(u[perm], off, lambda e: routed[e], u, shared)
    h2 = om.combine(u, y, ys, inv, rr["gate"])
    if not np.allclose(h2, h_exp, rtol=0, atol=1e-13):
        return False, f"stepwise h {h2.tolist()}"
    return True, ""


def check_golden_bias():
    g = _load("bias_update_worked_example.json")

    def f32(hexs):
        return np.array([int(x, 16) for x in hexs], dtype=np.uint32) \
            .view(np.float32)
    for name, c in g["cases"].items():
        b = f32(c["b_hex"]) if "b_hex" in c else np.array(c["b"], np.float32)
        out = om.update_bias(b, np.array(g["counts"]), g["total_assign"],
                             c["gamma"])
        if out.dtype != np.float32:
            return False, "bias must stay float32"
        if "expected_hex" in c:
            got = [f"0x{v:08X}" for v in out.view(np.uint32).tolist()]
            if got != c["expected_hex"]:
                return False, f"{name}: {got} != {c['expected_hex']}"
        else:
            if out.tolist() != c["expected"]:
                return False, f"{name}: {out.tolist()}"
    return True, ""


def check_silu_vs_torch():
    a = np.linspace(-12, 12, 2001)
    ref = F.silu(torch.from_numpy(a)).numpy()
    got = om.silu(a)
    ok = np.allclose(got, ref, rtol=1e-14, atol=1e-300)
    return ok, "" if ok else f"max err {np.abs(got - ref).max()}"


def check_ffn_vs_torch(seed=0):
    rng = np.random.default_rng(seed)
    M, d, I = 5, 12, 7                       # non-square: a transposed
    x = rng.standard_normal((M, d))          # operand cannot pass
    wg = rng.standard_normal((I, d))
    wu = rng.standard_normal((I, d))
    wd = rng.standard_normal((d, I))
    t = torch.from_numpy
    ref = F.linear(F.silu(F.linear(t(x), t(wg))) * F.linear(t(x), t(wu)),
                   t(wd)).numpy()
    try:
        got = om.swiglu_ffn(x, wg, wu, wd)
    except ValueError as exc:                 # shape mismatch
        return False, str(exc)
    ok = got.shape == ref.shape and np.allclose(got, ref, rtol=1e-12,
                                                atol=1e-12)
    return ok, "" if ok else "swiglu mismatch"


def check_topk_bruteforce(T=64, N=16, K=4, seed=3):
    """Enumerate all C(N,K) subsets: the top-K set is the unique subset whose
    smallest biased score beats every score left out; it is also the subset
    with the largest score sum.  Scores drawn continuous, so ties have
    probability zero."""
    rng = np.random.default_rng(seed)
    s = scipy.special.expit(rng.standard_normal((T, N)))
    b = rng.uniform(-0.05, 0.05, N)
    idx, margin = om.biased_topk(s, b, K)
    beta = s + b
    subsets = list(itertools.combinations(range(N), K))
    for t in range(T):
        winners = [S for S in subsets
                   if min(beta[t, list(S)]) >
                   max(np.delete(beta[t], list(S)))]
        if len(winners) != 1:
            return False, f"token {t}: {len(winners)} dominating subsets"
        best_sum = max(subsets, key=lambda S: beta[t, list(S)].sum())
        if set(idx[t].tolist()) != set(winners[0]) or \
                set(best_sum) != set(winners[0]):
            return False, f"token {t}: {idx[t]} vs {winners[0]}"
        if not np.all(np.diff(beta[t, idx[t]]) <= 0):
            return False, f"token {t}: not sorted descending"
        rest = np.delete(beta[t], idx[t])
        if not math.isclose(margin[t], beta[t, idx[t][-1]] - rest.max(),
                            rel_tol=0, abs_tol=1e-15):
            return False, f"token {t}: margin"
    return True, ""


def check_ties_lowest_index():
    # E = 0: every affinity is exactly 1/2, selection follows the bias alone
    T, d, N, K = 3, 8, 6, 3
    u = np.random.default_rng(0).standard_normal((T, d))
    E = np.zeros((N, d))
    r = om.route(u, E, np.zeros(N), K)
    if r["idx"].tolist() != [[0, 1, 2]] * T:
        return False, f"b=0: {r['idx'].tolist()}"
    if not np.all(r["gate"] == 0.5):
        return False, "gate != 1/2"
    b = np.array([0.1, 0.3, 0.2, 0.3, -0.1, 0.2])
    r = om.route(u, E, b, K)
    if r["idx"].tolist() != [[1, 3, 2]] * T:
        return False, f"bias only: {r['idx'].tolist()}"
    return True, ""


def check_bias_sign_dynamics():
    """A skewed router with the +-gamma rule must move towards balance:
    with the sign flipped the imbalance grows."""
    rng = np.random.default_rng(7)
    T, d, N, K = 512, 32, 16, 2
    E = rng.standard_normal((N, d)) / math.sqrt(d)
    E *= (np.arange(1, N + 1) ** -1.1)[:, None]
    b = np.zeros(N, np.float32)
    first = last = None
    for step in range(40):
        u = rng.standard_normal((T, d))
        r = om.route(u, E, b, K)
        ml = om.relative_load(r["counts"], T * K).max()
        first = ml if first is None else first
        last = ml
        b = om.update_bias(b, r["counts"], T * K, 1e-2)
    ok = last < 0.6 * first
    return ok, "" if ok else f"max load {first:.2f} -> {last:.2f}"


def check_golden_group_routing():
    g = _load("group_routing_worked_example.json")
    beta = np.array(g["beta"])[None, :]
    s = beta.copy()
    b = np.zeros(beta.shape[1])
    for c in g["cases"]:
        idx, _ = om.group_limited_topk(s, b, c["K"], g["G"], g["M"])
        if idx[0].tolist() != c["idx"]:
            return False, f"K={c['K']}: {idx[0].tolist()}"
        if "ungrouped" in c:
            u_idx, _ = om.biased_topk(s, b, c["K"])
            if u_idx[0].tolist() != c["ungrouped"]:
                return False, "ungrouped"
    t = g["ties"]
    idx, _ = om.group_limited_topk(np.full_like(s, 0.5), b, t["K"], g["G"],
                                   g["M"])
    if idx[0].tolist() != t["idx"]:
        return False, f"ties: {idx[0].tolist()}"
    return True, ""


def check_group_bruteforce(T=40, N=12, G=4, M=2, K=3, seed=11):
    """Enumerate every choice of M groups: the kept groups are the unique set
    whose weakest group score beats every group left out, and the experts
    are the unique top-K of the pool of kept groups (continuous scores, no
    ties)."""
    rng = np.random.default_rng(seed)
    s = scipy.special.expit(rng.standard_normal((T, N)))
    b = rng.uniform(-0.05, 0.05, N)
    idx, _ = om.group_limited_topk(s, b, K, G, M)
    beta = s + b
    per = N // G
    for t in range(T):
        gsc = beta[t].reshape(G, per).max(axis=1)
        kept = [S for S in itertools.combinations(range(G), M)
                if min(gsc[list(S)]) > max(np.delete(gsc, list(S)))]
        if len(kept) != 1:
            return False, f"token {t}: {len(kept)} group sets"
        pool = [e for g_ in kept[0] for e in range(g_ * per, (g_ + 1) * per)]
        best = [S for S in itertools.combinations(pool, K)
                if min(beta[t, list(S)]) >
                max(beta[t, [e for e in pool if e not in S]])]
        if len(best) != 1 or set(best[0]) != set(idx[t].tolist()):
            return False, f"token {t}: {idx[t]} vs {best}"
    return True, ""


# --- the pins as tests ----------------------------------------------------

def test_golden_routing():
    ok, msg = check_golden_routing()
    assert ok, msg


def test_golden_layer():
    ok, msg = check_golden_layer()
    assert ok, msg


def test_golden_bias():
    ok, msg = check_golden_bias()
    assert ok, msg


def test_sigmoid_vs_scipy_expit():
    z = np.linspace(-30, 30, 4001)
    assert np.allclose(om.sigmoid(z), scipy.special.expit(z), rtol=1e-14,
                       atol=1e-300)
    assert om.sigmoid(0.0) == 0.5
    assert np.allclose(om.sigmoid(z) + om.sigmoid(-z), 1.0, atol=1e-15)


def test_silu_vs_torch():
    ok, msg = check_silu_vs_torch()
    assert ok, msg


def test_swiglu_vs_torch_linear():
    ok, msg = check_ffn_vs_torch()
    assert ok, msg


def test_topk_bruteforce():
    ok, msg = check_topk_bruteforce()
    assert ok, msg


def test_ties_lowest_index():
    ok, msg = check_ties_lowest_index()
    assert ok, msg


def test_bias_moves_towards_balance():
    ok, msg = check_bias_sign_dynamics()
    assert ok, msg


def test_bias_step_is_plus_minus_gamma_or_zero():
    rng = np.random.default_rng(1)
    N, TK = 64, 64 * 6
    g32 = np.float32(1e-3)
    for _ in range(20):
        counts = rng.multinomial(TK, np.ones(N) / N)
        out = om.update_bias(np.zeros(N, np.float32), counts, TK, 1e-3)
        want = np.where(counts * N > TK, -g32,
                        np.where(counts * N < TK, g32, np.float32(0)))
        assert out.tobytes() == want.astype(np.float32).tobytes()


def test_relative_load():
    c = np.array([4, 2, 2, 0])
    assert om.relative_load(c, 8).tolist() == [2.0, 1.0, 1.0, 0.0]


def _tiny_layer(cfg_name="tiny", **over):
    cfg = get_config(cfg_name).with_(**over)
    t = generate(cfg, "cpu")
    u, E, b = as_f64(t["u"]), as_f64(t["E"]), as_f64(t["b"])
    wg, wu, wd = (as_f64(t[k]) for k in ("w_gate", "w_up", "w_down"))
    sg, su, sd = (as_f64(t[k]) for k in ("ws_gate", "ws_up", "ws_down"))
    routed = lambda e: (wg[e], wu[e], wd[e])      # noqa: E731
    shared = [(sg[s], su[s], sd[s]) for s in range(cfg.n_shared)]
    return cfg, u, E, b, routed, shared


def test_route_invariants():
    for cfg in (get_config("tiny"), get_config("mid").with_(T=512)):
        t = generate(cfg, "cpu", experts=False)
        u, E, b = as_f64(t["u"]), as_f64(t["E"]), as_f64(t["b"])
        r = om.route(u, E, b, cfg.top_k)
        idx = r["idx"]
        assert idx.shape == (cfg.T, cfg.top_k)
        assert all(len(set(row)) == cfg.top_k for row in idx.tolist())
        assert r["counts"].sum() == cfg.T * cfg.top_k
        assert np.array_equal(r["counts"],
                              np.bincount(idx.ravel(), minlength=cfg.n_routed))
        assert np.array_equal(r["gate"],
                              r["s"][np.arange(cfg.T)[:, None], idx])
        assert np.all((r["gate"] > 0) & (r["gate"] < 1))


def test_permute_vs_lexsort():
    cfg, u, E, b, _, _ = _tiny_layer()
    r = om.route(u, E, b, cfg.top_k)
    off, perm, inv = om.permute(r["idx"], r["counts"])
    T, K = r["idx"].shape
    t_flat = np.repeat(np.arange(T), K)
    e_flat = r["idx"].ravel()
    order = np.lexsort((t_flat, e_flat))        # by expert, then token
    assert np.array_equal(perm, t_flat[order])
    inv_alt = np.empty(T * K, np.int64)
    inv_alt[order] = np.arange(T * K)
    assert np.array_equal(inv.ravel(), inv_alt)
    assert off[0] == 0 and off[-1] == T * K
    for e in range(cfg.n_routed):
        seg = perm[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)         # stable, distinct tokens
        assert np.all((r["idx"][seg] == e).any(axis=1))


def test_stepwise_equals_definition():
    cfg, u, E, b, routed, shared = _tiny_layer()
    h, r = om.layer_forward(u, E, b, cfg.top_k, routed, shared)
    rr = om.route(u, E, b, cfg.top_k)
    off, perm, inv = om.permute(rr["idx"], rr["counts"])
    y, ys = om.expert_ffn(u[perm], off, routed, u, shared)
    h2 = om.combine(u, y, ys, inv, rr["gate"])
    assert np.allclose(h, h2, rtol=0, atol=1e-12)


def test_micro_oracle_matches():
    cfg, u, E, b, routed, shared = _tiny_layer()
    n = 6
    tolist = lambda a: a.tolist()                # noqa: E731
    R = [tuple(map(tolist, routed(e))) for e in range(cfg.n_routed)]
    S = [tuple(map(tolist, w)) for w in shared]
    Hm, IDXm = micro.layer(u[:n].tolist(), E.tolist(), b.tolist(), cfg.top_k,
                           R, S)
    h, r = om.layer_forward(u[:n], E, b, cfg.top_k, routed, shared)
    assert r["idx"].tolist() == IDXm
    assert np.allclose(h, np.array(Hm), rtol=0, atol=1e-12)


def test_single_expert_reduces_to_ffn():
    rng = np.random.default_rng(5)
    T, d, I = 7, 10, 6
    u = rng.standard_normal((T, d))
    E = rng.standard_normal((1, d))
    w = (rng.standard_normal((I, d)), rng.standard_normal((I, d)),
         rng.standard_normal((d, I)))
    h, _ = om.layer_forward(u, E, np.zeros(1), 1, lambda e: w, ())
    t = torch.from_numpy
    ffn = F.linear(F.silu(F.linear(t(u), t(w[0]))) * F.linear(t(u), t(w[1])),
                   t(w[2])).numpy()
    g = scipy.special.expit(u @ E[0])
    assert np.allclose(h, u + g[:, None] * ffn, rtol=1e-12, atol=1e-12)


def test_dense_mixture_all_experts():
    cfg, u, E, b, routed, shared = _tiny_layer(T=16)
    N = cfg.n_routed
    h, _ = om.layer_forward(u, E, b, N, routed, shared)
    t = torch.from_numpy
    s = scipy.special.expit(u @ E.T)
    ref = u.copy()
    for w in shared:
        ref += F.linear(F.silu(F.linear(t(u), t(w[0]))) *
                        F.linear(t(u), t(w[1])), t(w[2])).numpy()
    for e in range(N):
        w = routed(e)
        ref += s[:, e:e + 1] * F.linear(F.silu(F.linear(t(u), t(w[0]))) *
                                        F.linear(t(u), t(w[1])),
                                        t(w[2])).numpy()
    assert np.allclose(h, ref, rtol=1e-12, atol=1e-12)


def test_zero_weights_identity():
    cfg, u, E, b, routed, shared = _tiny_layer(T=16)
    z = lambda e: tuple(np.zeros_like(x) for x in routed(e))   # noqa: E731
    zs = [tuple(np.zeros_like(x) for x in w) for w in shared]
    h, _ = om.layer_forward(u, E, b, cfg.top_k, z, zs)
    assert np.array_equal(h, u)


def test_down_projection_linearity():
    cfg, u, E, b, routed, shared = _tiny_layer(T=16)
    a = 2.5
    sc = lambda e: (routed(e)[0], routed(e)[1], a * routed(e)[2])  # noqa
    ss = [(w[0], w[1], a * w[2]) for w in shared]
    h1, _ = om.layer_forward(u, E, b, cfg.top_k, routed, shared)
    h2, _ = om.layer_forward(u, E, b, cfg.top_k, sc, ss)
    assert np.allclose(h2 - u, a * (h1 - u), rtol=1e-12, atol=1e-12)


def test_token_permutation_equivariance():
    cfg, u, E, b, routed, shared = _tiny_layer(T=32)
    p = np.random.default_rng(2).permutation(u.shape[0])
    h1, r1 = om.layer_forward(u, E, b, cfg.top_k, routed, shared)
    h2, r2 = om.layer_forward(u[p], E, b, cfg.top_k, routed, shared)
    assert np.array_equal(r2["idx"], r1["idx"][p])
    assert np.allclose(h2, h1[p], rtol=0, atol=1e-12)


def test_token_subset_matches_full():
    cfg, u, E, b, routed, shared = _tiny_layer(T=32)
    sel = np.array([3, 0, 17, 31])
    h1, r1 = om.layer_forward(u, E, b, cfg.top_k, routed, shared)
    h2, r2 = om.layer_forward(u, E, b, cfg.top_k, routed, shared, tokens=sel)
    assert np.array_equal(r2["idx"], r1["idx"][sel])
    assert np.allclose(h2, h1[sel], rtol=0, atol=1e-12)


def test_near_tie_acceptance():
    s = np.array([0.9, 0.5, 0.5 + 2e-6, 0.1])
    b = np.zeros(4)
    assert oracle.topk_near_tie_ok(s, b, [0, 2], 2)
    assert oracle.topk_near_tie_ok(s, b, [0, 1], 2)      # within 1e-5
    assert not oracle.topk_near_tie_ok(s, b, [0, 3], 2)
    assert not oracle.topk_near_tie_ok(s, b, [0, 0], 2)


# --- planted mistakes: each must be caught by a pin -----------------------

def _mut_gate_from_biased(monkeypatch):
    orig = om.route

    def route(u, E, b, K):
        r = orig(u, E, b, K)
        r["gate"] = r["gate"] + np.asarray(b)[r["idx"]]
        return r
    monkeypatch.setattr(om, "route", route)


def _mut_select_unbiased(monkeypatch):
    orig = om.biased_topk
    monkeypatch.setattr(om, "biased_topk",
                        lambda s, b, K: orig(s, np.zeros_like(b), K))


def _mut_tie_highest_index(monkeypatch):
    def biased_topk(s, b, K):
        beta = np.asarray(s, float) + np.asarray(b, float)[None, :]
        rev = beta[:, ::-1]
        order = beta.shape[1] - 1 - np.argsort(-rev, axis=1, kind="stable")
        idx = order[:, :K]
        return idx, np.zeros(beta.shape[0])
    monkeypatch.setattr(om, "biased_topk", biased_topk)


def _mut_drop_shared(monkeypatch):
    orig = om.layer_forward
    monkeypatch.setattr(om, "layer_forward",
                        lambda u, E, b, K, routed, shared=(), **kw:
                        orig(u, E, b, K, routed, (), **kw))


def _mut_bias_sign(monkeypatch):
    orig = om.update_bias
    monkeypatch.setattr(om, "update_bias",
                        lambda b, c, TK, gamma=1e-3: orig(b, c, TK, -gamma))


def _mut_down_transposed(monkeypatch):
    def swiglu_ffn(x, wg, wu, wd):
        x = np.asarray(x, float)
        return (om.silu(x @ np.asarray(wg).T) * (x @ np.asarray(wu).T)) @ \
            np.asarray(wd)
    monkeypatch.setattr(om, "swiglu_ffn", swiglu_ffn)


def _mut_silu_sign(monkeypatch):
    monkeypatch.setattr(om, "silu",
                        lambda a: np.asarray(a, float) *
                        om.sigmoid(-np.asarray(a, float)))


def _mut_overload_threshold(monkeypatch):
    # compares with T*K instead of the balanced load T*K/N
    def update_bias(b, counts, total_assign, gamma=1e-3):
        b32 = np.asarray(b, np.float32).copy()
        c = np.asarray(counts)
        g = np.float32(gamma)
        b32[c > total_assign] -= g
        b32[c < total_assign] += g
        return b32
    monkeypatch.setattr(om, "update_bias", update_bias)


MUTANTS = {
    "gate_from_biased": (_mut_gate_from_biased, [check_golden_routing]),
    "select_unbiased": (_mut_select_unbiased, [check_golden_routing]),
    "tie_highest_index": (_mut_tie_highest_index, [check_golden_routing,
                                                   check_ties_lowest_index]),
    "drop_shared": (_mut_drop_shared, [check_golden_layer]),
    "bias_sign": (_mut_bias_sign, [check_golden_bias,
                                   check_bias_sign_dynamics]),
    "overload_threshold": (_mut_overload_threshold, [check_golden_bias]),
    "down_transposed": (_mut_down_transposed, [check_ffn_vs_torch]),
    "silu_sign": (_mut_silu_sign, [check_silu_vs_torch, check_golden_layer]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    plant, checks = MUTANTS[name]
    plant(monkeypatch)
    for chk in checks:
        try:
            ok, _ = chk()
        except Exception:          # a crash also counts as caught
            ok = False
        assert not ok, f"pin {chk.__name__} missed mutant {name}"


def test_golden_group_routing():
    ok, msg = check_golden_group_routing()
    assert ok, msg


def test_group_routing_bruteforce():
    ok, msg = check_group_bruteforce()
    assert ok, msg


def test_group_routing_reduces_to_plain():
    """M = G keeps every group: plain routing.  G = N and M = K: each expert
    is its own group, so the kept groups are the plain top-K experts."""
    rng = np.random.default_rng(4)
    s = scipy.special.expit(rng.standard_normal((50, 16)))
    b = rng.uniform(-0.02, 0.02, 16)
    plain, _ = om.biased_topk(s, b, 4)
    a, _ = om.group_limited_topk(s, b, 4, 4, 4)
    c, _ = om.group_limited_topk(s, b, 4, 16, 4)
    assert np.array_equal(a, plain) and np.array_equal(c, plain)


def test_group_near_tie_check():
    beta = np.array([0.70, 0.69, 0.20, 0.95, 0.90, 0.85, 0.10, 0.60])
    z = np.zeros(8)
    assert om.group_topk_near_tie_ok(beta, z, [3, 4], 2, 4, 2)
    assert not om.group_topk_near_tie_ok(beta, z, [3, 0], 2, 4, 2)
    tied = beta.copy()
    tied[0] = 0.90 - 2e-6          # group 0 now ties group 2 within 1e-5
    assert om.group_topk_near_tie_ok(tied, z, [3, 0], 2, 4, 2)


def _mut_group_score_sum(monkeypatch):
    def glt(s, b, K, G, M):
        beta = np.asarray(s, float) + np.asarray(b, float)[None, :]
        T, N = beta.shape
        per = N // G
        gscore = beta.reshape(T, G, per).sum(axis=2)      # wrong rule
        gorder = np.argsort(-gscore, axis=1, kind="stable")[:, :M]
        el = np.zeros((T, G), bool)
        np.put_along_axis(el, gorder, True, axis=1)
        masked = np.where(np.repeat(el, per, axis=1), beta, -np.inf)
        return np.argsort(-masked, axis=1, kind="stable")[:, :K], None
    monkeypatch.setattr(om, "group_limited_topk", glt)


def test_mutant_group_score_caught(monkeypatch):
    _mut_group_score_sum(monkeypatch)
    ok, _ = check_golden_group_routing()
    assert not ok
