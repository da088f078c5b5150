"""Plain fp64 CPU oracle of the DeepSeekMoE layer forward and bias update.

TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU
baseline call this; the product path never does.

Sources (web pages summarising the DeepSeek-V3 technical report, cited by
title and section):

* [V3-paper-notes] "【推理llm論文精讀】DeepSeek V3技術論文" (hk.pswp.cn),
  section 2.2 "DeepSeekMoE": the FFN-output equation
  h_t = u_t + sum_{i<=N_s} FFN^(s)_i(u_t) + sum_{i<=N_r} g_{i,t} FFN^(r)_i(u_t);
  the routing-weight equation g_{i,t} = s_{i,t} if s_{i,t} is among the
  Top-K_r, else 0; the affinity equation s_{i,t} = Sigmoid(u_t . e_i); the
  auxiliary-loss-free paragraph (a bias b_i is added to s_{i,t} to decide the
  top-K; b_i is lowered for an overloaded expert and raised for an
  underloaded one during training).
* [lineage] "解码DeepSeek创新之道：三代模型演进路线图" (10100.com), V3 part,
  auxiliary-loss-free bullet: the bias is used only for routing selection.
* [tech-reveal] "AI新顶流-DeepSeek 技术大揭秘" (blog.csdn.net), section
  "无辅助损失的负载均衡策略": load is monitored over all batches of a step and
  the adjustment happens at the end of each step.
* [report-commentary] DeepSeek-V3 technical-report commentary
  (cooktownmusic.com), Fig. 9 caption: relative expert load = actual load /
  theoretically balanced load.

Readings where the pages are silent (each one is listed with its reason in
the project's design notes):

* expert FFN form: SwiGLU, FFN(x) = W_down (SiLU(W_gate x) * (W_up x)) with
  SiLU(a) = a * Sigmoid(a) -- the pages give no FFN form;
* gate: g = s at the selected experts, no renormalisation (the equation as
  printed);
* top-K ties: the lowest expert index wins;
* overloaded / underloaded: compared with the balanced load T*K/N, done as
  the exact integer test c_i*N vs T*K; equal load leaves b_i unchanged;
* bias step: b_i <- fl32(b_i -/+ gamma), one float32 rounding, bias held in
  float32;
* shared experts: weight 1, plain sum.

Everything here is float64 except the bias update, which the bias's own
storage type (float32) fixes.  Library primitives used as single steps:
numpy matmul, exp, argsort (stable), bincount, cumsum.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np

Weights = Tuple[np.ndarray, np.ndarray, np.ndarray]   # (W_gate, W_up, W_down)


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# --- affinity ------------------------------------------------------------

def sigmoid(z):
    """Sigmoid(z) = 1 / (1 + exp(-z)), fp64."""
    z = _f64(z)
    return 1.0 / (1.0 + np.exp(-z))


def silu(a):
    """SiLU(a) = a * Sigmoid(a), fp64 (the FFN form is a reading: SwiGLU)."""
    a = _f64(a)
    return a * sigmoid(a)


def affinity(u, E) -> np.ndarray:
    """s[t, i] = Sigmoid(u_t . e_i)  ([V3-paper-notes] 2.2, affinity eq.).

    u: [T, d], E: [N_r, d] (row i is centroid e_i) -> s: [T, N_r], fp64.
    """
    z = _f64(u) @ _f64(E).T
    return sigmoid(z)


# --- selection -----------------------------------------------------------

def biased_topk(s, b, K: int):
    """Top-K_r experts per token by s + b, lowest index first among ties.

    [V3-paper-notes] 2.2 auxiliary-loss-free paragraph: the bias is added to
    the affinity to decide the top-K; [lineage]: the bias only selects.

    Returns (idx [T, K] int64 sorted by (s+b desc, index asc), margin [T]),
    where margin = beta_(K) - beta_(K+1) (inf when K == N_r), the distance
    between the last selected and the first unselected biased score.
    """
    s = _f64(s)
    beta = s + _f64(b)[None, :]
    T, N = beta.shape
    if not 1 <= K <= N:
        raise ValueError("need 1 <= K <= N_r")
    # a stable sort of -beta keeps equal scores in ascending index order
    order = np.argsort(-beta, axis=1, kind="stable")
    idx = order[:, :K]
    if K < N:
        rows = np.arange(T)
        margin = beta[rows, order[:, K - 1]] - beta[rows, order[:, K]]
    else:
        margin = np.full(T, np.inf)
    return idx.astype(np.int64), margin


def group_limited_topk(s, b, K: int, G: int, M: int):
    """Top-K_r experts restricted to the M best of G expert groups.

    [report-commentary], training-framework paragraph: each token is sent to
    at most 4 nodes; [lineage], V3 part: node-limited routing.  The pages
    give no group-score rule; the reading taken here: experts form G
    contiguous groups of N/G; a group's score is the largest biased score
    s + b among its experts; the M groups with the highest score are kept
    (lower group index first on ties); the top-K of s + b is then taken
    among the experts of the kept groups only (lower index first on ties).

    Returns (idx [T, K] sorted by (s+b desc, index asc), margin [T]) with
    margin the smaller of the gap between the K-th and (K+1)-th eligible
    biased scores and the gap between the M-th and (M+1)-th group scores
    (either gap being tiny makes the selection fragile under rounding).
    """
    s = _f64(s)
    beta = s + _f64(b)[None, :]
    T, N = beta.shape
    if G < 1 or N % G != 0 or not 1 <= M <= G:
        raise ValueError("need N % G == 0 and 1 <= M <= G")
    per = N // G
    if K > M * per:
        raise ValueError("K larger than the experts of the kept groups")
    gscore = beta.reshape(T, G, per).max(axis=2)
    gorder = np.argsort(-gscore, axis=1, kind="stable")[:, :M]
    eligible = np.zeros((T, G), dtype=bool)
    np.put_along_axis(eligible, gorder, True, axis=1)
    masked = np.where(np.repeat(eligible, per, axis=1), beta, -np.inf)
    order = np.argsort(-masked, axis=1, kind="stable")
    idx = order[:, :K]
    rows = np.arange(T)
    if K < M * per:
        margin = masked[rows, order[:, K - 1]] - masked[rows, order[:, K]]
    else:
        margin = np.full(T, np.inf)
    if M < G:
        gs = -np.sort(-gscore, axis=1)
        margin = np.minimum(margin, gs[:, M - 1] - gs[:, M])
    return idx.astype(np.int64), margin


def group_topk_near_tie_ok(s, b, idx_sel, K: int, G: int, M: int,
                           tol: float = 1e-5) -> bool:
    """True when ``idx_sel`` is a valid group-limited top-K of s+b up to
    ``tol``: distinct experts from at most M groups, each of those groups
    scoring within tol of the M-th best group score, and the selection a
    valid top-K (within tol) among the experts of the groups it uses plus
    every group that scores above the M-th best by more than tol."""
    beta = _f64(s) + _f64(b)
    sel = np.asarray(idx_sel)
    N = beta.size
    per = N // G
    if len(set(sel.tolist())) != K:
        return False
    gscore = beta.reshape(G, per).max(axis=1)
    gth = np.sort(gscore)[::-1][M - 1]
    used = set((sel // per).tolist())
    if len(used) > M or any(gscore[g] < gth - tol for g in used):
        return False
    sure = {g for g in range(G) if gscore[g] > gth + tol}
    if not sure <= used and len(sure | used) > M:
        return False
    pool = sorted(used | sure)
    elig = np.concatenate([np.arange(g * per, (g + 1) * per) for g in pool])
    sub = beta[elig]
    pos = {int(e): i for i, e in enumerate(elig)}
    return topk_near_tie_ok(sub, np.zeros_like(sub),
                            [pos[int(e)] for e in sel], K, tol)


def route(u, E, b, K: int, groups=None):
    """Routing of [V3-paper-notes] 2.2: affinity, biased top-K, gate, load.

    Returns dict with s [T,N], idx [T,K], gate [T,K] (= s at idx, never s+b),
    counts [N] (tokens per expert over the whole batch) and margin [T].
    ``groups=(G, M)`` selects the group-limited variant.
    """
    s = affinity(u, E)
    if groups is None:
        idx, margin = biased_topk(s, b, K)
    else:
        idx, margin = group_limited_topk(s, b, K, *groups)
    gate = np.take_along_axis(s, idx, axis=1)
    counts = np.bincount(idx.ravel(), minlength=s.shape[1]).astype(np.int64)
    return {"s": s, "idx": idx, "gate": gate, "counts": counts,
            "margin": margin}


def topk_near_tie_ok(s, b, idx_sel, K: int, tol: float = 1e-5) -> bool:
    """True when ``idx_sel`` is a valid top-K of s+b up to ``tol``.

    Used for tokens whose top-K is not unique under fp32 rounding: every
    selected biased score must be >= beta_(K) - tol and every unselected one
    <= beta_(K+1) + tol, and the K indices must be distinct.
    """
    beta = _f64(s) + _f64(b)
    sel = np.asarray(idx_sel)
    if len(set(sel.tolist())) != K:
        return False
    srt = np.sort(beta)[::-1]
    kth = srt[K - 1]
    nxt = srt[K] if K < beta.size else -np.inf
    mask = np.zeros(beta.size, dtype=bool)
    mask[sel] = True
    return bool(np.all(beta[mask] >= kth - tol) and
                np.all(beta[~mask] <= nxt + tol))


# --- expert FFN ----------------------------------------------------------

def swiglu_ffn(x, w_gate, w_up, w_down) -> np.ndarray:
    """FFN(x) = W_down (SiLU(W_gate x) * (W_up x)) for rows x [M, d].

    w_gate, w_up: [I, d]; w_down: [d, I].  Returns [M, d] fp64.
    """
    x = _f64(x)
    a = x @ _f64(w_gate).T            # [M, I]
    c = x @ _f64(w_up).T              # [M, I]
    return (silu(a) * c) @ _f64(w_down).T


# --- dispatch / FFN / combine, step by step ------------------------------

def permute(idx, counts):
    """Expert-contiguous order of the (token, k) assignments.

    offsets = exclusive prefix sum of counts (length N+1).  Within expert e
    the assignments keep ascending token order (stable).  perm[slot] = the
    token whose row fills ``slot``; inv[t, k] = the slot of assignment
    (t, k).  Plain loop over tokens in order.
    """
    idx = np.asarray(idx)
    counts = np.asarray(counts, dtype=np.int64)
    T, K = idx.shape
    offsets = np.zeros(counts.size + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    nxt = offsets[:-1].copy()
    perm = np.empty(T * K, dtype=np.int64)
    inv = np.empty((T, K), dtype=np.int64)
    for t in range(T):
        for k in range(K):
            e = idx[t, k]
            inv[t, k] = nxt[e]
            perm[nxt[e]] = t
            nxt[e] += 1
    return offsets, perm, inv


def expert_ffn(x_perm, offsets, routed: Callable[[int], Weights],
               u=None, shared: Sequence[Weights] = ()):
    """y_perm[rows of e] = FFN^(r)_e(x_perm[rows of e]) for every expert e;
    y_shared = sum_s FFN^(s)_s(u) (0 when there are no shared experts).

    ``routed(e)`` returns expert e's (W_gate, W_up, W_down).
    """
    x_perm = _f64(x_perm)
    offsets = np.asarray(offsets)
    y = np.zeros_like(x_perm)
    for e in range(offsets.size - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            y[lo:hi] = swiglu_ffn(x_perm[lo:hi], *routed(e))
    ys = None
    if u is not None:
        u = _f64(u)
        ys = np.zeros_like(u)
        for w in shared:
            ys += swiglu_ffn(u, *w)
    return y, ys


def combine(u, y_perm, y_shared, inv, gate) -> np.ndarray:
    """h_t = u_t + y_shared_t + sum_k gate[t,k] * y_perm[inv[t,k]]
    ([V3-paper-notes] 2.2, FFN-output equation, with the routed sum taken
    over the selected experts only, since g is zero elsewhere)."""
    h = _f64(u).copy()
    if y_shared is not None:
        h += _f64(y_shared)
    y_perm = _f64(y_perm)
    inv = np.asarray(inv)
    gate = _f64(gate)
    for k in range(inv.shape[1]):
        h += gate[:, k:k + 1] * y_perm[inv[:, k]]
    return h


# --- whole layer, by the definition --------------------------------------

def layer_forward(u, E, b, K: int, routed: Callable[[int], Weights],
                  shared: Sequence[Weights] = (),
                  idx_override: Optional[np.ndarray] = None,
                  tokens: Optional[np.ndarray] = None, groups=None):
    """h = u + sum_s FFN^(s)(u) + sum_i g_i FFN^(r)_i(u), by the definition.

    No permutation buffer: for each expert, the tokens that selected it are
    pushed through its FFN and added with their gate.  ``idx_override``
    replaces the selection (used to recompute h on another valid top-K of a
    near-tied token); the gate is then s at those experts.  ``tokens``
    restricts the output to a subset of rows (sampled checks at full size):
    routing is still computed for those rows only, since it is per token.
    ``groups=(G, M)`` routes by the group-limited rule.
    Returns (h, routing dict).
    """
    u = _f64(u)
    if tokens is not None:
        u = u[np.asarray(tokens)]
    r = route(u, E, b, K, groups)
    idx = r["idx"] if idx_override is None else np.asarray(idx_override)
    gate = np.take_along_axis(r["s"], idx, axis=1)
    h = u.copy()
    for w in shared:
        h += swiglu_ffn(u, *w)
    for e in np.unique(idx):
        rows, ks = np.nonzero(idx == e)
        h[rows] += gate[rows, ks][:, None] * swiglu_ffn(u[rows], *routed(int(e)))
    r = dict(r, idx=idx, gate=gate)
    return h, r


# --- bias update ---------------------------------------------------------

def update_bias(b, counts, total_assign: int, gamma: float = 1e-3):
    """Auxiliary-loss-free bias step after a batch ([V3-paper-notes] 2.2:
    lower b_i when expert i is overloaded, raise it when underloaded;
    [tech-reveal]: counts over the whole step).

    Overloaded means counts[i] * N > T*K (above the balanced load T*K/N);
    underloaded means counts[i] * N < T*K.  Done in float32 arithmetic,
    because the bias is stored in float32: b_i <- fl32(b_i - gamma) or
    fl32(b_i + gamma), with gamma rounded to float32 first.
    """
    b32 = np.asarray(b, dtype=np.float32).copy()
    c = np.asarray(counts, dtype=np.int64)
    N = c.size
    g32 = np.float32(gamma)
    over = c * N > int(total_assign)
    under = c * N < int(total_assign)
    b32[over] = b32[over] - g32
    b32[under] = b32[under] + g32
    return b32


def relative_load(counts, total_assign: int) -> np.ndarray:
    """counts[i] / (T*K/N): actual over balanced load ([report-commentary]
    Fig. 9 caption)."""
    c = np.asarray(counts, dtype=np.float64)
    return c / (float(total_assign) / c.size)
