"""Helpers shared by the GPU parity tests: setting up a workload on the
device, running the oracle on the same (rounded) inputs, and the comparison
rules.

Comparison rules (the layer's acceptance bar):
* routing indices and per-expert counts bit-exact, except tokens whose fp64
  margin beta_(K) - beta_(K+1) is below 1e-5: those are counted, and their
  GPU selection must be a valid top-K within 1e-5;
* outputs within max-abs 2e-2 and relative Frobenius 5e-3 (bf16 inputs,
  fp32 accumulation);
* bias vectors bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.moe as om
from moe_inputs import as_f64, generate

NEAR_TIE = 1e-5
MAX_ABS = 2e-2
REL_FRO = 5e-3
# gradients of the backward pass: the relative bar unchanged, the absolute
# one scaled to the tensor's largest entry
GRAD_REL_FRO = 5e-3
GRAD_MAX_ABS_FRAC = 1e-2


def grad_max_abs(ref) -> float:
    """max|err| allowed for a gradient tensor: max(2e-2, 1% of max|ref|)."""
    ref = np.asarray(ref, dtype=np.float64)
    top = float(np.abs(ref).max()) if ref.size else 0.0
    return max(MAX_ABS, GRAD_MAX_ABS_FRAC * top)


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def to_dev(t: dict, device="cuda"):
    return {k: v.to(device) for k, v in t.items()}


def make_inputs(cfg, device="cuda"):
    """Seeded inputs, drawn on the CPU for small workloads and on the device
    for large ones (the draw itself is deterministic either way)."""
    big = cfg.n_routed * cfg.d * cfg.d_ff > 64 * 2048 * 2048
    if big:
        return generate(cfg, device)
    return to_dev(generate(cfg, "cpu"), device)


def oracle_weights(t: dict):
    """Lazy per-expert fp64 weights (exact widening) for the oracle."""
    cache = {}

    def routed(e):
        if e not in cache:
            cache.clear()   # one expert at a time keeps host memory small
            cache[e] = tuple(as_f64(t[k][e]) for k in
                             ("w_gate", "w_up", "w_down"))
        return cache[e]
    shared = [tuple(as_f64(t[k][s]) for k in ("ws_gate", "ws_up", "ws_down"))
              for s in range(t["ws_gate"].shape[0])]
    return routed, shared


def check_routing(r, b64, idx_gpu, counts_gpu, K, rows=None, groups=None):
    """Returns the number of near-tied tokens; asserts the rules above.
    ``groups=(G, M)``: ``r`` comes from group-limited routing, and a
    near-tied token is checked against the group-limited rule."""
    idx_gpu = np.asarray(idx_gpu)
    s = r["s"]
    near = r["margin"] < NEAR_TIE
    ok = ~near
    # the selected set is unique away from near-ties ...
    np.testing.assert_array_equal(np.sort(idx_gpu[ok], axis=1),
                                  np.sort(r["idx"][ok], axis=1))
    # ... and so is its order (s+b descending) wherever consecutive selected
    # scores are further apart than the near-tie threshold
    beta = s + np.asarray(b64)[None, :]
    sel_beta = np.take_along_axis(beta, r["idx"], axis=1)
    gaps = -np.diff(sel_beta, axis=1)
    ordered = ok & (gaps.min(axis=1, initial=np.inf) >= NEAR_TIE)
    np.testing.assert_array_equal(idx_gpu[ordered], r["idx"][ordered])
    for t in np.nonzero(near)[0]:
        if groups is None:
            assert om.topk_near_tie_ok(s[t], b64, idx_gpu[t], K, NEAR_TIE), t
        else:
            assert om.group_topk_near_tie_ok(s[t], b64, idx_gpu[t], K,
                                             *groups, NEAR_TIE), t
    # counts: consistent with the GPU's own selection, and with the oracle's
    # on every token that is not near-tied
    N = s.shape[1]
    if counts_gpu is not None:
        np.testing.assert_array_equal(
            np.asarray(counts_gpu),
            np.bincount(idx_gpu.ravel(), minlength=N))
        if not near.any():
            np.testing.assert_array_equal(np.asarray(counts_gpu), r["counts"])
    np.testing.assert_array_equal(
        np.bincount(idx_gpu[ok].ravel(), minlength=N),
        np.bincount(r["idx"][ok].ravel(), minlength=N))
    return int(near.sum())


def errors(got, ref, base=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = got - ref
    out = {"max_abs": float(np.abs(diff).max()) if diff.size else 0.0,
           "rel_fro": float(np.linalg.norm(diff) /
                            max(np.linalg.norm(ref), 1e-30))}
    if base is not None:
        dm = ref - np.asarray(base, dtype=np.float64)
        out["rel_fro_moe"] = float(np.linalg.norm(diff) /
                                   max(np.linalg.norm(dm), 1e-30))
    return out


def assert_close(got, ref, base=None, max_abs=MAX_ABS, rel_fro=REL_FRO,
                 what=""):
    e = errors(got, ref, base)
    assert e["max_abs"] <= max_abs and e["rel_fro"] <= rel_fro, (what, e)
    return e
