"""Pure-Python scalar-loop restatement of the DeepSeekMoE layer forward.

TEST INFRASTRUCTURE ONLY.  An independent second writing of the same
definition ("【推理llm論文精讀】DeepSeek V3技術論文", section 2.2: FFN-output,
routing-weight, affinity and biased-selection equations), with no numpy: every
dot product is an explicit loop and the top-K is a selection loop rather than
a sort.  It is slow and meant for tiny shapes only; it cross-checks
``oracle.moe`` so that a slip in one writing shows up as a disagreement.
"""
from __future__ import annotations

import math
from typing import List, Sequence


def _dot(a: Sequence[float], b: Sequence[float]) -> float:
    acc = 0.0
    for x, y in zip(a, b):
        acc += x * y
    return acc


def _sig(z: float) -> float:
    if z >= 0:
        return 1.0 / (1.0 + math.exp(-z))
    ez = math.exp(z)
    return ez / (1.0 + ez)


def _matvec(W: Sequence[Sequence[float]], x: Sequence[float]) -> List[float]:
    """(W x)_r = sum_c W[r][c] x[c]."""
    return [_dot(row, x) for row in W]


def ffn(x, Wg, Wu, Wd) -> List[float]:
    """Down(SiLU(Gate x) * (Up x)) with SiLU(a) = a * Sigmoid(a)."""
    a = _matvec(Wg, x)
    c = _matvec(Wu, x)
    hid = [ai * _sig(ai) * ci for ai, ci in zip(a, c)]
    return _matvec(Wd, hid)


def select(beta: Sequence[float], K: int) -> List[int]:
    """K rounds of "take the largest remaining; on a tie keep the lower index"."""
    taken: List[int] = []
    for _ in range(K):
        best = -1
        for i, v in enumerate(beta):
            if i in taken:
                continue
            if best < 0 or v > beta[best]:
                best = i
        taken.append(best)
    return taken


def layer(u, E, b, K, routed, shared):
    """h for every token; ``routed``/``shared`` are lists of (Wg, Wu, Wd)
    given as nested Python lists ([I][d], [I][d], [d][I])."""
    H, IDX = [], []
    for ut in u:
        s = [_sig(_dot(ut, ei)) for ei in E]
        beta = [si + bi for si, bi in zip(s, b)]
        sel = select(beta, K)
        h = list(ut)
        for w in shared:
            y = ffn(ut, *w)
            h = [hv + yv for hv, yv in zip(h, y)]
        for i in sel:
            y = ffn(ut, *routed[i])
            h = [hv + s[i] * yv for hv, yv in zip(h, y)]
        H.append(h)
        IDX.append(sel)
    return H, IDX
