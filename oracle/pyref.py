"""Pure-Python attention forward for tiny shapes (TEST INFRASTRUCTURE ONLY).

Every sum is ``math.fsum`` (correctly rounded), so this leg does not depend on
summation order.  It follows the definition of section 1 of "CUDA FlashAttention：
从在线 Softmax 到长序列 IO 极限": s_ij = scale * q_i . k_j over the unmasked j,
softmax with the row maximum subtracted, then the weighted sum of the v_j.
Nested lists in, nested lists out: q[b][h][i][d].
"""
from __future__ import annotations

import math


def attention(q, k, v, causal: bool, scale: float):
    out, lses = [], []
    for qb, kb, vb in zip(q, k, v):
        ob, lb = [], []
        for qh, kh, vh in zip(qb, kb, vb):
            n = len(qh)
            oh, lh = [], []
            for i in range(n):
                keys = range(i + 1) if causal else range(n)
                s = [scale * math.fsum(a * b for a, b in zip(qh[i], kh[j])) for j in keys]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                total = math.fsum(e)
                d = len(vh[0])
                oh.append([math.fsum(e[t] * vh[j][c] for t, j in enumerate(keys)) / total
                           for c in range(d)])
                lh.append(m + math.log(total))
            ob.append(oh)
            lb.append(lh)
        out.append(ob)
        lses.append(lb)
    return out, lses
