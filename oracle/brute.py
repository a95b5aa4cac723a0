"""Pure-Python triple loop for tiny attention shapes (oracle; test-only).

Independent of torch arithmetic: nested Python lists and ``math.exp`` only,
so it shares no library routine with ``attention.py``.  It follows the same
definition (the "flash attention v3 paper" search page, first snippet: S =
QK^T, row softmax, O = PV) with the scale of the FA2 pseudocode on "Hacker
News Digest — gpu-computing" and the causal reading key j visible to query i
iff j <= i.  GQA reading: query head h uses kv head h // (Hq // Hkv).
"""

import math


def attention_loops(q, k, v, scale, causal):
    """q: nested lists [B][Hq][Nq][D]; k, v: [B][Hkv][Nkv][D] (floats).

    Returns (O, LSE) as nested lists [B][Hq][Nq][D] and [B][Hq][Nq].
    """
    B, Hq, Nq, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv, Nkv = len(k[0]), len(k[0][0])
    group = Hq // Hkv
    O, LSE = [], []
    for b in range(B):
        Ob, Lb = [], []
        for h in range(Hq):
            g = h // group
            Oh, Lh = [], []
            for i in range(Nq):
                scores = []
                for j in range(Nkv):
                    if causal and j > i:
                        continue
                    dot = 0.0
                    for t in range(D):
                        dot += q[b][h][i][t] * k[b][g][j][t]
                    scores.append((j, dot * scale))
                mx = max(s for _, s in scores)
                weights = [(j, math.exp(s - mx)) for j, s in scores]
                den = sum(w for _, w in weights)
                row = []
                for t in range(D):
                    acc = 0.0
                    for j, w in weights:
                        acc += w * v[b][g][j][t]
                    row.append(acc / den)
                Oh.append(row)
                Lh.append(mx + math.log(den))
            Ob.append(Oh)
            Lb.append(Lh)
        O.append(Ob)
        LSE.append(Lb)
    return O, LSE
