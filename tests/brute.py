"""Pure-Python triple-loop attention forward / backward for tiny shapes.

An independent restatement (scalar loops, math.exp / math.log, no NumPy
arithmetic) used only to pin the float64 oracle. Layout: nested lists or
arrays indexed [b][h][i][d] (dense) as in the oracle.
"""

import math


def dense_forward(Q, K, V, scale, live, bias=None):
    """live(i, j) -> bool. Returns (O, LSE) as nested lists."""
    B, Hq, Sq, D = len(Q), len(Q[0]), len(Q[0][0]), len(Q[0][0][0])
    Hk, Sk, Dv = len(K[0]), len(K[0][0]), len(V[0][0][0])
    r = Hq // Hk
    O = [[[[0.0] * Dv for _ in range(Sq)] for _ in range(Hq)] for _ in range(B)]
    L = [[[-math.inf] * Sq for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            g = h // r
            for i in range(Sq):
                logits = {}
                for j in range(Sk):
                    if not live(i, j):
                        continue
                    s = 0.0
                    for d in range(D):
                        s += Q[b][h][i][d] * K[b][g][j][d]
                    s *= scale
                    if bias is not None:
                        s += float(bias[h][i][j])
                    logits[j] = s
                if not logits:
                    continue
                mx = max(logits.values())
                tot = sum(math.exp(x - mx) for x in logits.values())
                L[b][h][i] = mx + math.log(tot)
                for j, x in logits.items():
                    p = math.exp(x - L[b][h][i])
                    for d in range(Dv):
                        O[b][h][i][d] += p * V[b][g][j][d]
    return O, L


def dense_backward(Q, K, V, O, dO, L, scale, live, bias=None):
    """Returns (dQ, dK, dV, dbias) as nested lists."""
    B, Hq, Sq, D = len(Q), len(Q[0]), len(Q[0][0]), len(Q[0][0][0])
    Hk, Sk, Dv = len(K[0]), len(K[0][0]), len(V[0][0][0])
    r = Hq // Hk
    dQ = [[[[0.0] * D for _ in range(Sq)] for _ in range(Hq)] for _ in range(B)]
    dK = [[[[0.0] * D for _ in range(Sk)] for _ in range(Hk)] for _ in range(B)]
    dV = [[[[0.0] * Dv for _ in range(Sk)] for _ in range(Hk)] for _ in range(B)]
    dB = [[[0.0] * Sk for _ in range(Sq)] for _ in range(Hq)]
    for b in range(B):
        for h in range(Hq):
            g = h // r
            for i in range(Sq):
                if L[b][h][i] == -math.inf:
                    continue
                rowdot = 0.0
                for d in range(Dv):
                    rowdot += dO[b][h][i][d] * O[b][h][i][d]
                for j in range(Sk):
                    if not live(i, j):
                        continue
                    s = 0.0
                    for d in range(D):
                        s += Q[b][h][i][d] * K[b][g][j][d]
                    s *= scale
                    if bias is not None:
                        s += float(bias[h][i][j])
                    p = math.exp(s - L[b][h][i])
                    dp = 0.0
                    for d in range(Dv):
                        dp += dO[b][h][i][d] * V[b][g][j][d]
                    ds = p * (dp - rowdot)
                    dB[h][i][j] += ds
                    for d in range(D):
                        dQ[b][h][i][d] += scale * ds * K[b][g][j][d]
                        dK[b][g][j][d] += scale * ds * Q[b][h][i][d]
                    for d in range(Dv):
                        dV[b][g][j][d] += p * dO[b][h][i][d]
    return dQ, dK, dV, dB


def sparse_backward(q, ori_kv, cmp_kv, idx, O, dO, L, scale, win_left, win_right):
    """Shared-KV selected-row backward on nested lists; layout as the oracle's."""
    Sq, Hq, D = len(q), len(q[0]), len(q[0][0])
    n_ori, Hk = len(ori_kv), len(ori_kv[0])
    r = Hq // Hk
    dQ = [[[0.0] * D for _ in range(Hq)] for _ in range(Sq)]
    d_ori = [[[0.0] * D for _ in range(Hk)] for _ in range(n_ori)]
    d_cmp = None
    if cmp_kv is not None:
        d_cmp = [[[0.0] * D for _ in range(Hk)] for _ in range(len(cmp_kv))]
    for i in range(Sq):
        pos = n_ori - Sq + i
        for h in range(Hq):
            g = h // r
            rows = []
            for j in range(n_ori):
                if (win_left < 0 or j >= pos - win_left) and (win_right < 0 or j <= pos + win_right):
                    rows.append(("o", j, ori_kv[j][g]))
            if idx is not None:
                for c in idx[i][g]:
                    if c >= 0:
                        rows.append(("c", int(c), cmp_kv[int(c)][g]))
            if not rows:
                continue
            rowdot = sum(dO[i][h][d] * O[i][h][d] for d in range(D))
            for src, j, kv in rows:
                s = scale * sum(q[i][h][d] * kv[d] for d in range(D))
                p = math.exp(s - L[h][i])
                dp = sum(dO[i][h][d] * kv[d] for d in range(D))
                ds = p * (dp - rowdot)
                tgt = d_ori[j][g] if src == "o" else d_cmp[j][g]
                for d in range(D):
                    dQ[i][h][d] += scale * ds * kv[d]
                    tgt[d] += scale * ds * q[i][h][d] + p * dO[i][h][d]
    return dQ, d_ori, d_cmp
