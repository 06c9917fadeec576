"""Pure-Python brute force of RoPE attention, for pinning the oracle on tiny inputs.

Written independently of oracle/: the rotation is done as a complex
multiplication (pair (x[i], x[i+D/2]) as x[i] + j*x[i+D/2] times
exp(j * pos * base^(-2i/D))), which expands to the rotation of a half-dimension
pair in the LazyAttention paper, §3.2 "Prefilling"; the softmax is summed term by
term with math.exp. Only small cases: everything is a Python loop.
"""
import cmath
import math


def bf_rope(x, pos, theta):
    D = len(x)
    h = D // 2
    out = [0.0] * D
    for i in range(h):
        w = theta ** (-2.0 * i / D)
        z = complex(x[i], x[i + h]) * cmath.exp(1j * pos * w)
        out[i], out[i + h] = z.real, z.imag
    return out


def bf_attention(q, k, v, q_pos, k_pos, theta):
    """q: nested list [Lq][Hq][D]; k, v: [L][Hkv][D]; positions: lists of ints.

    Query head h reads KV head h // (Hq // Hkv); key j is visible to query i
    iff k_pos[j] <= q_pos[i]. Returns nested list [Lq][Hq][D].
    """
    Lq, Hq, D = len(q), len(q[0]), len(q[0][0])
    L, Hkv = len(k), len(k[0])
    g = Hq // Hkv
    out = []
    for i in range(Lq):
        row = []
        for h in range(Hq):
            kv = h // g
            qr = bf_rope(q[i][h], q_pos[i], theta)
            scores = []
            for j in range(L):
                if k_pos[j] > q_pos[i]:
                    continue
                kr = bf_rope(k[j][kv], k_pos[j], theta)
                s = sum(a * b for a, b in zip(qr, kr)) / math.sqrt(D)
                scores.append((s, j))
            m = max(s for s, _ in scores)
            w = [(math.exp(s - m), j) for s, j in scores]
            z = sum(e for e, _ in w)
            o = [0.0] * D
            for e, j in w:
                for d in range(D):
                    o[d] += e / z * v[j][kv][d]
            row.append(o)
        out.append(row)
    return out
