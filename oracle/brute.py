"""Pure-Python brute force for tiny shapes. TEST INFRASTRUCTURE ONLY.

Written independently of moe_oracle.py (scalar loops, the printed 16-value
E2M1 table, exhaustive subset search for the router) so that each can catch
an indexing or ordering mistake in the other. Only usable for tiny inputs.
"""

from __future__ import annotations

import itertools
import math

# The 16-value E2M1 table printed for the mx4 kernels ("dasLLAMA: dig the last
# two board reds green", section "gpt-oss: mx4 kernels to the lab-winning
# shape": llama.cpp's 16-value LUT), in code order 0..15.
E2M1_PRINTED = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def dequant(qs, sc):
    """qs: R x (C/2) ints, sc: R x (C/32) ints -> R x C list of floats."""
    R = len(qs)
    C = len(qs[0]) * 2
    out = []
    for r in range(R):
        row = []
        for c in range(C):
            blk, i = divmod(c, 32)
            byte = int(qs[r][blk * 16 + (i % 16)])
            nib = (byte & 15) if i < 16 else (byte >> 4)
            s = int(sc[r][blk])
            scale = float("nan") if s == 255 else 2.0 ** (s - 127)
            row.append(E2M1_PRINTED[nib] * scale)
        out.append(row)
    return out


def matvec(W, x, b=None):
    out = []
    for r in range(len(W)):
        acc = 0.0
        for c in range(len(x)):
            acc += W[r][c] * x[c]
        if b is not None:
            acc += float(b[r])
        out.append(acc)
    return out


def topk(logits, k):
    """Exhaustive: the unique k-subset whose members all precede every non-member
    in (descending logit, ascending index) order; then sorted into slot order."""
    E = len(logits)

    def before(a, b):
        return logits[a] > logits[b] or (logits[a] == logits[b] and a < b)

    chosen = None
    for S in itertools.combinations(range(E), k):
        rest = [b for b in range(E) if b not in S]
        if all(before(a, b) for a in S for b in rest):
            assert chosen is None
            chosen = list(S)
    # insertion sort into slot order
    order = []
    for a in chosen:
        pos = 0
        while pos < len(order) and before(order[pos], a):
            pos += 1
        order.insert(pos, a)
    mx = max(logits[a] for a in order)
    ex = [math.exp(logits[a] - mx) for a in order]
    tot = sum(ex)
    return order, [v / tot for v in ex]


def bucket(ids, E, tile, k=None):
    """ids: T x k. Returns counts, basep, rows (length mpad), inv."""
    T = len(ids)
    k = len(ids[0]) if T else k
    counts = [0] * E
    for t in range(T):
        for j in range(k):
            counts[ids[t][j]] += 1
    basep = [0]
    for e in range(E):
        basep.append(basep[-1] + -(-counts[e] // tile) * tile)
    rows = [-1] * basep[E]
    inv = [-1] * (T * k)
    for e in range(E):
        p = basep[e]
        for t in range(T):
            for j in range(k):
                if ids[t][j] == e:
                    rows[p] = t * k + j
                    inv[t * k + j] = p
                    p += 1
    return counts, basep, rows, inv


def swiglu(g, u, alpha=1.702, limit=7.0):
    g = min(g, limit)
    u = max(-limit, min(u, limit))
    z = alpha * g
    if z >= 0:
        s = 1.0 / (1.0 + math.exp(-z))
    else:
        s = math.exp(z) / (1.0 + math.exp(z))
    return g * s * (u + 1.0)


def layer(L, x, k):
    """Whole layer by loops. L holds numpy arrays; x is T x D. Returns y (T x D), ids, weights."""
    E = L["w_router"].shape[0]
    Wr = L["w_router"].tolist()
    br = L["b_router"].tolist() if L.get("b_router") is not None else [0.0] * E
    deq = {}
    y_all, ids_all, w_all = [], [], []
    for t in range(len(x)):
        xt = [float(v) for v in x[t]]
        logits = [sum(float(Wr[e][i]) * xt[i] for i in range(len(xt))) + float(br[e]) for e in range(E)]
        ids, ws = topk(logits, k)
        y = [0.0] * L["d_qs"].shape[1]
        for j, e in enumerate(ids):
            if e not in deq:
                deq[e] = (dequant(L["g_qs"][e].tolist(), L["g_sc"][e].tolist()),
                          dequant(L["u_qs"][e].tolist(), L["u_sc"][e].tolist()),
                          dequant(L["d_qs"][e].tolist(), L["d_sc"][e].tolist()))
            Wg, Wu, Wd = deq[e]
            g = matvec(Wg, xt, L["bg"][e])
            u = matvec(Wu, xt, L["bu"][e])
            h = [swiglu(a, b) for a, b in zip(g, u)]
            o = matvec(Wd, h, L["bd"][e])
            for c in range(len(y)):
                y[c] += ws[j] * o[c]
        y_all.append(y)
        ids_all.append(ids)
        w_all.append(ws)
    return y_all, ids_all, w_all
