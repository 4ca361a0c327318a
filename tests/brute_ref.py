"""A second, independently written float64 restatement of one mHC site, in plain
Python scalar loops over nested lists, for brute-force cross-checks of the C
oracle on tiny shapes (hidden = 8, streams = 2 or 3).  It shares no code with
oracle/ and is only usable for a handful of tokens.

Formulas: memra-engine hyper.rs page, module header "ARITHMETIC CONTRACT",
with the split read as in the oracle (sigmoid gates, exp + alternating
row/column normalisation with eps in both denominators).
"""

import math


def site(x, fn_w, scale, base, f, iters, eps):
    """x: [T][s][d] lists, fn_w: [R][s*d], f: [T][d].  Returns per-token dicts."""
    out = []
    for xt, ft in zip(x, f):
        s, d = len(xt), len(xt[0])
        flat = [xt[c][i] for c in range(s) for i in range(d)]
        mean_sq = sum(v * v for v in flat) / len(flat)
        r = 1.0 / math.sqrt(mean_sq + eps)
        rows = (2 + s) * s
        logit = []
        for row in range(rows):
            dot = 0.0
            for q in range(s * d):
                dot += fn_w[row][q] * flat[q]
            if row < s:
                g = scale[0]
            elif row < 2 * s:
                g = scale[1]
            else:
                g = scale[2]
            logit.append(dot * r * g + base[row])
        pre = [1.0 / (1.0 + math.exp(-logit[c])) + eps for c in range(s)]
        post = [2.0 / (1.0 + math.exp(-logit[s + c])) for c in range(s)]
        m = [[math.exp(logit[2 * s + j * s + k]) for k in range(s)] for j in range(s)]
        for _ in range(iters):
            for j in range(s):
                tot = sum(m[j]) + eps
                m[j] = [v / tot for v in m[j]]
            for k in range(s):
                tot = sum(m[j][k] for j in range(s)) + eps
                for j in range(s):
                    m[j][k] = m[j][k] / tot
        y = [sum(pre[c] * xt[c][i] for c in range(s)) for i in range(d)]
        x_out = [[post[k] * ft[i] + sum(m[j][k] * xt[j][i] for j in range(s)) for i in range(d)]
                 for k in range(s)]
        out.append(dict(pre=pre, post=post, comb=m, y=y, x_out=x_out))
    return out


def head(x, fn_w, scale, base, eps):
    """Gated-head exit: rows = streams, one scale; gate = sigmoid(logit) + eps, then the
    collapse.  x: [T][s][d], fn_w: [s][s*d].  Returns per-token dicts (gates, y)."""
    out = []
    for xt in x:
        s, d = len(xt), len(xt[0])
        flat = [xt[c][i] for c in range(s) for i in range(d)]
        r = 1.0 / math.sqrt(sum(v * v for v in flat) / len(flat) + eps)
        gates = []
        for c in range(s):
            dot = sum(fn_w[c][q] * flat[q] for q in range(s * d))
            gates.append(1.0 / (1.0 + math.exp(-(dot * r * scale[0] + base[c]))) + eps)
        y = [sum(gates[c] * xt[c][i] for c in range(s)) for i in range(d)]
        out.append(dict(gates=gates, y=y))
    return out
