"""The decoder step in scalar Python loops: a second, independent evaluation.

TEST INFRASTRUCTURE ONLY (see the package docstring).  No numpy arithmetic:
every product and sum is an explicit Python float (IEEE double) loop, so a
transposed operand, a wrong axis or a wrong head mapping in the vectorised
oracle (``oracle.model``) shows up as a disagreement.  Only tiny shapes are
practical (the 2-layer, d_model 64 decoder runs in well under a second).

It follows the same passages as ``oracle.model`` (tinyllm L10.1 section 2.4;
octlm "A real model in our own decoder", the five switches) and the same
readings: eps inside the square root, QK-norm gains shared by heads,
rotate-half RoPE with phi_j = pos * base^(-2j/D), query head h reading
key/value head floor(h * Hkv / H).
"""

from __future__ import annotations

import math


def _mat(a):
    """numpy-or-list 2-D array -> list of lists of Python floats."""
    return [[float(v) for v in row] for row in a]


def _vec(a):
    return [float(v) for v in a]


def _rmsnorm(x, w, eps):
    ms = 0.0
    for v in x:
        ms += v * v
    ms /= len(x)
    r = 1.0 / math.sqrt(ms + eps)
    return [x[i] * r * w[i] for i in range(len(x))]


def _matvec(W, x):
    """y[o] = sum_i W[o][i] * x[i] (weights stored [out, in])."""
    out = []
    for row in W:
        acc = 0.0
        for i, v in enumerate(row):
            acc += v * x[i]
        out.append(acc)
    return out


def _rope(vec, pos, base):
    D = len(vec)
    half = D // 2
    out = list(vec)
    for j in range(half):
        phi = pos * base ** (-2.0 * j / D)
        c, s = math.cos(phi), math.sin(phi)
        a, b = vec[j], vec[j + half]
        out[j] = a * c - b * s
        out[j + half] = b * c + a * s
    return out


def _silu(z):
    return z / (1.0 + math.exp(-z))


class BruteDecoder:
    """Scalar-loop decoder over one sequence with a dict-of-lists cache."""

    def __init__(self, cfg, weights: dict, round_fn=None):
        self.cfg = cfg
        conv = (lambda a: round_fn(a)) if round_fn else (lambda a: a)
        self.E = _mat(conv(weights["embed"]))
        self.final_norm = _vec(weights["final_norm"])
        self.L = []
        for l in range(cfg.n_layers):
            p = f"layers.{l}."
            self.L.append({k: (_vec(weights[p + k]) if k.endswith("norm") else _mat(conv(weights[p + k])))
                           for k in ("attn_norm", "q", "k", "v", "q_norm", "k_norm", "o",
                                     "mlp_norm", "gate", "up", "down")})
        self.kc = [dict() for _ in range(cfg.n_layers)]  # pos -> [kv_head][D]
        self.vc = [dict() for _ in range(cfg.n_layers)]

    def step(self, tokens, start):
        """Logits (list of lists) at every new position."""
        cfg = self.cfg
        H, Hkv, D, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_model
        eps = cfg.rms_eps
        xs = [list(self.E[t]) for t in tokens]
        for l, w in enumerate(self.L):
            # projections, QK-norm, RoPE and the cache write, token by token
            qs = []
            for i, x in enumerate(xs):
                pos = start + i
                h = _rmsnorm(x, w["attn_norm"], eps)
                q = _matvec(w["q"], h)
                k = _matvec(w["k"], h)
                v = _matvec(w["v"], h)
                qh = [_rope(_rmsnorm(q[a * D:(a + 1) * D], w["q_norm"], eps), pos, cfg.rope_base) for a in range(H)]
                kh = [_rope(_rmsnorm(k[a * D:(a + 1) * D], w["k_norm"], eps), pos, cfg.rope_base) for a in range(Hkv)]
                vh = [v[a * D:(a + 1) * D] for a in range(Hkv)]
                self.kc[l][pos] = kh
                self.vc[l][pos] = vh
                qs.append(qh)
            # attention of every new token over keys 0..pos(t)
            for i, x in enumerate(xs):
                pos = start + i
                o = []
                for a in range(H):
                    g = (a * Hkv) // H
                    scores = []
                    for j in range(pos + 1):
                        dot = 0.0
                        for c in range(D):
                            dot += qs[i][a][c] * self.kc[l][j][g][c]
                        scores.append(dot / math.sqrt(D))
                    m = max(scores)
                    e = [math.exp(s - m) for s in scores]
                    z = sum(e)
                    head = [0.0] * D
                    for j in range(pos + 1):
                        pj = e[j] / z
                        vj = self.vc[l][j][g]
                        for c in range(D):
                            head[c] += pj * vj[c]
                    o.extend(head)
                att = _matvec(w["o"], o)
                for c in range(d):
                    x[c] += att[c]
                h2 = _rmsnorm(x, w["mlp_norm"], eps)
                gt = _matvec(w["gate"], h2)
                up = _matvec(w["up"], h2)
                a_ = [_silu(gt[f]) * up[f] for f in range(cfg.ff_hidden)]
                dn = _matvec(w["down"], a_)
                for c in range(d):
                    x[c] += dn[c]
        out = []
        for x in xs:
            hf = _rmsnorm(x, self.final_norm, eps)
            out.append(_matvec(self.E, hf))
        return out
