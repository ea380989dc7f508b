"""Naive float64 OPT-style decoder with explicit scalar loops (a pin for the oracle).

It shares nothing with ``oracle/``: no KV cache (every position's prefix is
recomputed from the token ids at every step), no matrix library, plain Python
loops over every index.  It is only usable on tiny models (d_model ~ 8).
"""
from __future__ import annotations

import math

import numpy as np


def _f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << 16).view(np.float32)
    return [list(map(float, row)) for row in np.atleast_2d(a.astype(np.float64))]


def _vec(a):
    return _f64(a)[0]


def _linear(x, w, b):
    # y_o = sum_i x_i * w[o][i] + b_o
    return [sum(x[i] * w[o][i] for i in range(len(x))) + b[o] for o in range(len(w))]


def _ln(x, g, b, eps):
    n = len(x)
    mu = sum(x) / n
    var = sum((xi - mu) ** 2 for xi in x) / n
    return [(x[i] - mu) / math.sqrt(var + eps) * g[i] + b[i] for i in range(n)]


class BruteForce:
    def __init__(self, inputs, lora: bool = True):
        cfg = self.cfg = inputs.cfg
        g = inputs.globals
        self.E = _f64(g["tok_emb"])
        self.P = _f64(g["pos_emb"])
        self.gf, self.bf = _vec(g["lnf_g"]), _vec(g["lnf_b"])
        s = cfg.lora_alpha / cfg.lora_r
        self.layers = []
        for li, p in enumerate(inputs.layers):
            lw = {}
            for k, v in p.items():
                lw[k] = _f64(v) if k.startswith("w") else _vec(v)
            if lora and inputs.lora:
                for name, (a, b) in inputs.lora[li].items():
                    A, B = _f64(a), _f64(b)
                    W = lw[name]
                    for o in range(len(W)):
                        for i in range(len(W[0])):
                            W[o][i] += s * sum(B[o][j] * A[j][i] for j in range(cfg.lora_r))
            self.layers.append(lw)

    def last_logits(self, seq):
        """Logits for the last position of ``seq``, recomputing the whole prefix."""
        cfg = self.cfg
        d, nh = cfg.d_model, cfg.n_heads
        hd = d // nh
        T = len(seq)
        xs = [[self.E[seq[t]][i] + self.P[t + cfg.pos_offset][i] for i in range(d)]
              for t in range(T)]
        for lw in self.layers:
            hs = [_ln(x, lw["ln1_g"], lw["ln1_b"], cfg.ln_eps) for x in xs]
            qs = [[v / math.sqrt(hd) for v in _linear(h, lw["wq"], lw["bq"])] for h in hs]
            ks = [_linear(h, lw["wk"], lw["bk"]) for h in hs]
            vs = [_linear(h, lw["wv"], lw["bv"]) for h in hs]
            new = []
            for t in range(T):
                ctx = [0.0] * d
                for hh in range(nh):
                    sl = range(hh * hd, (hh + 1) * hd)
                    sc = [sum(qs[t][i] * ks[j][i] for i in sl) for j in range(t + 1)]
                    m = max(sc)
                    ex = [math.exp(s - m) for s in sc]
                    z = sum(ex)
                    for i in sl:
                        ctx[i] = sum(ex[j] / z * vs[j][i] for j in range(t + 1))
                o = _linear(ctx, lw["wo"], lw["bo"])
                x1 = [xs[t][i] + o[i] for i in range(d)]
                h2 = _ln(x1, lw["ln2_g"], lw["ln2_b"], cfg.ln_eps)
                f = [max(0.0, v) for v in _linear(h2, lw["w1"], lw["b1"])]
                f2 = _linear(f, lw["w2"], lw["b2"])
                new.append([x1[i] + f2[i] for i in range(d)])
            xs = new
        y = _ln(xs[-1], self.gf, self.bf, cfg.ln_eps)
        return [sum(y[i] * self.E[v][i] for i in range(d)) for v in range(cfg.vocab)]

    def generate(self, prompt, gen_len, force=None):
        seq = list(map(int, prompt))
        ids, lps, rows = [], [], []
        for k in range(gen_len):
            lg = self.last_logits(seq)
            m = max(lg)
            tok = lg.index(m)  # first maximum
            if force is not None:
                tok = int(force[k])
            lse = m + math.log(sum(math.exp(v - m) for v in lg))
            ids.append(tok)
            lps.append(lg[tok] - lse)
            rows.append(lg)
            seq.append(tok)
        return ids, lps, rows
