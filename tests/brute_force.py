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


def e4m3_values():
    """Every finite OCP FP8 E4M3 value with its code, decoded bit by bit from the
    format's definition: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent
    field 0 is subnormal (2^-6 * m / 8); the pattern S.1111.111 is NaN."""
    out = []
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            continue  # NaN
        v = sign * (2.0 ** -6 * m / 8.0 if e == 0 else 2.0 ** (e - 7) * (1.0 + m / 8.0))
        out.append((v, code))
    return out


def nearest_e4m3(x, table=None):
    """Nearest E4M3 value of x by search over every finite value (ties: the code
    with the even mantissa bit); |x| beyond the largest value saturates."""
    table = table or e4m3_values()
    best = None
    for v, code in table:
        d = abs(x - v)
        if best is None or d < best[0] or (d == best[0] and (code & 1) == 0 and best[2] & 1):
            best = (d, v, code)
    return best[1]


def quantize_rows_brute(W):
    """Per row: scale = max |w| / 448 (fp32, as the format's scale is stored), each
    element the nearest E4M3 value of w / scale (fp32 division), times the scale."""
    table = e4m3_values()
    out = []
    for row in W:
        amax = np.float32(max(abs(v) for v in row))
        s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
        out.append([nearest_e4m3(float(np.float32(np.float32(v) / s)), table) * float(s)
                    for v in row])
    return out


class BruteForce:
    def __init__(self, inputs, lora: bool = True, fp8: bool = False):
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
            if fp8:
                for name in ("wq", "wk", "wv", "wo", "w1", "w2"):
                    lw[name] = quantize_rows_brute(lw[name])
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
