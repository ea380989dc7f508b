"""CPU oracle for Hybrid-Engine experience generation with an OPT-style actor.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this module.  The CUDA library never calls
it, shares no code with it, and has no CPU fallback through it.

What it computes, and from where:

* "DeepSpeed-Chat: Easy, Fast and Affordable RLHF Training of ChatGPT-like Models
  at All Scales" (paper summary), §3.4 "Step 3: RLHF Training via PPO", item 1
  (generation phase): the actor generates the answer to each prompt token by
  token, 256-token prompts and 256-token answers.
* Same page, §3.4 "Inference Mode: Generation Phase Optimizations",
  Optimization 2 (lightweight KV-cache management): keys and values of earlier
  tokens are cached; each step appends the new token's key and value and reuses
  the stored ones.
* Same page, §3.4 "Training Mode: ZeRO and LoRA Optimizations", Optimization 2
  (LoRA): a weight W in R^{d x k} is used as W + B A with B in R^{d x r},
  A in R^{r x k}.  The alpha / r scale (alpha = 16, r = 8) is the workload's.
* "DeepSpeed-Chat 选型指南：Hybrid Engine 驱动的 RLHF 训练全解析", §三 (engine
  internals): generate() merges the LoRA weights into the inference model before
  generation (fuse_lora_weight) and restores them afterwards (unfuse_lora_weight);
  the inference containers replace the OPT layers, including OPT's positional
  embedding layer.
* "Chapter 11 System Architecture & Infrastructure at Scale", "The Generation
  Bottleneck: Quantitative Analysis": the generation step must hand back the
  log-probabilities of the generated tokens (needed for the PPO ratio); the
  production setup there samples with a temperature and a nucleus (top-p)
  cut-off instead of taking the argmax.

Sampling (``sample_token``; greedy when the temperature is 0).  Readings, where
the page only names the two parameters: the sampling distribution is
softmax(logits / T); the nucleus is the smallest set of most probable tokens whose
probability reaches top_p, every token tied with the least probable member
included; the token is drawn from the nucleus renormalised, as the argmax of
log q_i + G_i over the nucleus (the Gumbel-max form of that draw, lowest index on
ties), G_i = -log(-log u_i) with u_i from SplitMix64 (Steele, Lea and Flood,
2014) used as a counter: u for (sequence b, step k, token i) comes from output
number c + 1 of the generator seeded with the sampling seed, c = (b * 2^20 + k)
* 2^20 + i, as (2 * (z >> 41) + 1) / 2^24 (never 0 or 1).  The reported log-prob
is log softmax(logits / T) of the chosen token over the full vocabulary.

Readings where the pages are silent (the plainest OPT reading):
pre-LN decoder layers; LayerNorm with biased variance and eps 1e-5; learned
positions indexed at position + 2; q scaled by head_dim^-1/2 after its bias;
ReLU feed-forward; final LayerNorm; LM head tied to the token embedding with no
bias; greedy decoding, lowest index on exact ties; no end-of-sequence stop
(exactly gen_len tokens); log-prob = natural-log softmax of the chosen token
over the full vocabulary; 1 prefill pass + (gen_len - 1) single-token passes
(the last generated token is not fed back).

Precision: fp32 weights (bf16 storage widened exactly) and fp32 arithmetic.
The LoRA-merged weight W + (alpha/r) B A is kept unrounded in fp32.

FP8 weights for generation ("Chapter 11 System Architecture & Infrastructure at
Scale", "The Generation Bottleneck: Quantitative Analysis", the optimisation stack:
INT8/FP8 weights for generation halve the bandwidth the weights need).  The page
names the idea, not a format; the reading taken here (``weights="fp8"``): each of
the six projections of every layer, after the LoRA merge, is stored as OCP FP8
E4M3 values (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest finite
value 448; subnormals down to 2^-9; no infinity) with one fp32 scale per output
row, s_n = max_k |W[n][k]| / 448, codes q = nearest E4M3 value of W[n][k] / s_n
(fp32 division, ties to the even mantissa, beyond 448 saturated), and generation
runs with the dequantized weight q * s_n in fp32.  Activations, the KV cache and
the tied LM head are not quantized.

Parameters arrive as the synthetic-input dictionaries of ``synth.workloads``:
projections are [out][in] (y = x W^T + b); bf16 tensors are raw uint16 bits.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

TARGETS = ("wq", "wk", "wv", "wo", "w1", "w2")
_BIAS = {"wq": "bq", "wk": "bk", "wv": "bv", "wo": "bo", "w1": "b1", "w2": "b2"}


def to_f32(a: np.ndarray) -> np.ndarray:
    """Exact fp32 value of a stored tensor (bf16 bits are widened by a 16-bit shift)."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return np.asarray(a, dtype=np.float32)


_MASK64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15


def splitmix64_output(seed: int, n: int) -> int:
    """Output number n (n >= 1) of SplitMix64 started from state `seed`: the state
    advances by the golden-ratio increment and each state is mixed."""
    z = (seed + n * _GAMMA) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def sample_uniforms(seed: int, b: int, step: int, n_tokens: int) -> np.ndarray:
    """u_i in (0, 1) for tokens 0 .. n_tokens-1 of (sequence b, step), fp64."""
    base = ((b << 20) + step) << 20
    return np.array([(2 * (splitmix64_output(seed, base + i + 1) >> 41) + 1) / float(1 << 24)
                     for i in range(n_tokens)], dtype=np.float64)


def sample_token(logits: np.ndarray, temperature: float, top_p: float, seed: int, b: int,
                 step: int) -> tuple:
    """One draw from softmax(logits / T) restricted to its top_p nucleus (see the
    module notes); returns (token, log-prob of the token under softmax(logits / T))."""
    lg = np.asarray(logits, dtype=np.float64)
    z = (lg - lg.max()) / temperature
    q = np.exp(z)
    total = q.sum()
    if top_p < 1.0:
        order = np.argsort(-q, kind="stable")
        mass = np.cumsum(q[order])
        k = int(np.searchsorted(mass, top_p * total))  # first prefix reaching top_p
        tau = q[order[min(k, len(order) - 1)]]
        member = q >= tau
    else:
        member = np.ones_like(q, dtype=bool)
    g = -np.log(-np.log(sample_uniforms(seed, b, step, len(q))))
    score = np.where(member, z + g, -np.inf)
    tok = int(np.argmax(score))  # first index of the maximum
    return tok, float(z[tok] - np.log(total))


E4M3_MAX = 448.0


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Nearest OCP FP8 E4M3 value of each element (ties to the even mantissa); values
    beyond +-448 saturate to +-448 (the format has no infinity); NaN stays NaN.

    In the binade [2^e, 2^(e+1)), e >= -6, the format has 8 values 2^(e-3) apart;
    below 2^-6 the subnormals continue with spacing 2^-9.  Rounding |x| / spacing to
    the nearest integer, half to even, is the round-to-nearest-even of the format
    (an even integer is an even mantissa, the implicit bit included).  fp32 in and out:
    every E4M3 value and every spacing is exact in fp32."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x)
    _, e = np.frexp(a)  # a = m 2^e with m in [0.5, 1): the binade is 2^(e - 1)
    e = np.maximum(e - 1, -6)
    spacing = np.ldexp(np.float32(1.0), e - 3).astype(np.float32)
    q = np.rint(a / spacing) * spacing  # exact: spacing is a power of two
    q = np.minimum(q, np.float32(E4M3_MAX))
    return np.where(np.isnan(x), np.float32(np.nan), np.copysign(q, x)).astype(np.float32)


def quantize_rows_e4m3(w: np.ndarray) -> tuple:
    """Per output row n of w [out][in] (fp32): scale s_n = max |w[n]| / 448 (1 for an
    all-zero row) and codes q = e4m3_round(w / s_n), the division in fp32.  Returns
    (q as fp32 values, s fp32 [out])."""
    w = np.asarray(w, dtype=np.float32)
    amax = np.abs(w).max(axis=1)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = np.empty_like(w)

    def rows(i):  # a block of rows at a time (bounded temporaries, one per thread)
        q[i:i + 256] = e4m3_round(w[i:i + 256] / s[i:i + 256, None])

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(rows, range(0, w.shape[0], 256)))
    return q, s


def dequantize_rows(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """The weight generation runs with: q * s_n per row, fp32."""
    return (np.asarray(q, np.float32) * np.asarray(s, np.float32)[:, None]).astype(np.float32)


def lora_delta(a: np.ndarray, b: np.ndarray, alpha: float, r: int) -> np.ndarray:
    """(alpha / r) * B @ A: the low-rank update of the LoRA passage, [out][in], fp32."""
    return np.float32(alpha / r) * (to_f32(b) @ to_f32(a))


def merge_lora(w: np.ndarray, a: np.ndarray, b: np.ndarray, alpha: float, r: int) -> np.ndarray:
    """W + (alpha / r) B A in fp32 (the weight generation runs with after the fuse)."""
    return to_f32(w) + lora_delta(a, b, alpha, r)


def layer_norm(x: np.ndarray, g: np.ndarray, b: np.ndarray, eps: float) -> np.ndarray:
    """LayerNorm over the last axis: biased variance, eps inside the square root."""
    mean = x.mean(axis=-1, keepdims=True, dtype=np.float32)
    c = x - mean
    var = (c * c).mean(axis=-1, keepdims=True, dtype=np.float32)
    return (c / np.sqrt(var + np.float32(eps))) * g + b


def log_softmax_pick(logits: np.ndarray, token: np.ndarray) -> np.ndarray:
    """log softmax(logits)[token] per row, max-subtracted: l[t] - (m + log sum exp(l - m))."""
    m = logits.max(axis=-1, keepdims=True)
    lse = m[..., 0] + np.log(np.exp(logits - m).sum(axis=-1, dtype=np.float32))
    picked = np.take_along_axis(logits, token[..., None].astype(np.int64), axis=-1)[..., 0]
    return (picked - lse).astype(np.float32)


def greedy(logits: np.ndarray) -> np.ndarray:
    """Greedy choice per row; np.argmax returns the lowest index among equal maxima."""
    return logits.argmax(axis=-1).astype(np.int32)


class OracleModel:
    """fp32 OPT-style decoder with a KV cache.

    ``lora`` selects how the LoRA factors enter: "merged" (W + (alpha/r) B A, what
    generation runs with), "unmerged" (base projection plus an explicit low-rank
    branch, the training-mode form) or "none" (base weights only).  ``weights``:
    "exact" (the fp32 values above) or "fp8" (the six projections, after the merge,
    quantized per row to E4M3 and dequantized; see the module notes; needs lora
    "merged" or "none").
    """

    def __init__(self, inputs, lora: str = "merged", weights: str = "exact"):
        if lora not in ("merged", "unmerged", "none"):
            raise ValueError(lora)
        if weights not in ("exact", "fp8") or (weights == "fp8" and lora == "unmerged"):
            raise ValueError(weights)
        self.cfg = cfg = inputs.cfg
        self.lora_mode = lora
        self.scale = np.float32(cfg.lora_alpha / cfg.lora_r)
        g = inputs.globals
        self.tok_emb = to_f32(g["tok_emb"])
        self.pos_emb = to_f32(g["pos_emb"])
        self.lnf_g, self.lnf_b = to_f32(g["lnf_g"]), to_f32(g["lnf_b"])
        self.layers = []
        for li, p in enumerate(inputs.layers):
            lw = {k: to_f32(v) for k, v in p.items() if not k.startswith("w")}
            for name in TARGETS:
                if lora == "merged" and inputs.lora:
                    a, b = inputs.lora[li][name]
                    lw[name] = merge_lora(p[name], a, b, cfg.lora_alpha, cfg.lora_r)
                else:
                    lw[name] = to_f32(p[name])
                if lora == "unmerged" and inputs.lora:
                    a, b = inputs.lora[li][name]
                    lw[name + "_A"], lw[name + "_B"] = to_f32(a), to_f32(b)
                if weights == "fp8":
                    lw[name] = dequantize_rows(*quantize_rows_e4m3(lw[name]))
            self.layers.append(lw)

    # -- one projection: y = x W^T + b (+ (alpha/r) (x A^T) B^T when unmerged) --
    def _proj(self, lw: dict, name: str, x: np.ndarray) -> np.ndarray:
        y = x @ lw[name].T + lw[_BIAS[name]]
        if name + "_A" in lw:
            y = y + self.scale * ((x @ lw[name + "_A"].T) @ lw[name + "_B"].T)
        return y

    def embed(self, ids: np.ndarray, positions: np.ndarray) -> np.ndarray:
        """x = E_tok[id] + E_pos[position + 2] (OPT's learned positions, offset 2)."""
        return self.tok_emb[ids] + self.pos_emb[positions + self.cfg.pos_offset]

    def new_cache(self, batch: int, length: int) -> list:
        cfg = self.cfg
        shape = (batch, cfg.n_heads, length, cfg.head_dim)
        return [(np.zeros(shape, np.float32), np.zeros(shape, np.float32))
                for _ in range(cfg.n_layers)]

    def layer(self, li: int, x: np.ndarray, cache, p0: int) -> np.ndarray:
        """One pre-LN decoder layer over new tokens x [B][n][d] at positions p0..p0+n-1.

        Appends their keys/values to ``cache`` at those positions and attends each
        new token to every cached position <= its own (causal).
        """
        cfg, lw = self.cfg, self.layers[li]
        bsz, n, d = x.shape
        nh, hd = cfg.n_heads, cfg.head_dim
        h = layer_norm(x, lw["ln1_g"], lw["ln1_b"], cfg.ln_eps)
        q = self._proj(lw, "wq", h) * np.float32(hd ** -0.5)
        k = self._proj(lw, "wk", h)
        v = self._proj(lw, "wv", h)
        split = lambda t: t.reshape(bsz, n, nh, hd).transpose(0, 2, 1, 3)  # [B][H][n][hd]
        kc, vc = cache
        kc[:, :, p0:p0 + n] = split(k)
        vc[:, :, p0:p0 + n] = split(v)
        keys, vals = kc[:, :, :p0 + n], vc[:, :, :p0 + n]
        s = split(q) @ keys.transpose(0, 1, 3, 2)  # [B][H][n][p0+n]
        qpos = p0 + np.arange(n)[:, None]
        kpos = np.arange(p0 + n)[None, :]
        s = np.where(kpos <= qpos, s, np.float32(-np.inf))
        s = s - s.max(axis=-1, keepdims=True)
        e = np.exp(s)
        pr = e / e.sum(axis=-1, keepdims=True)
        ctx = (pr @ vals).transpose(0, 2, 1, 3).reshape(bsz, n, d)
        x = x + self._proj(lw, "wo", ctx)
        h = layer_norm(x, lw["ln2_g"], lw["ln2_b"], cfg.ln_eps)
        x = x + self._proj(lw, "w2", np.maximum(self._proj(lw, "w1", h), np.float32(0.0)))
        return x

    def forward(self, ids: np.ndarray, cache, p0: int) -> np.ndarray:
        """Residual stream after all layers for new tokens ids [B][n] at positions p0.."""
        n = ids.shape[1]
        x = self.embed(ids, np.arange(p0, p0 + n)[None, :])
        for li in range(self.cfg.n_layers):
            x = self.layer(li, x, cache[li], p0)
        return x

    def logits(self, x: np.ndarray) -> np.ndarray:
        """Final LayerNorm, then the tied LM head: logits = LN_f(x) E_tok^T (no bias)."""
        y = layer_norm(x, self.lnf_g, self.lnf_b, self.cfg.ln_eps)
        return y @ self.tok_emb.T

    def generate(self, prompts: np.ndarray, gen_len: int, force_ids: np.ndarray | None = None,
                 log_steps=(), sampling=None) -> tuple:
        """Generation of ``gen_len`` tokens per prompt: greedy, or with ``sampling`` =
        (temperature, top_p, seed) and temperature > 0 drawn by ``sample_token``.

        Step 0 is the head of the prefill pass (last prompt position); step k >= 1
        feeds token k-1's id at position Lp + k - 1.  With ``force_ids`` [B][gen_len]
        the fed-back token of every step is the forced one (entries < 0 fall back to
        the greedy choice) and the returned log-prob is the forced token's.
        Returns (ids [B][gen_len] int32, logprobs [B][gen_len] fp32,
        {step: logits [B][V]} for the steps in ``log_steps``).
        """
        prompts = np.asarray(prompts, dtype=np.int64)
        bsz, lp = prompts.shape
        cache = self.new_cache(bsz, lp + gen_len)
        ids = np.zeros((bsz, gen_len), np.int32)
        lps = np.zeros((bsz, gen_len), np.float32)
        logged = {}
        x = self.forward(prompts, cache, 0)[:, -1:]
        for k in range(gen_len):
            if k > 0:
                x = self.forward(ids[:, k - 1:k].astype(np.int64), cache, lp + k - 1)
            lg = self.logits(x[:, 0])
            if sampling is not None and sampling[0] > 0:
                drawn = [sample_token(lg[b], sampling[0], sampling[1], sampling[2], b, k)
                         for b in range(bsz)]
                tok = np.array([t for t, _ in drawn], dtype=np.int32)
                lpk = np.array([v for _, v in drawn], dtype=np.float32)
            else:
                tok = greedy(lg)
                lpk = None
            if force_ids is not None:
                f = np.asarray(force_ids)[:, k]
                forced = f >= 0
                tok = np.where(forced, f, tok).astype(np.int32)
                if lpk is not None and forced.any():
                    lpk = lpk.copy()
                    t_inv = 1.0 / sampling[0]
                    for b in np.nonzero(forced)[0]:
                        zb = (lg[b].astype(np.float64) - lg[b].max()) * t_inv
                        lpk[b] = zb[tok[b]] - np.log(np.exp(zb).sum())
            ids[:, k] = tok
            lps[:, k] = log_softmax_pick(lg, tok) if lpk is None else lpk
            if k in log_steps:
                logged[k] = lg.copy()
        return ids, lps, logged

    def full_logits(self, seq: np.ndarray) -> np.ndarray:
        """Logits at every position of seq [B][T], computed in one causal pass, no reuse."""
        seq = np.asarray(seq, dtype=np.int64)
        cache = self.new_cache(seq.shape[0], seq.shape[1])
        return self.logits(self.forward(seq, cache, 0))


def generate(inputs, prompts, gen_len, force_ids=None, log_steps=()):
    """Convenience wrapper: merged-LoRA generation (what the library's fuse + generate runs)."""
    return OracleModel(inputs, "merged").generate(prompts, gen_len, force_ids, log_steps)
