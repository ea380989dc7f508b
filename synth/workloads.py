"""OPT-style workload shapes and their seeded synthetic inputs.

Shapes are the OPT family the DeepSpeed-Chat paper summary runs ("DeepSpeed-Chat:
Easy, Fast and Affordable RLHF Training of ChatGPT-like Models at All Scales",
§5 Experimental Analysis: OPT-1.3B .. OPT-175B actors; §3.4 Step 3 generation
phase: 256-token prompts, 256-token answers).  Inputs stand in for the
DeepSpeed-RLHF prompt data and trained OPT weights, which are not available:

* weights, embeddings, positions: N(0, 0.02); LayerNorm gamma = 1, beta = 0;
  biases 0 (the "-bias" tiny variant draws biases N(0, 0.02),
  gamma = 1 + N(0, 0.1), beta = N(0, 0.02) so those paths carry signal);
* LoRA factors A [r][in], B [out][r]: N(0, 0.02), r = 8, alpha = 16, on the
  q, k, v, out, fc1 and fc2 projections of every layer;
* prompts: token ids uniform in [3, vocab), every prompt full length.

Seeds: weights 1000 + index, prompts 2000 + index, LoRA 3000 + index.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

from . import normal, uniform_int

# Order of the LoRA-targeted projections inside a layer.
LORA_TARGETS = ("wq", "wk", "wv", "wo", "w1", "w2")
_SLOTS = {name: i for i, name in enumerate(
    ("wq", "wk", "wv", "wo", "w1", "w2", "bq", "bk", "bv", "bo", "b1", "b2",
     "ln1_g", "ln1_b", "ln2_g", "ln2_b"))}


@dataclass(frozen=True)
class OptConfig:
    name: str
    index: int
    n_layers: int
    d_model: int
    n_heads: int
    ffn: int
    vocab: int
    max_pos: int
    dtype: str  # "f32" or "bf16" (storage type of every parameter tensor)
    batch: int
    prompt_len: int
    gen_len: int
    pos_offset: int = 2
    ln_eps: float = 1e-5
    lora_r: int = 8
    lora_alpha: float = 16.0
    init_std: float = 0.02
    bias_std: float = 0.0
    ln_gamma_std: float = 0.0
    ln_beta_std: float = 0.0

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_heads

    @property
    def max_seq(self) -> int:
        return self.prompt_len + self.gen_len

    def with_(self, **kw) -> "OptConfig":
        return replace(self, **kw)

    def shapes(self) -> dict:
        d, f = self.d_model, self.ffn
        return {"wq": (d, d), "wk": (d, d), "wv": (d, d), "wo": (d, d),
                "w1": (f, d), "w2": (d, f), "bq": (d,), "bk": (d,), "bv": (d,),
                "bo": (d,), "b1": (f,), "b2": (d,), "ln1_g": (d,), "ln1_b": (d,),
                "ln2_g": (d,), "ln2_b": (d,)}

    def n_params(self) -> int:
        per_layer = sum(int(np.prod(s)) for s in self.shapes().values())
        return (self.vocab * self.d_model + (self.max_pos + self.pos_offset) * self.d_model
                + 2 * self.d_model + self.n_layers * per_layer)


WORKLOADS = {
    "opt-tiny-fp32": OptConfig("opt-tiny-fp32", 0, 2, 128, 4, 512, 1024, 64, "f32", 2, 16, 16),
    "opt-125m": OptConfig("opt-125m", 1, 12, 768, 12, 3072, 50272, 2048, "bf16", 16, 256, 256),
    "opt-1.3b": OptConfig("opt-1.3b", 2, 24, 2048, 32, 8192, 50272, 2048, "bf16", 32, 256, 256),
    "opt-6.7b": OptConfig("opt-6.7b", 3, 32, 4096, 32, 16384, 50272, 2048, "bf16", 64, 256, 256),
    "opt-13b": OptConfig("opt-13b", 4, 40, 5120, 40, 20480, 50272, 2048, "bf16", 128, 256, 256),
    # the OPT-13B layer and batch shapes in two layers and eight answer tokens: a few GB
    # on the device, for profiling single launches of the full-size kernels
    "opt-13b-2layer": OptConfig("opt-13b-2layer", 6, 2, 5120, 40, 20480, 50272, 2048, "bf16",
                                128, 256, 8),
    # tiny fp32 variant whose biases and LayerNorm affine parameters are not trivial
    "opt-tiny-fp32-bias": OptConfig("opt-tiny-fp32-bias", 5, 2, 128, 4, 512, 1024, 64, "f32",
                                    2, 16, 16, bias_std=0.02, ln_gamma_std=0.1,
                                    ln_beta_std=0.02),
}


def _tid_layer(layer: int, slot: str) -> int:
    return 1000 + 32 * layer + _SLOTS[slot]


def _tid_lora(layer: int, target: int, which: int) -> int:
    return 100000 + 16 * layer + 2 * target + which


def _param(cfg: OptConfig, shape, tid: int, mean: float, std: float) -> np.ndarray:
    seed = 1000 + cfg.index
    if std == 0.0:
        if cfg.dtype == "f32":
            return np.full(shape, mean, dtype=np.float32)
        arr = normal(shape, seed, tid, mean, 0.0, "bf16")  # exact constant, rounded
        return arr
    return normal(shape, seed, tid, mean, std, cfg.dtype)


def make_layer(cfg: OptConfig, layer: int) -> dict:
    """One decoder layer's parameters ([out][in] for projections)."""
    out = {}
    for name, shape in cfg.shapes().items():
        tid = _tid_layer(layer, name)
        if name.startswith("w"):
            out[name] = _param(cfg, shape, tid, 0.0, cfg.init_std)
        elif name.startswith("b"):
            out[name] = _param(cfg, shape, tid, 0.0, cfg.bias_std)
        elif name.endswith("_g"):
            out[name] = _param(cfg, shape, tid, 1.0, cfg.ln_gamma_std)
        else:
            out[name] = _param(cfg, shape, tid, 0.0, cfg.ln_beta_std)
    return out


def make_globals(cfg: OptConfig) -> dict:
    d = cfg.d_model
    return {
        "tok_emb": _param(cfg, (cfg.vocab, d), 1, 0.0, cfg.init_std),
        "pos_emb": _param(cfg, (cfg.max_pos + cfg.pos_offset, d), 2, 0.0, cfg.init_std),
        "lnf_g": _param(cfg, (d,), 3, 1.0, cfg.ln_gamma_std),
        "lnf_b": _param(cfg, (d,), 4, 0.0, cfg.ln_beta_std),
    }


def make_lora_layer(cfg: OptConfig, layer: int) -> dict:
    """LoRA factors of one layer: {target: (A [r][in], B [out][r])}."""
    seed = 3000 + cfg.index
    shapes = cfg.shapes()
    out = {}
    for t, name in enumerate(LORA_TARGETS):
        n_out, n_in = shapes[name]
        a = normal((cfg.lora_r, n_in), seed, _tid_lora(layer, t, 0), 0.0, cfg.init_std, cfg.dtype)
        b = normal((n_out, cfg.lora_r), seed, _tid_lora(layer, t, 1), 0.0, cfg.init_std, cfg.dtype)
        out[name] = (a, b)
    return out


def make_prompts(cfg: OptConfig, batch: int | None = None, prompt_len: int | None = None,
                 seed_offset: int = 0) -> np.ndarray:
    b = cfg.batch if batch is None else batch
    lp = cfg.prompt_len if prompt_len is None else prompt_len
    return uniform_int((b, lp), 2000 + cfg.index + seed_offset, 1, 3, cfg.vocab)


@dataclass
class ModelInputs:
    cfg: OptConfig
    globals: dict
    layers: list = field(default_factory=list)
    lora: list = field(default_factory=list)


def make_model(cfg: OptConfig, with_lora: bool = True) -> ModelInputs:
    m = ModelInputs(cfg, make_globals(cfg))
    for layer in range(cfg.n_layers):
        m.layers.append(make_layer(cfg, layer))
        if with_lora:
            m.lora.append(make_lora_layer(cfg, layer))
    return m
