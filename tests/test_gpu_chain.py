"""Chained decode (he_set_chained_decode): per layer the attention plus one stream-K
launch (out projection, residual + LayerNorm, fc1, fc2, residual + LayerNorm, the next
layer's QKV) gives bit-identical ids and log-probs to the separate launches, for every
token tile of the stream-K kernel (B 1 .. 130), fused (fp16 operands, tiled weights)
and unfused (bf16, row-major weights through tensor maps), with 1 to 4 row groups
per epilogue thread in the rows phases, and through the CUDA graph."""
import numpy as np
import pytest
import torch

from synth.workloads import WORKLOADS, make_model, make_prompts
from tests.gpu_helpers import engine_for

pytestmark = pytest.mark.gpu

BASE = WORKLOADS["opt-tiny-fp32"].with_(name="tiny-bf16-chain", index=31, dtype="bf16",
                                        n_layers=3, d_model=256, n_heads=4, ffn=1024,
                                        vocab=1000, batch=3, prompt_len=9, gen_len=6,
                                        bias_std=0.02, ln_gamma_std=0.1, ln_beta_std=0.02)


def _same(a, b):
    return all(torch.equal(x.view(torch.int32), y.view(torch.int32)) for x, y in zip(a, b))


def _compare(cfg, graph=False):
    inputs = make_model(cfg)
    prompts = torch.from_numpy(make_prompts(cfg)).cuda()
    eng, _w = engine_for(cfg, inputs, torch)
    L = cfg.gen_len
    if graph:
        eng.set_cuda_graph(True)
    for fused in (False, True):
        if fused:
            eng.fuse_lora()
        eng.set_chained_decode(False)
        l0 = eng.stats()["launches"]
        ref = [t.clone() for t in eng.generate(prompts, L)]
        sep = eng.stats()["launches"] - l0
        eng.set_chained_decode(True)
        l0 = eng.stats()["launches"]
        out = [t.clone() for t in eng.generate(prompts, L)]
        chained = eng.stats()["launches"] - l0
        assert _same(out, ref), f"fused={fused}"
        # per decode step: 7 launches per layer become 2 per layer plus layer 0's QKV
        assert sep - chained == (L - 1) * (5 * cfg.n_layers - 1), (sep, chained)
        if fused:
            eng.unfuse_lora()
    eng.check()
    eng.close()


@pytest.mark.parametrize("B", [1, 3, 20, 40, 100, 130])
def test_chained_decode_matches_separate_launches(cuda_device, B):
    _compare(BASE.with_(batch=B))


@pytest.mark.parametrize("d,heads,layers", [(2560, 20, 2), (6400, 50, 1)])
def test_chained_decode_wide_rows(cuda_device, d, heads, layers):
    """Two and four 8-element groups per epilogue thread in the rows phases."""
    _compare(BASE.with_(name=f"chain-d{d}", d_model=d, n_heads=heads, n_layers=layers, batch=5,
                        gen_len=4))


def test_chained_decode_in_graph(cuda_device):
    _compare(BASE.with_(batch=17), graph=True)


def test_chained_decode_against_oracle(cuda_device):
    """The chained path (default) against the CPU oracle, teacher-forced."""
    from tests.gpu_helpers import BF16_LOGIT_TOL, BF16_LP_TOL, teacher_forced_check
    logit_err, lp_err = teacher_forced_check(BASE.with_(batch=4), torch)
    assert logit_err <= BF16_LOGIT_TOL and lp_err <= BF16_LP_TOL, (logit_err, lp_err)
