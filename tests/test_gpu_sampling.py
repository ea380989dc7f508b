"""Sampled generation (he_set_sampling): the GPU's draw at every step equals the
oracle sampler's draw on the same logits (the GPU's own, captured); fp32
free-running generation equals the oracle's; graph replay, determinism, errors."""
import numpy as np
import pytest
import torch

import decode_opt_step_gb300 as he
from oracle import OracleModel, sample_token
from synth.workloads import WORKLOADS, make_model, make_prompts
from tests.gpu_helpers import FP32_LP_TOL, engine_for

pytestmark = pytest.mark.gpu

TINY_BF16 = WORKLOADS["opt-tiny-fp32"].with_(name="tiny-bf16-sample", index=23, dtype="bf16",
                                             d_model=256, n_heads=4, ffn=512, vocab=1000,
                                             batch=3, prompt_len=13, gen_len=9)


@pytest.mark.parametrize("cfg", [WORKLOADS["opt-tiny-fp32"], TINY_BF16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("t,top_p,seed", [(0.8, 0.9, 1234), (1.0, 1.0, 7), (1.5, 0.5, 2 ** 63 + 5)])
def test_sampled_draws_match_oracle_sampler(cuda_device, cfg, t, top_p, seed):
    inputs = make_model(cfg)
    prompts = torch.from_numpy(make_prompts(cfg)).cuda()
    B, L = cfg.batch, cfg.gen_len
    eng, _w = engine_for(cfg, inputs, torch)
    eng.fuse_lora()
    eng.set_sampling(t, top_p, seed)
    rows = [(b, k) for k in range(L) for b in range(B)]
    ids, lps, logits = eng.generate_ex(prompts, L, log_rows=rows)
    torch.cuda.synchronize()
    ids, lps, logits = ids.cpu().numpy(), lps.cpu().numpy(), logits.cpu().numpy()
    for i, (b, k) in enumerate(rows):
        tok, lp = sample_token(logits[i], t, top_p, seed, b, k)
        assert ids[b, k] == tok, (b, k)
        assert abs(lps[b, k] - lp) < 1e-4, (b, k)
    # same seed, same draws (also through the captured graph); another seed differs
    again = eng.generate(prompts, L)
    assert np.array_equal(again[0].cpu().numpy(), ids)
    eng.set_cuda_graph(True)
    assert np.array_equal(eng.generate(prompts, L)[0].cpu().numpy(), ids)
    eng.set_sampling(t, top_p, seed + 1)
    assert not np.array_equal(eng.generate(prompts, L)[0].cpu().numpy(), ids)
    eng.unfuse_lora()
    eng.close()


def test_sampled_generation_fp32_matches_oracle(cuda_device):
    cfg = WORKLOADS["opt-tiny-fp32"]
    inputs = make_model(cfg)
    prompts = make_prompts(cfg)
    t, top_p, seed = 0.9, 0.8, 4242
    ids_o, lps_o, _ = OracleModel(inputs, "merged").generate(prompts, cfg.gen_len,
                                                            sampling=(t, top_p, seed))
    eng, _w = engine_for(cfg, inputs, torch)
    eng.fuse_lora()
    eng.set_sampling(t, top_p, seed)
    ids, lps = eng.generate(torch.from_numpy(prompts).cuda(), cfg.gen_len)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.abs(lps.cpu().numpy() - lps_o).max() < FP32_LP_TOL
    eng.close()


def test_sampling_arguments(cuda_device):
    cfg = WORKLOADS["opt-tiny-fp32"]
    eng, _w = engine_for(cfg, make_model(cfg), torch)
    for bad in ((-1.0, 1.0), (float("nan"), 1.0), (1.0, 0.0), (1.0, 1.5)):
        with pytest.raises(he.HeError) as e:
            eng.set_sampling(*bad)
        assert e.value.status == he.HE_ERR_ARG
    eng.set_sampling(0.0)  # back to greedy
    eng.close()


@pytest.mark.parametrize("t,top_p,seed", [(0.7, 0.9, 1234), (1.0, 1.0, 7), (1.5, 0.5, 2 ** 63 + 5)])
def test_sampled_draws_match_oracle_at_full_vocabulary(cuda_device, t, top_p, seed):
    """OPT-125M shape (vocab 50272, batch 16, 256-token prompts), LoRA fused: at every
    step each thread of the GPU's nucleus search sums about 49 probabilities of the
    row; every draw must still equal the oracle sampler's on the same logits."""
    cfg = WORKLOADS["opt-125m"].with_(gen_len=4)
    inputs = make_model(cfg)
    prompts = torch.from_numpy(make_prompts(cfg)).cuda()
    B, L = cfg.batch, cfg.gen_len
    eng, _w = engine_for(cfg, inputs, torch)
    eng.fuse_lora()
    eng.set_sampling(t, top_p, seed)
    rows = [(b, k) for k in range(L) for b in range(B)]
    ids, lps, logits = eng.generate_ex(prompts, L, log_rows=rows)
    torch.cuda.synchronize()
    ids, lps, logits = ids.cpu().numpy(), lps.cpu().numpy(), logits.cpu().numpy()
    eng.unfuse_lora()
    eng.close()
    for i, (b, k) in enumerate(rows):
        tok, lp = sample_token(logits[i], t, top_p, seed, b, k)
        assert ids[b, k] == tok, (b, k, ids[b, k], tok)
        assert abs(lps[b, k] - lp) < 1e-4, (b, k)
