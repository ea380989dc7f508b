"""Generation without a LoRA fuse on bf16 engines, against the oracle's base-weight
model ("none": no LoRA factors), teacher-forced on the oracle's tokens.

Unfused bf16 generation converts the caller's bf16 projections to fp16 at the start
of every generation and then runs the fused path's fp16 kernels, so it meets the same
bars: logits within 3e-2 max-abs and chosen-token log-probs within 5e-2.  OPT-125M is
compared on every sequence, OPT-1.3B and OPT-13B on sequences 0 and 1, each on the
prefill row and decode steps 1..8, at the full batch and lengths.
"""
import numpy as np
import pytest
import torch

from oracle import OracleModel
from synth.workloads import WORKLOADS, make_model, make_prompts
from tests.gpu_helpers import BF16_LOGIT_TOL, BF16_LP_TOL, engine_for, teacher_forced_check

pytestmark = pytest.mark.gpu

STEPS = range(9)  # prefill head (step 0) + decode steps 1..8

TINY_BF16 = WORKLOADS["opt-tiny-fp32"].with_(name="tiny-bf16-unfused", index=24, dtype="bf16",
                                             d_model=256, n_heads=4, ffn=512, vocab=1000,
                                             batch=3, prompt_len=13, gen_len=9)


def test_tiny_unfused_all_steps(cuda_device):
    logit_err, lp_err = teacher_forced_check(TINY_BF16, torch, fused=False)
    assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (logit_err, lp_err)


def test_opt125m_unfused_all_sequences(cuda_device):
    logit_err, lp_err = teacher_forced_check(WORKLOADS["opt-125m"], torch, steps=STEPS,
                                             fused=False)
    assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (logit_err, lp_err)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["opt-1.3b", "opt-13b"])
def test_large_models_unfused_sampled_sequences(cuda_device, name):
    logit_err, lp_err = teacher_forced_check(WORKLOADS[name], torch, steps=STEPS,
                                             oracle_seqs=[0, 1], fused=False)
    assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (name, logit_err, lp_err)


def test_unfused_generation_reads_the_current_weights(cuda_device):
    """The fp16 copy is rewritten by every generation: a change to the caller's weights
    between two unfused calls (as a training step makes) shows in the second call, and
    a fuse / unfuse in between leaves the next unfused call unchanged."""
    cfg = TINY_BF16
    inputs = make_model(cfg)
    prompts_np = make_prompts(cfg)
    prompts = torch.from_numpy(prompts_np).cuda()
    eng, w = engine_for(cfg, inputs, torch)
    ids0, lps0 = [t.clone() for t in eng.generate(prompts, cfg.gen_len)]
    eng.fuse_lora()
    eng.generate(prompts, cfg.gen_len)
    eng.unfuse_lora()
    ids1, lps1 = eng.generate(prompts, cfg.gen_len)
    torch.cuda.synchronize()
    assert torch.equal(ids0, ids1) and torch.equal(lps0, lps1)
    # scale layer 0's fc2 on both sides, then compare with the oracle again
    w["layers"][0]["w2"].mul_(3.0)
    inputs.layers[0]["w2"] = (w["layers"][0]["w2"].cpu().view(torch.int16).numpy()
                              .view(np.uint16).copy())
    oracle = OracleModel(inputs, "none")
    ref_ids, ref_lps, ref_lg = oracle.generate(prompts_np, cfg.gen_len,
                                               log_steps=range(cfg.gen_len))
    force = torch.from_numpy(ref_ids).cuda()
    rows = [(b, k) for b in range(cfg.batch) for k in range(cfg.gen_len)]
    _ids, lps, lg = eng.generate_ex(prompts, cfg.gen_len, force_ids=force, log_rows=rows)
    torch.cuda.synchronize()
    lg = lg.cpu().numpy()
    err = max(np.abs(lg[i] - ref_lg[k][b]).max() for i, (b, k) in enumerate(rows))
    assert err < BF16_LOGIT_TOL, err
    assert np.abs(lps.cpu().numpy() - ref_lps).max() < BF16_LP_TOL
    # the changed weights changed the result
    assert not np.array_equal(ref_ids, ids0.cpu().numpy())
    eng.close()
