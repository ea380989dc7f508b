"""Parity at the full workload sizes, in the launch configuration bench.py times.

The GPU runs the whole batch at the full prompt and answer lengths, teacher-forced on
the oracle's tokens for the sequences the oracle computes.  The compared outputs are
the logits of the prefill row and decode steps 1..8 and the chosen-token log-probs:
all sequences for OPT-125M, sequences 0 and 1 for the larger models (rows of a batch
are independent, so the oracle computes only those).
"""
import pytest
import torch

from synth.workloads import WORKLOADS
from tests.gpu_helpers import BF16_LOGIT_TOL, BF16_LP_TOL, teacher_forced_check

pytestmark = pytest.mark.gpu

STEPS = range(9)  # prefill head (step 0) + decode steps 1..8


def test_opt125m_all_sequences(cuda_device):
    cfg = WORKLOADS["opt-125m"]
    logit_err, lp_err = teacher_forced_check(cfg, torch, steps=STEPS)
    assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (logit_err, lp_err)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["opt-1.3b", "opt-6.7b", "opt-13b"])
def test_large_models_sampled_sequences(cuda_device, name):
    cfg = WORKLOADS[name]
    logit_err, lp_err = teacher_forced_check(cfg, torch, steps=STEPS, oracle_seqs=[0, 1])
    assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (name, logit_err, lp_err)


def test_opt125m_graph_replay_and_score(cuda_device):
    """At the full OPT-125M size: the captured graph gives the direct launch's exact
    ids and log-probs, and one he_score pass over prompt + answer reproduces the
    decode path's log-probs within the log-prob bar (sequences 0 and 1 also against
    the oracle, teacher-forced on the GPU's answers)."""
    import numpy as np

    from oracle import OracleModel
    from synth.workloads import make_model, make_prompts
    from tests.gpu_helpers import engine_for

    cfg = WORKLOADS["opt-125m"]
    inputs = make_model(cfg)
    prompts_np = make_prompts(cfg)
    prompts = torch.from_numpy(prompts_np).cuda()
    L = cfg.gen_len
    eng, _w = engine_for(cfg, inputs, torch)
    eng.fuse_lora()
    ids, lps = [t.clone() for t in eng.generate(prompts, L)]
    eng.set_cuda_graph(True)
    for _ in range(2):
        ids_g, lps_g = eng.generate(prompts, L)
        assert torch.equal(ids_g, ids) and torch.equal(lps_g.view(torch.int32), lps.view(torch.int32))
    full = torch.cat([prompts, ids], dim=1).contiguous()
    sc = eng.score(full, cfg.prompt_len)
    torch.cuda.synchronize()
    assert (sc - lps).abs().max().item() < BF16_LP_TOL
    eng.unfuse_lora()
    eng.close()
    oracle = OracleModel(inputs, "merged")
    answers = ids.cpu().numpy()[:2]
    _, lps_o, _ = oracle.generate(prompts_np[:2], L, force_ids=answers)
    assert np.abs(sc.cpu().numpy()[:2] - lps_o).max() < BF16_LP_TOL


@pytest.mark.slow
@pytest.mark.parametrize("name", ["opt-1.3b", "opt-13b"])
def test_large_models_score_sampled_sequences(cuda_device, name):
    """he_score at the full batch and length (256 prompt + 256 answer tokens per
    sequence, one prefill-kernel pass), against the oracle's log-probs of its own
    greedy answer tokens 1..8 for sequences 0 and 1; the other answer tokens are random
    ids (each score row depends only on the tokens before it)."""
    import numpy as np

    from oracle import OracleModel
    from synth.workloads import make_model, make_prompts
    from tests.gpu_helpers import engine_for

    cfg = WORKLOADS[name]
    inputs = make_model(cfg)
    prompts = make_prompts(cfg)
    B, Lp = prompts.shape
    K = 8
    oracle = OracleModel(inputs, "merged")
    ref_ids, ref_lps, _ = oracle.generate(prompts[:2], K)
    del oracle
    answers = np.random.default_rng(7).integers(3, cfg.vocab, size=(B, cfg.gen_len))
    answers = answers.astype(np.int32)
    answers[:2, :K] = ref_ids
    full = np.ascontiguousarray(np.concatenate([prompts, answers], axis=1))
    eng, _w = engine_for(cfg, inputs, torch)
    eng.fuse_lora()
    sc = eng.score(torch.from_numpy(full).cuda(), Lp)
    eng.unfuse_lora()
    eng.check()
    torch.cuda.synchronize()
    err = np.abs(sc.cpu().numpy()[:2, :K] - ref_lps).max()
    assert err < BF16_LP_TOL, (name, err)
    eng.close()
