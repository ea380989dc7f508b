"""he_score: teacher-forced log-probs of an answer in one forward pass, against the
oracle (teacher-forced on the same tokens) and against the decode path."""
import numpy as np
import pytest
import torch

import decode_opt_step_gb300 as he
from oracle import OracleModel
from synth.workloads import WORKLOADS, make_model, make_prompts
from tests.gpu_helpers import BF16_LP_TOL, FP32_LP_TOL, engine_for

pytestmark = pytest.mark.gpu

TINY_BF16 = WORKLOADS["opt-tiny-fp32"].with_(name="tiny-bf16-score", index=22, dtype="bf16",
                                             d_model=256, n_heads=4, ffn=512, vocab=1000,
                                             batch=3, prompt_len=13, gen_len=9)


@pytest.mark.parametrize("cfg,tol", [(WORKLOADS["opt-tiny-fp32"], FP32_LP_TOL),
                                     (WORKLOADS["opt-tiny-fp32-bias"], FP32_LP_TOL),
                                     (TINY_BF16, BF16_LP_TOL)], ids=["fp32", "fp32-bias", "bf16"])
def test_score_matches_oracle_teacher_forced(cuda_device, cfg, tol):
    inputs = make_model(cfg)
    prompts = make_prompts(cfg)
    B, Lp = prompts.shape
    L = Lp + cfg.gen_len
    oracle = OracleModel(inputs, lora="merged")
    ids_o, lps_o, _ = oracle.generate(prompts, cfg.gen_len)
    answers = np.asarray(ids_o, dtype=np.int32)
    full = np.concatenate([prompts, answers], axis=1).astype(np.int32)
    # the oracle's own teacher-forced log-probs of these answers are its greedy ones
    eng, _w = engine_for(cfg, inputs, torch)
    eng.fuse_lora()
    got = eng.score(torch.from_numpy(full).cuda(), Lp)
    torch.cuda.synchronize()
    err = np.abs(got.cpu().numpy() - np.asarray(lps_o)).max()
    assert err < tol, err
    # the decode path, teacher-forced on the same answers, agrees within the same bar
    ids_g, lps_g, _ = eng.generate_ex(torch.from_numpy(prompts).cuda(), cfg.gen_len,
                                      force_ids=torch.from_numpy(answers).cuda())
    assert torch.equal(ids_g.cpu(), torch.from_numpy(answers))
    assert np.abs(got.cpu().numpy() - lps_g.cpu().numpy()).max() < tol
    eng.unfuse_lora()
    eng.close()


def test_score_arguments(cuda_device):
    cfg = WORKLOADS["opt-tiny-fp32"]
    inputs = make_model(cfg)
    eng, _w = engine_for(cfg, inputs, torch)
    ids = torch.zeros((2, cfg.max_seq + 1), dtype=torch.int32, device="cuda")
    with pytest.raises(he.HeError):
        eng.score(ids, 4)  # longer than max_seq
    with pytest.raises(he.HeError):
        eng.score(ids[:, :10], 10)  # no answer token
    eng.release_workspace()
    with pytest.raises(he.HeError) as e:
        eng.score(ids[:, :10], 4)
    assert e.value.status == he.HE_ERR_STATE
    eng.close()
