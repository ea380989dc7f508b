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
