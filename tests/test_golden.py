"""The oracle still reproduces its frozen tiny fp32 results (tests/golden/, CPU only)."""
import json
import os

import numpy as np
import pytest

from oracle import OracleModel
from synth.workloads import WORKLOADS, make_model, make_prompts

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name", ["opt-tiny-fp32", "opt-tiny-fp32-bias"])
def test_oracle_reproduces_golden(name):
    with open(os.path.join(GOLDEN, f"{name}.json")) as f:
        g = json.load(f)
    cfg = WORKLOADS[name]
    prompts = make_prompts(cfg)
    assert prompts.tolist() == g["prompts"]
    ids, lps, _ = OracleModel(make_model(cfg)).generate(prompts, cfg.gen_len)
    assert ids.tolist() == g["ids"]
    np.testing.assert_allclose(lps, np.array(g["logprobs"]), atol=1e-6, rtol=0)
