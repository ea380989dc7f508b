"""Writes the oracle's tiny fp32 generation results to tests/golden/ (calls only oracle/).

Run:  python tests/golden/make_golden.py
The pages print no worked example; these files freeze the pinned oracle's output
for the tiny fp32 workloads so that an unintended change to it shows up.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import OracleModel  # noqa: E402
from synth.workloads import WORKLOADS, make_model, make_prompts  # noqa: E402


def main():
    for name in ("opt-tiny-fp32", "opt-tiny-fp32-bias"):
        cfg = WORKLOADS[name]
        inputs = make_model(cfg)
        prompts = make_prompts(cfg)
        ids, lps, _ = OracleModel(inputs).generate(prompts, cfg.gen_len)
        out = {"workload": name, "prompts": prompts.tolist(), "ids": ids.tolist(),
               "logprobs": [[float(f"{v:.7g}") for v in row] for row in lps.tolist()]}
        with open(os.path.join(HERE, f"{name}.json"), "w") as f:
            json.dump(out, f, indent=None)
            f.write("\n")


if __name__ == "__main__":
    main()
