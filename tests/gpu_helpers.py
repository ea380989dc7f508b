"""Shared helpers of the GPU tests: build an engine from synthetic inputs, run the
CPU oracle on the same inputs, and compare."""
from __future__ import annotations

import numpy as np

from oracle import OracleModel
from synth.torch_io import model_to_device
from synth.workloads import make_model, make_prompts

# Parity bars: fp32 workload ids identical and log-probs within 1e-4 (fp32, different
# summation orders); bf16 workloads teacher-forced logits within 3e-2 max-abs and
# chosen-token log-probs within 5e-2 absolute.
FP32_LP_TOL = 1e-4
BF16_LOGIT_TOL = 3e-2
BF16_LP_TOL = 5e-2


def engine_for(cfg, inputs, torch, max_batch=None, max_seq=None, **kw):
    import decode_opt_step_gb300 as he
    w = model_to_device(inputs, torch.device("cuda:0"), torch)
    eng = he.Engine(cfg, w, max_batch=max_batch or cfg.batch, max_seq=max_seq or cfg.max_seq, **kw)
    return eng, w


def teacher_forced_check(cfg, torch, seqs=None, steps=None, inputs=None, prompts=None,
                         oracle_seqs=None, fused=True, weights="f16"):
    """Runs the GPU path teacher-forced on the oracle's tokens; returns the worst errors.

    ``oracle_seqs``: the sequences the oracle computes (batch rows are independent),
    default all; the GPU runs the whole batch.  ``steps``: the decode steps compared
    (default all).  ``fused``: LoRA merged before generating (oracle "merged"), or
    generation on the base weights without a fuse (oracle "none").  ``weights``: the
    engine's weight format, "f16" (oracle weights "exact") or "fp8" (oracle "fp8").
    """
    inputs = inputs if inputs is not None else make_model(cfg)
    prompts = prompts if prompts is not None else make_prompts(cfg)
    B, Lp = prompts.shape
    oseq = list(range(B)) if oracle_seqs is None else list(oracle_seqs)
    osteps = list(range(cfg.gen_len)) if steps is None else list(steps)
    n_or = max(osteps) + 1
    oracle = OracleModel(inputs, "merged" if fused else "none",
                         weights="fp8" if weights == "fp8" else "exact")
    ref_ids, ref_lps, ref_lg = oracle.generate(prompts[oseq], n_or, log_steps=osteps)
    del oracle
    eng, _w = engine_for(cfg, inputs, torch)
    if weights != "f16":
        eng.set_weight_format(weights)
    if fused:
        eng.fuse_lora()
    force = np.full((B, cfg.gen_len), -1, np.int32)
    force[oseq, :n_or] = ref_ids
    rows = [(b, k) for b in (oseq if seqs is None else seqs) for k in osteps]
    ids, lps, lg = eng.generate_ex(torch.from_numpy(prompts).cuda(), cfg.gen_len,
                                   force_ids=torch.from_numpy(force), log_rows=rows)
    if fused:
        eng.unfuse_lora()
    eng.check()
    torch.cuda.synchronize()
    lg = lg.cpu().numpy()
    lps = lps.cpu().numpy()
    pos = {b: i for i, b in enumerate(oseq)}
    logit_err = max(np.abs(lg[i] - ref_lg[k][pos[b]]).max() for i, (b, k) in enumerate(rows))
    lp_err = max(abs(float(lps[b, k]) - float(ref_lps[pos[b], k])) for b, k in rows)
    eng.close()
    return logit_err, lp_err
