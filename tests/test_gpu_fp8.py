"""FP8 (E4M3) weight streaming (he_set_weight_format HE_WEIGHTS_FP8).

* the fp8 stream-K GEMM (he_op_linear_fp8) against exact float64 products of the
  decoded codes and their row scales, within the fp32 accumulation bound;
* the fused fp8 weights (codes in the fp8 tiled layout and row scales) against the
  oracle's quantization of the merged weight;
* generation teacher-forced on the oracle's tokens against the oracle's fp8 model
  (weights = codes * scale) at the bf16 bars: logits within 3e-2, log-probs within
  5e-2, fused and unfused, OPT-125M on every sequence and OPT-1.3B / OPT-13B on
  sequences 0 and 1 (prefill row + 8 decode steps);
* graph replay equals direct launch with fp8 weights.
"""
import numpy as np
import pytest
import torch

import decode_opt_step_gb300 as he
from oracle import merge_lora, quantize_rows_e4m3
from synth.workloads import WORKLOADS, make_model, make_prompts
from tests.brute_force import e4m3_values
from tests.gpu_helpers import BF16_LOGIT_TOL, BF16_LP_TOL, engine_for, teacher_forced_check

pytestmark = pytest.mark.gpu

_TABLE = {code: v for v, code in e4m3_values()}


def _decode(codes):
    lut = np.array([_TABLE.get(c, np.nan) for c in range(256)], np.float64)
    return lut[codes]


def tiled8_positions(N, K):
    """Flat position of element (n, k) in the fp8 tiled layout (formula of he_ops.h)."""
    n = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    return (((n // 128) * (K // 128) + k // 128) * 16384 + (n % 128) * 128
            + (((k % 128) // 16) ^ (n % 8)) * 16 + k % 16)


@pytest.mark.parametrize("M,N,K,P", [(1, 128, 256, 0), (16, 256, 768, -5), (33, 512, 1024, 0),
                                     (128, 1280, 5120, 0), (100, 384, 2048, -1),
                                     (64, 2560, 768, -60)])
def test_fp8_stream_k_gemm_matches_exact(cuda_device, M, N, K, P):
    rng = np.random.default_rng(M + N + K)
    valid = np.array([c for c in range(256) if c in _TABLE], np.uint8)
    codes = rng.choice(valid, size=(N, K))
    scale = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    x = (rng.normal(0, 1, (M, K))).astype(np.float16)
    tiled = np.empty(N * K, np.uint8)
    tiled[tiled8_positions(N, K)] = codes
    w = _decode(codes) * scale[:, None].astype(np.float64)
    ref = x.astype(np.float64) @ w.T
    y = he.linear_fp8(torch.from_numpy(x).cuda(), torch.from_numpy(tiled).cuda(),
                      torch.from_numpy(scale).cuda(), N, K, split=P)
    torch.cuda.synchronize()
    bound = K * 2.0 ** -23 * (np.abs(x.astype(np.float64)) @ np.abs(w).T) + 1e-30
    err = np.abs(y.cpu().numpy() - ref)
    assert (err <= 4 * bound).all(), (err / bound).max()


TINY_BF16 = WORKLOADS["opt-tiny-fp32"].with_(name="tiny-bf16-fp8", index=26, dtype="bf16",
                                             d_model=256, n_heads=4, ffn=512, vocab=1000,
                                             batch=3, prompt_len=13, gen_len=9)


def test_fused_fp8_weights_are_the_oracle_quantization(cuda_device):
    cfg = TINY_BF16
    inputs = make_model(cfg)
    eng, _w = engine_for(cfg, inputs, torch)
    eng.set_weight_format("fp8")
    eng.fuse_lora()
    proj = {"wq": he.HE_PROJ_Q, "wo": he.HE_PROJ_O, "w1": he.HE_PROJ_FC1, "w2": he.HE_PROJ_FC2}
    mismatched, total = 0, 0
    for li in range(cfg.n_layers):
        for name, p in proj.items():
            a, b = inputs.lora[li][name]
            q_ref, s_ref = quantize_rows_e4m3(
                merge_lora(inputs.layers[li][name], a, b, cfg.lora_alpha, cfg.lora_r))
            codes, scales = eng.read_fused_fp8(li, p)
            torch.cuda.synchronize()
            N, K = q_ref.shape
            got = _decode(codes.cpu().numpy()[tiled8_positions(N, K)])
            np.testing.assert_allclose(scales.cpu().numpy(), s_ref, rtol=2e-6)
            diff = got != q_ref
            mismatched += int(diff.sum())
            total += diff.size
            # a different code only where the merged value sits at a rounding tie of
            # the two sides' last-bit differences: one E4M3 step apart
            if diff.any():
                step = np.abs(got[diff] - q_ref[diff]) / np.maximum(np.abs(q_ref[diff]), 2.0 ** -9)
                assert (step <= 0.13).all()
    assert mismatched <= max(2, total // 10000), (mismatched, total)
    eng.unfuse_lora()
    with pytest.raises(he.HeError) as e:
        eng.read_fused_fp8(0, he.HE_PROJ_Q)
    assert e.value.status == he.HE_ERR_STATE
    eng.close()


@pytest.mark.parametrize("fused", [True, False])
def test_tiny_fp8_teacher_forced(cuda_device, fused):
    logit_err, lp_err = teacher_forced_check(TINY_BF16, torch, fused=fused, weights="fp8")
    assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (logit_err, lp_err)


def test_opt125m_fp8_all_sequences(cuda_device):
    logit_err, lp_err = teacher_forced_check(WORKLOADS["opt-125m"], torch, steps=range(9),
                                             weights="fp8")
    assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (logit_err, lp_err)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["opt-1.3b", "opt-13b"])
def test_large_models_fp8_sampled_sequences(cuda_device, name):
    logit_err, lp_err = teacher_forced_check(WORKLOADS[name], torch, steps=range(9),
                                             oracle_seqs=[0, 1], weights="fp8")
    assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (name, logit_err, lp_err)


def test_fp8_graph_replay_and_format_switch(cuda_device):
    cfg = TINY_BF16
    inputs = make_model(cfg)
    prompts = torch.from_numpy(make_prompts(cfg)).cuda()
    eng, _w = engine_for(cfg, inputs, torch)
    f16 = [t.clone() for t in eng.generate(prompts, cfg.gen_len)]
    eng.set_weight_format("fp8")
    eng.fuse_lora()
    with pytest.raises(he.HeError) as e:
        eng.set_weight_format("f16")  # not while fused
    assert e.value.status == he.HE_ERR_STATE
    direct = [t.clone() for t in eng.generate(prompts, cfg.gen_len)]
    eng.set_cuda_graph(True)
    for _ in range(2):
        g = eng.generate(prompts, cfg.gen_len)
        assert torch.equal(g[0], direct[0]) and torch.equal(g[1], direct[1])
    eng.unfuse_lora()
    eng.set_weight_format("f16")
    back = eng.generate(prompts, cfg.gen_len)
    assert torch.equal(back[0], f16[0]) and torch.equal(back[1], f16[1])
    eng.close()
