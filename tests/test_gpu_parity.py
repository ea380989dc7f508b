"""End-to-end parity of the CUDA path with the CPU oracle (small and medium sizes)."""
import numpy as np
import pytest
import torch

import decode_opt_step_gb300 as he
from oracle import OracleModel
from synth.workloads import WORKLOADS, make_model, make_prompts
from tests.gpu_helpers import (BF16_LOGIT_TOL, BF16_LP_TOL, FP32_LP_TOL, engine_for,
                               teacher_forced_check)

pytestmark = pytest.mark.gpu

TINY_BF16 = WORKLOADS["opt-tiny-fp32"].with_(name="tiny-bf16", index=20, dtype="bf16",
                                             d_model=256, n_heads=4, ffn=512, vocab=1000,
                                             batch=3, prompt_len=13, gen_len=9)


@pytest.mark.parametrize("name", ["opt-tiny-fp32", "opt-tiny-fp32-bias"])
def test_fp32_ids_identical_to_oracle(cuda_device, name):
    cfg = WORKLOADS[name]
    inputs = make_model(cfg)
    prompts = make_prompts(cfg)
    ref_ids, ref_lps, _ = OracleModel(inputs).generate(prompts, cfg.gen_len)
    eng, _w = engine_for(cfg, inputs, torch)
    eng.fuse_lora()
    ids, lps = eng.generate(torch.from_numpy(prompts).cuda(), cfg.gen_len)
    eng.unfuse_lora()
    eng.check()
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.abs(lps.cpu().numpy() - ref_lps).max() < FP32_LP_TOL
    eng.close()


def test_fp32_ragged_batch_and_lengths(cuda_device):
    cfg = WORKLOADS["opt-tiny-fp32-bias"].with_(batch=5, prompt_len=67, gen_len=30, max_pos=128)
    inputs = make_model(cfg)
    prompts = make_prompts(cfg)
    ref_ids, ref_lps, _ = OracleModel(inputs).generate(prompts, cfg.gen_len)
    eng, _w = engine_for(cfg, inputs, torch, max_batch=8, max_seq=100)
    eng.fuse_lora()
    ids, lps = eng.generate(torch.from_numpy(prompts).cuda(), cfg.gen_len)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.abs(lps.cpu().numpy() - ref_lps).max() < FP32_LP_TOL
    eng.close()


def test_bf16_tiny_teacher_forced(cuda_device):
    logit_err, lp_err = teacher_forced_check(TINY_BF16, torch)
    assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (logit_err, lp_err)


@pytest.mark.parametrize("heads", [2, 4, 8])  # head_dim 128, 64, 32
def test_bf16_head_dims_and_ragged_prompt(cuda_device, heads):
    cfg = TINY_BF16.with_(n_heads=heads, batch=2, prompt_len=131, gen_len=5, max_pos=160)
    logit_err, lp_err = teacher_forced_check(cfg, torch)
    assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (heads, logit_err, lp_err)


def test_bf16_ragged_batches(cuda_device):
    for b in (1, 17, 33):
        cfg = TINY_BF16.with_(batch=b, prompt_len=70, gen_len=6, max_pos=128)
        logit_err, lp_err = teacher_forced_check(cfg, torch)
        assert logit_err < BF16_LOGIT_TOL and lp_err < BF16_LP_TOL, (b, logit_err, lp_err)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fuse_unfuse_restores_bits(cuda_device, dtype):
    cfg = TINY_BF16 if dtype == "bf16" else WORKLOADS["opt-tiny-fp32"]
    inputs = make_model(cfg)
    eng, w = engine_for(cfg, inputs, torch)
    before = [{k: v.clone() for k, v in lw.items()} for lw in w["layers"]]
    eng.fuse_lora()
    torch.cuda.synchronize()
    changed = sum(int(not torch.equal(w["layers"][0][k], before[0][k]))
                  for k in ("wq", "wk", "wv", "wo", "w1", "w2"))
    # fp32 engines merge in place; bf16 engines write the merge to their own buffer
    assert changed == (6 if dtype == "f32" else 0)
    eng.unfuse_lora()
    torch.cuda.synchronize()
    for lw, ref in zip(w["layers"], before):
        for k in ref:
            assert torch.equal(lw[k].view(torch.int16) if lw[k].dtype == torch.bfloat16
                               else lw[k].view(torch.int32),
                               ref[k].view(torch.int16) if ref[k].dtype == torch.bfloat16
                               else ref[k].view(torch.int32)), k
    eng.close()


def test_fused_weight_is_rounded_merge(cuda_device):
    cfg = TINY_BF16
    inputs = make_model(cfg)
    eng, w = engine_for(cfg, inputs, torch)
    eng.fuse_lora()
    torch.cuda.synchronize()
    from oracle import merge_lora
    proj = {"wq": he.HE_PROJ_Q, "w1": he.HE_PROJ_FC1, "w2": he.HE_PROJ_FC2}
    for li in (0, cfg.n_layers - 1):
        for name in ("wq", "w1", "w2"):
            a, b = inputs.lora[li][name]
            exact = merge_lora(inputs.layers[li][name], a, b, cfg.lora_alpha, cfg.lora_r)
            t = w["layers"][li][name]
            # while fused, generation reads fp16 in the tiled layout
            flat = eng.read_fused_weight(li, proj[name]).float().cpu().numpy()
            from tests.test_gpu_kernels import tiled_positions
            got = flat[tiled_positions(*t.shape)]
            # one fp16 rounding of the fp32 merge: half an ulp, 2^-11 relative
            # (2^-25 absolute in the subnormal range)
            assert (np.abs(got - exact) <= np.abs(exact) * 2.0 ** -11 + 2.0 ** -25).all(), name
    eng.unfuse_lora()
    with pytest.raises(he.HeError) as e:
        eng.read_fused_weight(0, he.HE_PROJ_Q)
    assert e.value.status == he.HE_ERR_STATE
    eng.close()


def test_release_retake_and_state_errors(cuda_device):
    cfg = WORKLOADS["opt-tiny-fp32"]
    inputs = make_model(cfg)
    prompts = torch.from_numpy(make_prompts(cfg)).cuda()
    eng, _w = engine_for(cfg, inputs, torch)
    with pytest.raises(he.HeError) as e:
        eng.unfuse_lora()
    assert e.value.status == he.HE_ERR_STATE
    eng.fuse_lora()
    with pytest.raises(he.HeError) as e:
        eng.fuse_lora()
    assert e.value.status == he.HE_ERR_STATE
    ids1, lps1 = eng.generate(prompts, cfg.gen_len)
    torch.cuda.synchronize()
    ids1, lps1 = ids1.cpu(), lps1.cpu()
    eng.release_workspace()
    assert eng.stats()["workspace_bytes"] == 0
    with pytest.raises(he.HeError) as e:
        eng.generate(prompts, cfg.gen_len)
    assert e.value.status == he.HE_ERR_STATE
    with pytest.raises(he.HeError) as e:
        eng.release_workspace()
    assert e.value.status == he.HE_ERR_STATE
    eng.retake_workspace()
    ids2, lps2 = eng.generate(prompts, cfg.gen_len)
    torch.cuda.synchronize()
    assert torch.equal(ids1, ids2.cpu()) and torch.equal(lps1, lps2.cpu())
    eng.unfuse_lora()
    with pytest.raises(he.HeError) as e:
        eng.generate(prompts, cfg.max_seq)  # Lp + Lgen > max_seq
    assert e.value.status == he.HE_ERR_ARG
    big = torch.zeros((cfg.batch + 1, cfg.prompt_len), dtype=torch.int32, device="cuda")
    with pytest.raises(he.HeError) as e:
        eng.generate(big, 2)
    assert e.value.status == he.HE_ERR_ARG
    eng.close()


def test_out_of_range_token_is_reported(cuda_device):
    cfg = WORKLOADS["opt-tiny-fp32"]
    inputs = make_model(cfg)
    p = make_prompts(cfg)
    p[1, 3] = cfg.vocab + 5
    eng, _w = engine_for(cfg, inputs, torch)
    eng.generate(torch.from_numpy(p).cuda(), 2)
    with pytest.raises(he.HeError) as e:
        eng.check()
    assert e.value.status == he.HE_ERR_DEVICE_CHECK
    eng.check()  # cleared
    eng.close()


def test_minimal_shapes(cuda_device):
    # B = 1, Lp = 1, Lgen = 1: only the prefill pass and its head
    cfg = WORKLOADS["opt-tiny-fp32"].with_(batch=1, prompt_len=1, gen_len=1)
    inputs = make_model(cfg)
    prompts = make_prompts(cfg)
    # no fuse: the engine runs the base weights, the oracle's "none" model
    ref_ids, ref_lps, _ = OracleModel(inputs, "none").generate(prompts, 1)
    eng, _w = engine_for(cfg, inputs, torch)
    ids, lps = eng.generate(torch.from_numpy(prompts).cuda(), 1)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.abs(lps.cpu().numpy() - ref_lps).max() < FP32_LP_TOL
    eng.close()


def test_allocator_failure_leaves_engine_usable(cuda_device):
    cfg = WORKLOADS["opt-tiny-fp32"]
    inputs = make_model(cfg)
    prompts = torch.from_numpy(make_prompts(cfg)).cuda()
    fail = {"on": False}
    eng, _w = engine_for(cfg, inputs, torch, alloc_filter=lambda n: not fail["on"])
    eng.release_workspace()
    fail["on"] = True
    with pytest.raises(he.HeError) as e:
        eng.retake_workspace()
    assert e.value.status == he.HE_ERR_OOM
    with pytest.raises(he.HeError) as e:
        eng.fuse_lora()  # the restore copy cannot be taken either
    assert e.value.status == he.HE_ERR_OOM
    fail["on"] = False
    eng.retake_workspace()
    eng.fuse_lora()
    ids, _ = eng.generate(prompts, cfg.gen_len)
    torch.cuda.synchronize()
    assert ids.shape == (cfg.batch, cfg.gen_len)
    eng.close()


def test_host_buffer_entry_matches_device_entry(cuda_device):
    cfg = TINY_BF16
    inputs = make_model(cfg)
    prompts = make_prompts(cfg)
    eng, _w = engine_for(cfg, inputs, torch)
    eng.fuse_lora()
    ids_d, lps_d = eng.generate(torch.from_numpy(prompts).cuda(), cfg.gen_len)
    ids_h, lps_h = eng.generate_host(prompts, cfg.gen_len)
    assert np.array_equal(ids_d.cpu().numpy(), ids_h)
    assert np.array_equal(lps_d.cpu().numpy(), lps_h)
    eng.close()
