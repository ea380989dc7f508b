"""CUDA-graph generation (he_set_cuda_graph): the replayed graph gives bit-identical
results to the direct launch, across re-captures (fuse / unfuse, released and
retaken workspace, another shape) and through the host-buffer entry point."""
import numpy as np
import pytest
import torch

import decode_opt_step_gb300 as he
from synth.workloads import WORKLOADS, make_model, make_prompts
from tests.gpu_helpers import engine_for

pytestmark = pytest.mark.gpu

TINY_BF16 = WORKLOADS["opt-tiny-fp32"].with_(name="tiny-bf16-graph", index=21, dtype="bf16",
                                             d_model=256, n_heads=4, ffn=512, vocab=1000,
                                             batch=3, prompt_len=13, gen_len=9)


def _same(a, b):
    return all(torch.equal(x.view(torch.int32), y.view(torch.int32)) for x, y in zip(a, b))


@pytest.mark.parametrize("cfg", [WORKLOADS["opt-tiny-fp32"], TINY_BF16], ids=["fp32", "bf16"])
def test_graph_generation_matches_direct(cuda_device, cfg):
    inputs = make_model(cfg)
    prompts = torch.from_numpy(make_prompts(cfg)).cuda()
    eng, _w = engine_for(cfg, inputs, torch)
    L = cfg.gen_len
    direct = [t.clone() for t in eng.generate(prompts, L)]
    eng.fuse_lora()
    direct_fused = [t.clone() for t in eng.generate(prompts, L)]
    eng.unfuse_lora()
    l0 = eng.stats()["launches"]
    eng.generate(prompts, L)
    per_call = eng.stats()["launches"] - l0

    eng.set_cuda_graph(True)
    for _ in range(3):  # capture, then replays
        assert _same(eng.generate(prompts, L), direct)
    l0 = eng.stats()["launches"]
    eng.generate(prompts, L)
    assert eng.stats()["launches"] - l0 == per_call  # the replay counts the captured launches
    eng.fuse_lora()  # another weight buffer and activation type: re-captured
    assert _same(eng.generate(prompts, L), direct_fused)
    assert _same(eng.generate(prompts, L), direct_fused)
    eng.unfuse_lora()
    eng.release_workspace()
    eng.retake_workspace()
    assert _same(eng.generate(prompts, L), direct)
    # another shape, then back
    short = [t.clone() for t in eng.generate(prompts[:2, :7], 4)]
    eng.set_cuda_graph(False)
    assert _same(eng.generate(prompts[:2, :7], 4), short)
    eng.set_cuda_graph(True)
    ids, lps = eng.generate_host(prompts.cpu().numpy(), L)
    assert np.array_equal(ids, direct[0].cpu().numpy())
    assert np.array_equal(lps.view(np.int32), direct[1].cpu().numpy().view(np.int32))
    eng.close()


def test_graph_mode_with_profiling_and_teacher_forcing(cuda_device):
    """Profiling and generate_ex launch directly even with graphs on."""
    cfg = TINY_BF16
    inputs = make_model(cfg)
    prompts = torch.from_numpy(make_prompts(cfg)).cuda()
    eng, _w = engine_for(cfg, inputs, torch)
    ref = [t.clone() for t in eng.generate(prompts, cfg.gen_len)]
    eng.set_cuda_graph(True)
    eng.set_profiling("all")
    assert _same(eng.generate(prompts, cfg.gen_len), ref)
    st = eng.stats()
    assert st["kclass_launches"]["gemm"] > 0
    eng.set_profiling(())
    force = ref[0].clone()
    ids, lps, _ = eng.generate_ex(prompts, cfg.gen_len, force_ids=force)
    # teacher forcing takes the log-prob from the stored logits, free-running greedy
    # decode steps from the LM head's merged tile statistics: the same value up to
    # the order of the fp32 sums
    assert torch.equal(ids, ref[0]) and (lps - ref[1]).abs().max().item() < 2e-5
    assert torch.equal(lps[:, 0], ref[1][:, 0])  # the prefill head takes the same path
    eng.close()
