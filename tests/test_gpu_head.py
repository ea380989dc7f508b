"""The greedy choice fused into the LM-head GEMM (EPI_ARGMAX + the tile merge).

* he_op_head_greedy against the logits of the same stream-K GEMM (he_op_linear):
  the chosen index is the logits' argmax (lowest index on ties) and the log-prob is
  the chosen logit's log-softmax, for ragged vocabularies (a partial last tile),
  batches of 1 to 200 rows and both 16-bit types;
* exact ties planted across tiles and inside a tile resolve to the lowest index;
* inside generation, a free-running greedy decode (fused head) chooses the argmax
  of the logits the teacher-forced path captures for the same tokens, and reports
  the same log-probs.
"""
import numpy as np
import pytest
import torch

import decode_opt_step_gb300 as he
from synth.workloads import WORKLOADS, make_model, make_prompts
from tests.gpu_helpers import engine_for

pytestmark = pytest.mark.gpu


def _ref(logits):
    lg = logits.double().cpu().numpy()
    ids = lg.argmax(axis=1)  # first (lowest) index of the maximum
    m = lg.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(lg - m).sum(axis=1))
    return ids, lg[np.arange(len(ids)), ids] - lse


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("M,N,K", [(1, 1000, 256), (5, 50272, 768), (16, 1028, 512),
                                   (100, 4100, 1024), (128, 50272, 5120), (200, 1000, 256)])
def test_head_greedy_matches_gemm_logits(cuda_device, dt, M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N)
    x = torch.randn(M, K, generator=g).to(dt).cuda()
    w = (torch.randn(N, K, generator=g) * 0.05).to(dt).cuda()
    ids, lp = he.head_greedy(x, w)
    logits = he.linear(x, w, split=0)  # the same stream-K GEMM, fp32 logits stored
    torch.cuda.synchronize()
    ref_ids, ref_lp = _ref(logits)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(lp.cpu().numpy(), ref_lp, atol=2e-5, rtol=0)


def test_head_greedy_exact_ties_take_the_lowest_index(cuda_device):
    # one-hot rows of x pick one column of w, so every logit is one exact weight
    M, N, K = 64, 1000, 256
    rng = np.random.default_rng(5)
    x = np.zeros((M, K), np.float32)
    x[np.arange(M), np.arange(M) * 3 % K] = 1.0
    w = rng.integers(-8, 8, size=(N, K)).astype(np.float32)
    for m in range(M):
        k = m * 3 % K
        ties = np.sort(rng.choice(N, size=2 + m % 4, replace=False))
        if m % 3 == 0:  # a pair inside one 128-row tile, and one across
            t0 = ties[0] // 128 * 128
            ties = np.unique(np.concatenate([[t0 + 5, t0 + 77], ties]))
        w[:, k] = np.minimum(w[:, k], 7)
        w[ties, k] = 100.0
    xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    wt = torch.from_numpy(w).to(torch.bfloat16).cuda()
    ids, lp = he.head_greedy(xt, wt)
    torch.cuda.synchronize()
    lg = x @ w.T
    assert np.array_equal(ids.cpu().numpy(), lg.argmax(axis=1))
    m = lg.max(axis=1, keepdims=True).astype(np.float64)
    ref_lp = -np.log(np.exp(lg - m).sum(axis=1))
    np.testing.assert_allclose(lp.cpu().numpy(), ref_lp, atol=1e-5, rtol=0)


TINY_BF16 = WORKLOADS["opt-tiny-fp32"].with_(name="tiny-bf16-head", index=25, dtype="bf16",
                                             d_model=256, n_heads=4, ffn=512, vocab=1000,
                                             batch=5, prompt_len=13, gen_len=9)


@pytest.mark.parametrize("cfg", [TINY_BF16, WORKLOADS["opt-125m"].with_(gen_len=6)],
                         ids=["tiny", "opt-125m"])
@pytest.mark.parametrize("fused", [True, False])
def test_fused_head_in_generation_matches_logits_path(cuda_device, cfg, fused):
    inputs = make_model(cfg)
    prompts = torch.from_numpy(make_prompts(cfg)).cuda()
    B, L = cfg.batch, cfg.gen_len
    eng, _w = engine_for(cfg, inputs, torch)
    if fused:
        eng.fuse_lora()
    ids, lps = [t.clone() for t in eng.generate(prompts, L)]  # greedy: fused head
    rows = [(b, k) for b in range(B) for k in range(L)]
    ids2, lps2, lg = eng.generate_ex(prompts, L, force_ids=ids, log_rows=rows)
    torch.cuda.synchronize()
    eng.close()
    lg = torch.as_tensor(lg)
    ref_ids, ref_lp = _ref(lg)
    got = np.array([ids[b, k].item() for b, k in rows])
    assert np.array_equal(got, ref_ids)
    lp = np.array([lps[b, k].item() for b, k in rows])
    np.testing.assert_allclose(lp, ref_lp, atol=2e-5, rtol=0)
    np.testing.assert_allclose(lps.cpu().numpy(), lps2.cpu().numpy(), atol=2e-5, rtol=0)
