"""he_op_attn_decode_noalloc through the C ABI: same results as he_op_attn_decode
(which takes caller scratch), on two calls in a row, and a clear error past the
built-in scratch size.  Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

import decode_opt_step_gb300 as he

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 4 * 1024 * 1024  # the documented built-in scratch


def _inputs(seed, B, H, hd, T, dtype):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H * hd, generator=g) * hd ** -0.5).to(dtype).cuda()
    kc = torch.randn(B, H, T, hd, generator=g).to(dtype).cuda()
    vc = torch.randn(B, H, T, hd, generator=g).to(dtype).cuda()
    return q, kc, vc


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_noalloc_matches_caller_scratch_twice(cuda_device, dtype):
    # Same kernels, same key slices and the same merge order as he_op_attn_decode with
    # caller scratch, so the results are bit-identical.  Two different calls in a row:
    # the second must not see the first's partials.  split 1 uses no scratch; the last
    # case fills the built-in scratch almost to its limit (4126720 of 4194304 floats).
    cases = [(8, 8, 128, 512, 301, 8), (3, 5, 64, 200, 133, 3), (4, 6, 32, 96, 77, 1),
             (128, 8, 128, 512, 500, 31)]
    for seed, (B, H, hd, T, n, split) in enumerate(cases):
        assert B * H * split * (hd + 2) <= SCRATCH_FLOATS
        q, kc, vc = _inputs(seed, B, H, hd, T, dtype)
        ref = he.attn_decode(q, kc, vc, n, split)
        got = he.attn_decode_noalloc(q, kc, vc, n, split)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16 if dtype != torch.float32 else torch.int32),
                           ref.view(torch.int16 if dtype != torch.float32 else torch.int32)), \
            (B, H, hd, n, split)


def test_noalloc_rejects_sizes_past_the_scratch(cuda_device):
    B, H, hd, T = 128, 40, 128, 64
    q, kc, vc = _inputs(7, B, H, hd, T, torch.float16)
    split = 64  # 128 * 40 * 64 * 130 floats > 4194304
    assert B * H * split * (hd + 2) > SCRATCH_FLOATS
    with pytest.raises(he.HeError) as e:
        he.attn_decode_noalloc(q, kc, vc, T, split)
    assert e.value.status == he.HE_ERR_ARG and "16 MiB" in str(e.value)
