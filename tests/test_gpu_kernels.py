"""Kernel-level GPU tests through the C ABI (he_op_linear) on ragged shapes."""
import numpy as np
import pytest
import torch

import decode_opt_step_gb300 as he

pytestmark = pytest.mark.gpu


def _exact(x, w):
    return x.double().cpu().numpy() @ w.double().cpu().numpy().T


def _bound(x, w, K):
    # fp32 accumulation of K products: |err| <= K * 2^-23 * sum |x_k w_k| (+ slack)
    mag = x.abs().double().cpu().numpy() @ w.abs().double().cpu().numpy().T
    return K * 2.0 ** -23 * mag + 1e-6


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (3, 256, 8), (16, 384, 768), (17, 200, 136),
                                   (100, 640, 1024), (129, 128, 520), (300, 1000, 256),
                                   (513, 384, 64), (4133, 2560, 320)])
def test_linear_16bit_tcgen05_matches_exact(cuda_device, M, N, K, dt):
    g = torch.Generator().manual_seed(M * 7919 + N * 31 + K)
    x = torch.randn(M, K, generator=g).to(dt).cuda()
    w = torch.randn(N, K, generator=g).to(dt).cuda()
    y = he.linear(x, w)
    torch.cuda.synchronize()
    ref = _exact(x, w)
    err = np.abs(y.cpu().numpy() - ref)
    assert (err <= _bound(x, w, K)).all(), f"max err {err.max()}"


@pytest.mark.parametrize("split", [2, 3, 5])
def test_linear_bf16_split_k(cuda_device, split):
    M, N, K = 64, 512, 1280
    g = torch.Generator().manual_seed(split)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    w = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    y = he.linear(x, w, split=split)
    torch.cuda.synchronize()
    err = np.abs(y.cpu().numpy() - _exact(x, w))
    assert (err <= _bound(x, w, K)).all()


def test_linear_bf16_strided_rows(cuda_device):
    # x rows with a stride larger than K (the LM head reads every Lp-th row)
    g = torch.Generator().manual_seed(5)
    big = torch.randn(7 * 9, 256, generator=g).to(torch.bfloat16).cuda()
    x = big[8::9]  # rows 8, 17, ... : stride 9*256
    w = torch.randn(384, 256, generator=g).to(torch.bfloat16).cuda()
    y = he.linear(x, w)
    torch.cuda.synchronize()
    err = np.abs(y.cpu().numpy() - _exact(x, w))
    assert (err <= _bound(x, w, 256)).all()


@pytest.mark.parametrize("M,N,K,split", [(2, 384, 128, 1), (5, 100, 72, 2), (70, 130, 200, 1)])
def test_linear_fp32_cuda_cores(cuda_device, M, N, K, split):
    g = torch.Generator().manual_seed(M + N + K)
    x = torch.randn(M, K, generator=g).cuda()
    w = torch.randn(N, K, generator=g).cuda()
    y = he.linear(x, w, split=split)
    torch.cuda.synchronize()
    err = np.abs(y.cpu().numpy() - _exact(x, w))
    assert (err <= _bound(x, w, K)).all()


def test_linear_rejects_bad_arguments(cuda_device):
    x = torch.zeros(4, 12, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(8, 12, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(he.HeError) as e:
        he.linear(x, w)  # K = 12 is not a multiple of 8 (16-byte TMA rows)
    assert e.value.status == he.HE_ERR_UNSUPPORTED
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(he.HeError):
        he.linear(x, w, split=3)  # K = 64 has one block: no 3-way split


def tiled_positions(N, K):
    """Index of element (n, k) in the tiled streaming layout (as stated in he_ops.h)."""
    n = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    return (((n // 128) * (K // 64) + k // 64) * 8192 + (n % 128) * 64
            + (((k % 64) // 8) ^ (n % 8)) * 8 + k % 8)


@pytest.mark.parametrize("N,K", [(128, 64), (256, 192), (384, 1024)])
def test_tile_weight_layout(cuda_device, N, K):
    g = torch.Generator().manual_seed(N + K)
    w = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    t = he.tile_weight(w)
    torch.cuda.synchronize()
    flat = t.view(torch.int16).cpu().numpy()
    ref = np.empty(N * K, np.int16)
    ref[tiled_positions(N, K).ravel()] = w.view(torch.int16).cpu().numpy().ravel()
    assert np.array_equal(flat, ref)


@pytest.mark.parametrize("M,N,K,split", [(1, 128, 64, 1), (17, 384, 512, 1), (128, 1280, 1024, 1),
                                         (128, 256, 2048, 4), (300, 256, 640, 1), (64, 640, 1280, 5),
                                         (4133, 2560, 192, 1)])
def test_linear_bf16_tiled_weights(cuda_device, M, N, K, split):
    g = torch.Generator().manual_seed(M + 3 * N + 7 * K)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    w = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    y = he.linear(x, w, split=split, w_tiled=he.tile_weight(w))
    torch.cuda.synchronize()
    err = np.abs(y.cpu().numpy() - _exact(x, w))
    assert (err <= _bound(x, w, K)).all(), err.max()


@pytest.mark.parametrize("M,N,K,ctas", [(1, 128, 64, 0), (17, 384, 320, 0), (128, 1280, 1024, 0),
                                        (128, 640, 5120, 0), (200, 256, 512, 0), (64, 384, 640, -1),
                                        (5, 128, 640, -5), (33, 256, 192, -6), (128, 1280, 128, -7),
                                        (9, 512, 1152, -13), (16, 15360, 256, 0),
                                        # 15 runs on one tile: the owner's staged reduction
                                        # does not fit, the register fallback finishes it
                                        (128, 128, 2048, -15), (200, 128, 4096, -15)])
@pytest.mark.parametrize("tiled", [False, True])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_linear_16bit_stream_k(cuda_device, M, N, K, ctas, tiled, dt):
    g = torch.Generator().manual_seed(M * 13 + N + K)
    x = torch.randn(M, K, generator=g).to(dt).cuda()
    w = torch.randn(N, K, generator=g).to(dt).cuda()
    y = he.linear(x, w, split=ctas, w_tiled=he.tile_weight(w) if tiled else None)
    torch.cuda.synchronize()
    err = np.abs(y.cpu().numpy() - _exact(x, w))
    assert (err <= _bound(x, w, K)).all(), err.max()


@pytest.mark.parametrize("M,N,K", [(128, 50272 // 8, 512), (3, 1000, 256), (64, 200, 1024)])
def test_linear_bf16_stream_k_ragged_rows(cuda_device, M, N, K):
    # row-major weights with N not a multiple of 128 (the LM head's vocabulary)
    g = torch.Generator().manual_seed(M + N)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    w = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    y = he.linear(x, w, split=0)
    torch.cuda.synchronize()
    err = np.abs(y.cpu().numpy() - _exact(x, w))
    assert (err <= _bound(x, w, K)).all(), err.max()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("B,H,hd,T,n,split", [(2, 4, 32, 40, 17, 1), (3, 5, 64, 300, 257, 1),
                                              (1, 2, 128, 512, 511, 4), (4, 3, 128, 64, 1, 1),
                                              (2, 2, 64, 200, 133, 3)])
def test_attn_decode_matches_softmax(cuda_device, dtype, B, H, hd, T, n, split):
    g = torch.Generator().manual_seed(B * 100 + n)
    q = (torch.randn(B, H * hd, generator=g) * hd ** -0.5).to(dtype).cuda()
    kc = torch.randn(B, H, T, hd, generator=g).to(dtype).cuda()
    vc = torch.randn(B, H, T, hd, generator=g).to(dtype).cuda()
    ctx = he.attn_decode(q, kc, vc, n, split)
    torch.cuda.synchronize()
    qd = q.double().cpu().view(B, H, 1, hd)
    kd, vd = kc.double().cpu()[:, :, :n], vc.double().cpu()[:, :, :n]
    p = torch.softmax(qd @ kd.transpose(-1, -2), -1)
    ref = (p @ vd).view(B, H * hd).numpy()
    got = ctx.double().cpu().numpy()
    tol = {torch.float32: 1e-5, torch.bfloat16: 1e-2, torch.float16: 2e-3}[dtype]  # output rounding
    np.testing.assert_allclose(got, ref, atol=tol, rtol=tol)


@pytest.mark.parametrize("mma_sync", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("B,H,hd,Lp,T", [(2, 3, 64, 256, 300), (3, 2, 128, 67, 128),
                                         (1, 2, 128, 511, 512), (2, 2, 64, 1, 8),
                                         (1, 3, 128, 129, 160), (2, 1, 64, 384, 384),
                                         (1, 2, 32, 100, 128)])
def test_attn_prefill_matches_causal_softmax(cuda_device, dtype, mma_sync, B, H, hd, Lp, T):
    """he_op_attn_prefill (tcgen05 for hd 64 / 128, mma.sync otherwise or on request)
    against a float64 causal softmax; cache rows past the prompt hold NaN, which no
    kernel may read."""
    g = torch.Generator().manual_seed(B * 1000 + Lp * 7 + hd)
    q = (torch.randn(B, Lp, H * hd, generator=g) * hd ** -0.5).to(dtype).cuda()
    kc = torch.full((B, H, T, hd), float("nan"), dtype=dtype)
    vc = torch.full((B, H, T, hd), float("nan"), dtype=dtype)
    kc[:, :, :Lp] = torch.randn(B, H, Lp, hd, generator=g).to(dtype)
    vc[:, :, :Lp] = torch.randn(B, H, Lp, hd, generator=g).to(dtype)
    kc, vc = kc.cuda(), vc.cuda()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx = he.attn_prefill(q, kc, vc, Lp, mma_sync=mma_sync, dev_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    qd = q.double().cpu().view(B, Lp, H, hd).transpose(1, 2)
    kd, vd = kc.double().cpu()[:, :, :Lp], vc.double().cpu()[:, :, :Lp]
    s = qd @ kd.transpose(-1, -2)
    s = s.masked_fill(torch.ones(Lp, Lp, dtype=torch.bool).triu(1), float("-inf"))
    ref = (torch.softmax(s, -1) @ vd).transpose(1, 2).reshape(B, Lp, H * hd).numpy()
    got = ctx.double().cpu().numpy()
    assert np.isfinite(got).all()
    # probabilities rounded to dtype for the P V product, plus the output rounding
    tol = {torch.bfloat16: 2e-2, torch.float16: 4e-3}[dtype]
    np.testing.assert_allclose(got, ref, atol=tol, rtol=tol)


def test_attn_prefill_tc_equals_reference_rounding_path(cuda_device):
    """The tcgen05 and mma.sync prompt attentions agree to within the rounding of the
    probabilities (they differ only in summation order and exp evaluation)."""
    B, H, hd, Lp, T = 2, 4, 128, 256, 256
    g = torch.Generator().manual_seed(5)
    q = (torch.randn(B, Lp, H * hd, generator=g) * hd ** -0.5).half().cuda()
    kc = torch.randn(B, H, T, hd, generator=g).half().cuda()
    vc = torch.randn(B, H, T, hd, generator=g).half().cuda()
    a = he.attn_prefill(q, kc, vc, Lp).float()
    b = he.attn_prefill(q, kc, vc, Lp, mma_sync=True).float()
    torch.cuda.synchronize()
    assert (a - b).abs().max().item() < 4e-3


@pytest.mark.parametrize("N,K,r", [(256, 192, 8), (384, 640, 16), (128, 64, 8), (256, 320, 4),
                                   (256, 192, 24), (1280, 512, 8)])
def test_fuse_tiled_is_one_rounding_of_the_merge(cuda_device, N, K, r):
    """he_op_fuse_tiled (one projection of the bf16 fuse): fp16 of W + scale B A, tiled;
    r = 8 and 16 take the tensor-core kernel, other ranks the SIMT one."""
    scale = 2.0
    g = torch.Generator().manual_seed(11 + N + K + r)
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    a = (torch.randn(r, K, generator=g) * 0.02).to(torch.bfloat16)
    b = (torch.randn(N, r, generator=g) * 0.02).to(torch.bfloat16)
    out = he.fuse_tiled(w.cuda(), a.cuda(), b.cuda(), scale)
    torch.cuda.synchronize()
    exact = w.double() + scale * (b.double() @ a.double())
    got = out.double().cpu().numpy()[tiled_positions(N, K)]
    ex = exact.numpy()
    assert (np.abs(got - ex) <= np.abs(ex) * 2.0 ** -11 * 1.001 + 2.0 ** -24).all()
    plain = he.fuse_tiled(w.cuda())  # r = 0: the weight rounded to fp16 (exact above 2^-14)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(plain.double().cpu().numpy()[tiled_positions(N, K)],
                                  w.to(torch.float16).double().numpy())
