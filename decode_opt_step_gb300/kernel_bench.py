"""Microbenchmark of single kernels at the OPT-13B decode shapes (B = 128).

    python -m decode_opt_step_gb300.kernel_bench
        [attn_decode|gemm_sk|gemm_prefill|fuse|attn_prefill|all] [--iters N] [--batch B]

Small, self-contained cases (a few GB on the device) that run one kernel of the
generation path the way a decode step does, for profiling one kernel at a time:

* attn_decode: one decode-attention launch, B=128, 40 heads of 128, 384 cached
  keys (1.0 GB of K and V, above the 126 MB L2);
* gemm_sk: the fc1 projection, 128 tokens x 5120 -> 20480, tiled weights,
  stream-K over one CTA per SM (210 MB of weights, two copies alternated);
* fuse: the LoRA merge of the fc1 projection, 20480 x 5120, r = 8, bf16 in and fp16
  out in the tiled layout (420 MB moved, two weights alternated);
* attn_prefill: the causal prompt attention of one layer, B=128 (--batch) prompts
  of 256 tokens, 40 heads of 128, fp16, tcgen05 and mma.sync kernels (1.34 GB of
  q, K, V and ctx at B=128);
* gemm_prefill: the fc1 projection of a prefill, 32768 tokens (128 prompts of
  256) x 5120 -> 20480, tiled weights, the persistent tensor-core kernel
  (fp32 output, 3.3 GB in all).

Prints the CUDA-event time per launch and the algorithmic GB/s (TFLOP/s for
the prefill GEMM).
"""
from __future__ import annotations

import argparse

import torch

import decode_opt_step_gb300 as he


def _time(fn, iters):
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(iters):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def attn_decode(iters):
    B, H, hd, T, n = 128, 40, 128, 512, 384
    q = (torch.randn(B, H * hd, device="cuda") * hd ** -0.5).to(torch.bfloat16)
    kc = torch.randn(B, H, T, hd, device="cuda").to(torch.bfloat16)
    vc = torch.randn(B, H, T, hd, device="cuda").to(torch.bfloat16)
    ms = _time(lambda i: he.attn_decode(q, kc, vc, n), iters)
    byts = 2 * B * H * n * hd * 2
    print(f"attn_decode B={B} H={H} hd={hd} keys={n}: {ms * 1e3:.1f} us/launch, "
          f"{byts / (ms / 1e3) / 1e9:.0f} GB/s")


def fuse(iters):
    N, K, r = 20480, 5120, 8
    ws = [torch.randn(N, K, device="cuda").to(torch.bfloat16) * 0.02 for _ in range(2)]
    a = (torch.randn(r, K, device="cuda") * 0.02).to(torch.bfloat16)
    b = (torch.randn(N, r, device="cuda") * 0.02).to(torch.bfloat16)
    ms = _time(lambda i: he.fuse_tiled(ws[i % 2], a, b, 2.0), iters)
    byts = N * K * 4
    print(f"fuse (LoRA merge into the fp16 tiled layout) N={N} K={K} r={r}: {ms * 1e3:.1f} "
          f"us/launch, {byts / (ms / 1e3) / 1e9:.0f} GB/s (bf16 read + fp16 write)")


def gemm_sk(iters):
    M, N, K = 128, 20480, 5120
    ws = [torch.randn(N, K, device="cuda").to(torch.bfloat16) for _ in range(2)]
    wt = [he.tile_weight(w) for w in ws]
    x = torch.randn(M, K, device="cuda").to(torch.bfloat16)
    ms = _time(lambda i: he.linear(x, ws[i % 2], split=0, w_tiled=wt[i % 2]), iters)
    print(f"gemm_sk M={M} N={N} K={K} (with the op's input tiling and slice reduction): "
          f"{ms * 1e3:.1f} us/call, {N * K * 2 / (ms / 1e3) / 1e9:.0f} GB/s of weights")


def gemm_prefill(iters):
    M, N, K = 32768, 20480, 5120
    w = torch.randn(N, K, device="cuda").to(torch.bfloat16)
    wt = he.tile_weight(w)
    x = torch.randn(M, K, device="cuda").to(torch.bfloat16)
    ms = _time(lambda i: he.linear(x, w, split=1, w_tiled=wt), iters)
    print(f"gemm_prefill M={M} N={N} K={K}: {ms * 1e3:.1f} us/call, "
          f"{2 * M * N * K / (ms / 1e3) / 1e12:.0f} TFLOP/s")


def attn_prefill(iters, B=128):
    H, hd, Lp, T = 40, 128, 256, 512
    q = (torch.randn(B, Lp, H * hd, device="cuda") * hd ** -0.5).half()
    kc = torch.randn(B, H, T, hd, device="cuda").half()
    vc = torch.randn(B, H, T, hd, device="cuda").half()
    byts = 4 * B * Lp * H * hd * 2  # q, k, v read once, ctx written
    flops = 4 * B * H * hd * Lp * (Lp + 1) // 2
    for name, mma in (("tcgen05", False), ("mma.sync", True)):
        ms = _time(lambda i: he.attn_prefill(q, kc, vc, Lp, mma_sync=mma), iters)
        print(f"attn_prefill[{name}] B={B} H={H} hd={hd} Lp={Lp}: {ms * 1e3:.1f} us/launch, "
              f"{byts / (ms / 1e3) / 1e9:.0f} GB/s, {flops / (ms / 1e3) / 1e12:.0f} TFLOP/s")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", nargs="?", default="all",
                    choices=["attn_decode", "gemm_sk", "gemm_prefill", "fuse", "attn_prefill",
                             "all"])
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--batch", type=int, default=128, help="attn_prefill: prompts")
    args = ap.parse_args()
    torch.cuda.set_device(0)
    if args.case in ("attn_decode", "all"):
        attn_decode(args.iters)
    if args.case in ("gemm_sk", "all"):
        gemm_sk(args.iters)
    if args.case in ("gemm_prefill", "all"):
        gemm_prefill(args.iters)
    if args.case in ("fuse", "all"):
        fuse(args.iters)
    if args.case in ("attn_prefill", "all"):
        attn_prefill(args.iters, args.batch)


if __name__ == "__main__":
    main()
