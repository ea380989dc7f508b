"""bench.py's algorithmic accounting -- the denominators of its GB/s, TFLOP/s and
roofline figures -- against counts written out here for the OPT-13B workload
(40 layers, d = 5120, ffn = 20480, vocab 50272, B = 128, 256-token prompts and answers)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth.workloads import WORKLOADS  # noqa: E402

CFG = WORKLOADS["opt-13b"]
L, D, F, V, H, HD = 40, 5120, 20480, 50272, 40, 128
B, LP, LGEN = 128, 256, 256


def test_workload_shape():
    assert (CFG.n_layers, CFG.d_model, CFG.ffn, CFG.vocab, CFG.n_heads, CFG.head_dim) == \
        (L, D, F, V, H, HD)
    assert (CFG.batch, CFG.prompt_len, CFG.gen_len) == (B, LP, LGEN)


def test_decode_step_bytes():
    # per layer: q, k, v, out (d x d each) and fc1, fc2 (d x ffn each), 2 bytes; the tied
    # head reads the vocab x d embedding once per step
    q = k = v = o = D * D * 2
    fc1 = fc2 = D * F * 2
    weights = L * (q + k + v + o + fc1 + fc2) + V * D * 2
    assert weights == 25_680_609_280
    for step in (1, 100, LGEN - 1):
        n_keys = LP + step  # cached positions 0 .. Lp + step - 1, the new one included
        kv_read = L * B * n_keys * (D + D) * 2  # K and V rows of every cached position
        kv_write = L * B * (D + D) * 2  # the step's own K and V rows
        total, w, kv = bench.decode_step_bytes(CFG, step, B, LP)
        assert (w, kv, total) == (weights, kv_read + kv_write, weights + kv_read + kv_write)
    # the mean over the 255 decode steps is the figure decode GB/s divides by
    mean = sum(bench.decode_step_bytes(CFG, s, B, LP)[0] for s in range(1, LGEN)) / (LGEN - 1)
    by_hand = weights + L * B * 2 * D * 2 * (LP + sum(range(1, LGEN)) / (LGEN - 1) + 1)
    assert abs(mean - by_hand) < 1.0
    assert abs(mean / 1e9 - 66.05) < 0.01


def test_attention_bytes_per_launch():
    # one layer at 384 cached keys (step 128): K and V, B x 384 rows of d values, 2 bytes
    assert bench.attn_decode_bytes(CFG, 128, B, LP) == 2 * B * 384 * D * 2 == 1_006_632_960


def test_prefill_flops():
    proj_macs_per_token = L * (4 * D * D + 2 * D * F)
    # causal pairs (query t sees keys 0..t), counted one by one
    pairs = sum(t + 1 for t in range(LP))
    attn = L * B * H * pairs * HD * 2 * 2  # q.k and p.v, one multiply-add = 2 flops each
    head = B * D * V * 2  # last prompt row of every sequence against the vocabulary
    total, proj = bench.prefill_flops(CFG, B, LP)
    assert proj == 2 * B * LP * proj_macs_per_token
    assert total == proj + attn + head
    assert abs(proj / 1e12 - 824.6) < 0.1
