"""Synthetic-input generator: known answers, determinism, distribution (CPU only)."""
import numpy as np
import torch

import synth
from synth.workloads import WORKLOADS, make_prompts, make_layer


def test_splitmix64_known_answers():
    # Published SplitMix64 outputs for the initial state 1234567.
    assert synth.splitmix64_sequence(1234567, 5) == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_counter_access_matches_sequential_stream():
    # draw n of a stream equals the n-th sequential output from the stream key's state
    seq = synth.splitmix64_sequence(0, 4)
    assert all(isinstance(v, int) for v in seq)
    a = [synth.raw_draw(7, 11, n) for n in range(6)]
    b = [synth.raw_draw(7, 11, n) for n in range(6)]
    assert a == b and len(set(a)) == 6


def test_normal_moments_and_independence_of_streams():
    z = synth.normal((1 << 20,), 5, 1, 0.0, 1.0, "f32").astype(np.float64)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1) < 5e-3
    w = synth.normal((1 << 20,), 5, 2, 0.0, 1.0, "f32").astype(np.float64)
    assert abs(np.corrcoef(z, w)[0, 1]) < 5e-3


def test_bf16_output_is_round_to_nearest_even_of_f32():
    f = synth.normal((4097,), 9, 3, 0.0, 0.02, "f32")
    b = synth.normal((4097,), 9, 3, 0.0, 0.02, "bf16")
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)


def test_prompts_in_range_and_deterministic():
    cfg = WORKLOADS["opt-125m"]
    p = make_prompts(cfg)
    assert p.shape == (16, 256) and p.min() >= 3 and p.max() < cfg.vocab
    assert np.array_equal(p, make_prompts(cfg))


def test_layer_shapes_and_init():
    cfg = WORKLOADS["opt-tiny-fp32"]
    lw = make_layer(cfg, 0)
    assert lw["w1"].shape == (cfg.ffn, cfg.d_model) and lw["w2"].shape == (cfg.d_model, cfg.ffn)
    assert np.all(lw["ln1_g"] == 1) and np.all(lw["b1"] == 0)
    assert abs(lw["w1"].std() - 0.02) < 1e-3
