"""Pins of the CPU oracle to things other than itself (CPU only).

* an independent float64 brute-force decoder with explicit loops (tests/brute_force.py);
* torch's own pre-LN transformer layer (nn.TransformerEncoderLayer, norm_first=True,
  ReLU, causal mask) in float64, and torch's layer_norm / logsumexp;
* invariants the pages state: the incremental KV cache gives the same logits as a
  full recompute; the LoRA-merged forward equals base + explicit low-rank branch;
* closed forms and special cases: zero layer weights, constant LayerNorm input,
  uniform attention, zero LoRA B factor, exact ties, log-prob identities;
* mutation checks: plausible mistakes planted in the oracle (on the CPU) must
  fail the brute-force pin.
"""
import math

import numpy as np
import pytest
import torch

from oracle import opt_oracle as oo
from oracle.opt_oracle import OracleModel, layer_norm, log_softmax_pick, greedy, merge_lora
from synth.workloads import WORKLOADS, OptConfig, make_model, make_prompts
from tests.brute_force import BruteForce

# A tiny model with large weights so that every term of the layer moves the logits.
BF_CFG = OptConfig("bf-tiny", 9, 1, 8, 2, 32, 16, 16, "f32", 2, 5, 6, init_std=0.5,
                   bias_std=0.3, ln_gamma_std=0.3, ln_beta_std=0.3)
BF_CFG2 = BF_CFG.with_(name="bf-tiny-2l", index=10, n_layers=2, init_std=0.4)


def _bf_case(cfg):
    inputs = make_model(cfg)
    prompts = make_prompts(cfg)
    return inputs, prompts


@pytest.mark.parametrize("cfg", [BF_CFG, BF_CFG2], ids=lambda c: c.name)
def test_oracle_matches_fp64_brute_force(cfg):
    inputs, prompts = _bf_case(cfg)
    bf = BruteForce(inputs)
    ids, lps, logged = OracleModel(inputs).generate(prompts, cfg.gen_len,
                                                   log_steps=range(cfg.gen_len))
    for b in range(cfg.batch):
        bids, blps, brows = bf.generate(prompts[b], cfg.gen_len)
        assert list(ids[b]) == bids
        np.testing.assert_allclose(lps[b], blps, atol=1e-5, rtol=0)
        for k in range(cfg.gen_len):
            np.testing.assert_allclose(logged[k][b], brows[k], atol=1e-5, rtol=1e-5)


def test_brute_force_pin_catches_planted_mistakes(monkeypatch):
    """Each plausible slip below, planted in the oracle, must break the brute-force pin."""
    inputs, prompts = _bf_case(BF_CFG)
    bf = BruteForce(inputs)
    _, ref_lps, ref_rows = bf.generate(prompts[0], BF_CFG.gen_len)
    ref = np.array(ref_rows)

    def deviation(model):
        _, _, logged = model.generate(prompts[:1], BF_CFG.gen_len, log_steps=range(BF_CFG.gen_len))
        return max(np.abs(logged[k][0] - ref[k]).max() for k in range(BF_CFG.gen_len))

    assert deviation(OracleModel(inputs)) < 1e-5

    class NoPosOffset(OracleModel):
        def embed(self, ids, positions):
            return self.tok_emb[ids] + self.pos_emb[positions]

    assert deviation(NoPosOffset(inputs)) > 1e-3

    def unbiased_ln(x, g, b, eps):
        mean = x.mean(axis=-1, keepdims=True)
        var = x.var(axis=-1, keepdims=True, ddof=1)
        return (x - mean) / np.sqrt(var + eps) * g + b

    with monkeypatch.context() as m:
        m.setattr(oo, "layer_norm", unbiased_ln)
        assert deviation(OracleModel(inputs)) > 1e-3

    def lora_without_scale(w, a, b, alpha, r):
        return oo.to_f32(w) + oo.to_f32(b) @ oo.to_f32(a)

    with monkeypatch.context() as m:
        m.setattr(oo, "merge_lora", lora_without_scale)
        assert deviation(OracleModel(inputs)) > 1e-3

    class TransposedLoRA(OracleModel):
        def __init__(self, inp):
            super().__init__(inp, "none")
            s = np.float32(inp.cfg.lora_alpha / inp.cfg.lora_r)
            for lw, fac in zip(self.layers, inp.lora):
                for name in ("wq", "wk", "wv", "wo"):  # square ones: a transposed delta fits
                    a, b = fac[name]
                    lw[name] = lw[name] + s * (oo.to_f32(b) @ oo.to_f32(a)).T

    assert deviation(TransposedLoRA(inputs)) > 1e-3

    class NoBiasOnFc1(OracleModel):
        def _proj(self, lw, name, x):
            y = super()._proj(lw, name, x)
            return y - lw["b1"] if name == "w1" else y

    assert deviation(NoBiasOnFc1(inputs)) > 1e-3

    class NoFinalLN(OracleModel):
        def logits(self, x):
            return x @ self.tok_emb.T

    assert deviation(NoFinalLN(inputs)) > 1e-3


def test_kv_cache_equals_full_recompute():
    """Incremental decode (one token per pass over the cache) == one causal pass."""
    for name in ("opt-tiny-fp32", "opt-tiny-fp32-bias"):
        cfg = WORKLOADS[name]
        inputs = make_model(cfg)
        prompts = make_prompts(cfg)
        model = OracleModel(inputs)
        ids, _, logged = model.generate(prompts, cfg.gen_len, log_steps=range(cfg.gen_len))
        seq = np.concatenate([prompts, ids[:, :-1]], axis=1)
        full = model.full_logits(seq)
        for k in range(cfg.gen_len):
            row = full[:, cfg.prompt_len - 1 + k]
            scale = np.abs(row).max()
            np.testing.assert_allclose(logged[k], row, atol=1e-5 * scale, rtol=0)


@pytest.mark.slow
def test_kv_cache_equals_full_recompute_opt125m_one_sequence():
    cfg = WORKLOADS["opt-125m"].with_(prompt_len=24, gen_len=8, batch=1)
    inputs = make_model(cfg)
    prompts = make_prompts(cfg)
    model = OracleModel(inputs)
    ids, _, logged = model.generate(prompts, cfg.gen_len, log_steps=range(cfg.gen_len))
    full = model.full_logits(np.concatenate([prompts, ids[:, :-1]], axis=1))
    for k in range(cfg.gen_len):
        row = full[:, cfg.prompt_len - 1 + k]
        np.testing.assert_allclose(logged[k], row, atol=1e-5 * np.abs(row).max(), rtol=0)


def test_lora_merged_equals_unmerged_branch():
    for name in ("opt-tiny-fp32", "opt-tiny-fp32-bias"):
        cfg = WORKLOADS[name]
        inputs = make_model(cfg)
        prompts = make_prompts(cfg)
        ids, lps_m, lg_m = OracleModel(inputs, "merged").generate(
            prompts, cfg.gen_len, log_steps=range(cfg.gen_len))
        _, lps_u, lg_u = OracleModel(inputs, "unmerged").generate(
            prompts, cfg.gen_len, force_ids=ids, log_steps=range(cfg.gen_len))
        np.testing.assert_allclose(lps_m, lps_u, atol=1e-5, rtol=0)
        for k in lg_m:
            np.testing.assert_allclose(lg_m[k], lg_u[k], atol=1e-5, rtol=0)
        # and the LoRA delta is not negligible: the base model differs
        _, _, lg_b = OracleModel(inputs, "none").generate(
            prompts, cfg.gen_len, force_ids=ids, log_steps=range(cfg.gen_len))
        assert max(np.abs(lg_m[k] - lg_b[k]).max() for k in lg_m) > 1e-4


def test_lora_zero_b_leaves_weight_bits():
    cfg = WORKLOADS["opt-125m"]
    rng = np.random.default_rng(0)
    w = rng.standard_normal((64, 48)).astype(np.float32)
    a = rng.standard_normal((8, 48)).astype(np.float32)
    b = np.zeros((64, 8), np.float32)
    out = merge_lora(w, a, b, cfg.lora_alpha, cfg.lora_r)
    assert out.tobytes() == w.tobytes()


def test_lora_delta_rank_and_scale():
    """B A has rank <= r and the update is exactly (alpha/r) times it (2 for 16/8)."""
    rng = np.random.default_rng(1)
    a = rng.standard_normal((8, 40)).astype(np.float32)
    b = rng.standard_normal((30, 8)).astype(np.float32)
    d = oo.lora_delta(a, b, 16.0, 8)
    sv = np.linalg.svd(d.astype(np.float64), compute_uv=False)
    assert sv[7] > 1e-2 * sv[0] and sv[8] < 1e-5 * sv[0]  # rank r up to fp32 rounding
    np.testing.assert_allclose(d, 2.0 * (b.astype(np.float64) @ a.astype(np.float64)),
                               rtol=1e-5, atol=1e-5)


def _torch_layer(cfg, lw):
    d = cfg.d_model
    layer = torch.nn.TransformerEncoderLayer(d, cfg.n_heads, cfg.ffn, dropout=0.0,
                                             activation="relu", layer_norm_eps=cfg.ln_eps,
                                             batch_first=True, norm_first=True,
                                             dtype=torch.float64)
    t = lambda a: torch.tensor(np.asarray(a, np.float64))
    with torch.no_grad():
        layer.self_attn.in_proj_weight.copy_(torch.cat([t(lw["wq"]), t(lw["wk"]), t(lw["wv"])]))
        layer.self_attn.in_proj_bias.copy_(torch.cat([t(lw["bq"]), t(lw["bk"]), t(lw["bv"])]))
        layer.self_attn.out_proj.weight.copy_(t(lw["wo"]))
        layer.self_attn.out_proj.bias.copy_(t(lw["bo"]))
        layer.linear1.weight.copy_(t(lw["w1"]))
        layer.linear1.bias.copy_(t(lw["b1"]))
        layer.linear2.weight.copy_(t(lw["w2"]))
        layer.linear2.bias.copy_(t(lw["b2"]))
        layer.norm1.weight.copy_(t(lw["ln1_g"]))
        layer.norm1.bias.copy_(t(lw["ln1_b"]))
        layer.norm2.weight.copy_(t(lw["ln2_g"]))
        layer.norm2.bias.copy_(t(lw["ln2_b"]))
    return layer.eval()


def test_layer_matches_torch_pre_ln_transformer_layer():
    """One oracle layer == torch's pre-LN encoder layer with a causal mask (float64)."""
    cfg = WORKLOADS["opt-tiny-fp32-bias"].with_(init_std=0.1)
    inputs = make_model(cfg)
    model = OracleModel(inputs)
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 11, cfg.d_model)).astype(np.float32)
    cache = model.new_cache(2, 11)
    ours = model.layer(1, x.copy(), cache[1], 0)
    layer = _torch_layer(cfg, model.layers[1])
    mask = torch.nn.Transformer.generate_square_subsequent_mask(11, dtype=torch.float64)
    with torch.no_grad():
        ref = layer(torch.tensor(x, dtype=torch.float64), src_mask=mask, is_causal=True).numpy()
    np.testing.assert_allclose(ours, ref, atol=2e-5, rtol=1e-5)
    # the same layer fed one token at a time over the cache gives the same rows
    cache2 = model.new_cache(2, 11)
    rows = [model.layer(1, x[:, t:t + 1].copy(), cache2[1], t) for t in range(11)]
    np.testing.assert_allclose(np.concatenate(rows, axis=1), ref, atol=2e-5, rtol=1e-5)


def test_layer_norm_matches_torch_and_constant_rows():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 96)).astype(np.float32) * 3 + 1
    g = rng.standard_normal(96).astype(np.float32)
    b = rng.standard_normal(96).astype(np.float32)
    ref = torch.nn.functional.layer_norm(torch.tensor(x, dtype=torch.float64), (96,),
                                         torch.tensor(g, dtype=torch.float64),
                                         torch.tensor(b, dtype=torch.float64), 1e-5).numpy()
    np.testing.assert_allclose(layer_norm(x, g, b, 1e-5), ref, atol=2e-5, rtol=1e-5)
    const = np.full((3, 96), 7.25, np.float32)
    assert np.array_equal(layer_norm(const, g, b, 1e-5), np.broadcast_to(b, (3, 96)))


def test_zero_layers_give_closed_form_logits():
    """All layer weights and biases zero: logits = LN_f(E[id] + P[t+2]) E^T at every step."""
    cfg = WORKLOADS["opt-tiny-fp32"]
    inputs = make_model(cfg, with_lora=False)
    for lw in inputs.layers:
        for k in lw:
            if k.startswith(("w", "b")):
                lw[k] = np.zeros_like(lw[k])
    prompts = make_prompts(cfg)
    ids, lps, logged = OracleModel(inputs).generate(prompts, 4, log_steps=range(4))
    E = torch.tensor(inputs.globals["tok_emb"], dtype=torch.float64)
    P = torch.tensor(inputs.globals["pos_emb"], dtype=torch.float64)
    for k in range(4):
        tok = prompts[:, -1] if k == 0 else ids[:, k - 1]
        pos = cfg.prompt_len - 1 + k
        x = E[torch.tensor(tok, dtype=torch.long)] + P[pos + 2]
        y = torch.nn.functional.layer_norm(x, (cfg.d_model,), eps=cfg.ln_eps)
        ref = (y @ E.T).numpy()
        np.testing.assert_allclose(logged[k], ref, atol=1e-5, rtol=0)
        assert np.array_equal(ids[:, k], ref.argmax(-1))


def test_uniform_attention_averages_values():
    """W_q = 0, b_q = 0: every score is equal, so the context is the mean of v_0..v_t."""
    cfg = WORKLOADS["opt-tiny-fp32-bias"]
    inputs = make_model(cfg, with_lora=False)
    lw0 = inputs.layers[0]
    lw0["wq"] = np.zeros_like(lw0["wq"])
    lw0["bq"] = np.zeros_like(lw0["bq"])
    d = cfg.d_model
    lw0["wo"] = np.eye(d, dtype=np.float32)
    for k in ("bo", "w1", "b1", "w2", "b2"):
        lw0[k] = np.zeros_like(lw0[k])
    model = OracleModel(inputs)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 9, d)).astype(np.float32)
    out = model.layer(0, x.copy(), model.new_cache(1, 9)[0], 0)
    X = torch.tensor(x[0], dtype=torch.float64)
    h = torch.nn.functional.layer_norm(X, (d,), torch.tensor(lw0["ln1_g"], dtype=torch.float64),
                                       torch.tensor(lw0["ln1_b"], dtype=torch.float64), cfg.ln_eps)
    v = h @ torch.tensor(lw0["wv"], dtype=torch.float64).T + torch.tensor(lw0["bv"], dtype=torch.float64)
    mean_v = torch.cumsum(v, 0) / torch.arange(1, 10, dtype=torch.float64)[:, None]
    np.testing.assert_allclose(out[0], (X + mean_v).numpy(), atol=1e-5, rtol=1e-5)


def test_greedy_lowest_index_on_exact_ties():
    lg = np.array([[0.5, 2.0, -1.0, 2.0, 2.0], [3.0, 3.0, 3.0, 3.0, 3.0]], np.float32)
    assert list(greedy(lg)) == [1, 0]


def test_logprob_identities():
    cfg = WORKLOADS["opt-tiny-fp32-bias"]
    inputs = make_model(cfg)
    prompts = make_prompts(cfg)
    ids, lps, logged = OracleModel(inputs).generate(prompts, cfg.gen_len,
                                                   log_steps=range(cfg.gen_len))
    assert (lps <= 0).all()
    for k, lg in logged.items():
        t = torch.tensor(lg, dtype=torch.float64)
        lse = torch.logsumexp(t, -1)
        np.testing.assert_allclose(lps[:, k], (t.max(-1).values - lse).numpy(), atol=1e-5)
        # greedy: log-prob of the chosen token = -log sum exp(l - l_max)
        np.testing.assert_allclose(
            lps[:, k], -np.log(np.exp((t - t.max(-1, keepdim=True).values).numpy()).sum(-1)),
            atol=1e-5)
    # a forced token that is not the argmax has a strictly smaller log-prob
    lg = np.array([[0.0, 1.0, 2.0]], np.float32)
    assert log_softmax_pick(lg, np.array([0]))[0] < log_softmax_pick(lg, np.array([2]))[0]
    assert math.isclose(float(log_softmax_pick(lg, np.array([2]))[0]),
                        2.0 - math.log(1 + math.e + math.e ** 2), abs_tol=1e-6)


# ---------------------------------------------------------------------------
# Sampling (temperature + nucleus, counter-based SplitMix64 uniforms)
# ---------------------------------------------------------------------------
def test_sampler_rng_is_published_splitmix64():
    from oracle import splitmix64_output
    # Published SplitMix64 outputs for the initial state 1234567 (outputs 1..5).
    assert [splitmix64_output(1234567, n) for n in range(1, 6)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def _draws(logits, t, top_p, n_seq=40, n_step=100, seed=99):
    from oracle import sample_token
    counts = np.zeros(len(logits))
    for b in range(n_seq):
        for k in range(n_step):
            tok, _ = sample_token(np.asarray(logits, np.float32), t, top_p, seed, b, k)
            counts[tok] += 1
    return counts / counts.sum()


def test_sampler_frequencies_follow_tempered_softmax():
    p = np.array([0.5, 0.3, 0.15, 0.05])
    freq = _draws(np.log(p), 1.0, 1.0)
    assert np.abs(freq - p).max() < 0.03, freq
    # temperature 2: probabilities proportional to p^(1/2)
    q = np.sqrt(p) / np.sqrt(p).sum()
    freq = _draws(np.log(p), 2.0, 1.0)
    assert np.abs(freq - q).max() < 0.03, freq
    # a tiny temperature is the argmax
    assert _draws(np.log(p), 1e-4, 1.0, n_seq=3, n_step=10)[0] == 1.0


def test_sampler_nucleus():
    p = np.array([0.5, 0.3, 0.15, 0.05])
    # top_p 0.7: {0, 1} (0.5 < 0.7 <= 0.8), renormalised 0.625 / 0.375
    freq = _draws(np.log(p), 1.0, 0.7)
    assert freq[2] == 0 and freq[3] == 0 and abs(freq[0] - 0.625) < 0.03, freq
    # a tie at the boundary joins the nucleus whole: 0.4 < 0.5 <= 0.7 cuts inside the tie
    freq = _draws(np.log(np.array([0.4, 0.3, 0.3])), 1.0, 0.5)
    assert (freq > 0.2).all(), freq
    # top_p at or below the largest probability keeps the argmax alone
    assert _draws(np.log(p), 1.0, 0.5, n_seq=5, n_step=20)[0] == 1.0


def test_sampler_logprob_is_tempered_log_softmax():
    from oracle import sample_token
    rng = np.random.default_rng(3)
    lg = rng.normal(size=64).astype(np.float32) * 3
    for t in (0.5, 1.0, 1.7):
        tok, lp = sample_token(lg, t, 0.9, 7, 1, 2)
        ref = torch.log_softmax(torch.from_numpy(lg).double() / t, 0)[tok].item()
        assert abs(lp - ref) < 1e-12


# ---------------------------------------------------------------------------
# FP8 (E4M3) weights: the rounding, the per-row scale, and the model that uses them
# ---------------------------------------------------------------------------
from tests.brute_force import e4m3_values, nearest_e4m3  # noqa: E402


def test_e4m3_grid_round_trips_and_has_the_format_extremes():
    vals = sorted({v for v, _ in e4m3_values()})
    assert len(vals) == 253  # 254 finite codes, +0 and -0 the same value
    assert max(vals) == 448.0 and min(vals) == -448.0
    pos = [v for v in vals if v > 0]
    assert pos[0] == 2.0 ** -9 and pos[1] == 2.0 ** -8  # subnormal spacing
    np.testing.assert_array_equal(oo.e4m3_round(np.array(vals)), np.array(vals))


def test_e4m3_round_is_the_nearest_value_ties_to_even_by_brute_force():
    table = e4m3_values()
    vals = np.array(sorted({v for v, _ in table}))
    rng = np.random.default_rng(8)
    mids = (vals[1:] + vals[:-1]) / 2  # every exact tie
    xs = np.concatenate([mids, rng.normal(0, 60, 400), rng.normal(0, 0.02, 200),
                         rng.uniform(-600, 600, 100), [448.0, 463.9, 464.0, 1e6, -1e6]])
    got = oo.e4m3_round(xs)
    want = np.array([nearest_e4m3(float(x), table) for x in xs])
    np.testing.assert_array_equal(got, want)


def test_row_quantization_scale_and_error_bound():
    rng = np.random.default_rng(3)
    w = (rng.normal(0, 0.02, (64, 300)) * rng.uniform(0.1, 10, (64, 1))).astype(np.float32)
    w[5] = 0.0
    q, s = oo.quantize_rows_e4m3(w)
    assert s.dtype == np.float32 and s[5] == 1.0 and (q[5] == 0).all()
    amax = np.abs(w).max(axis=1)
    np.testing.assert_allclose(s[amax > 0], amax[amax > 0] / 448.0, rtol=1e-7)
    assert (np.abs(q).max(axis=1)[amax > 0] == 448.0).all()  # the largest element: +-448
    wq = oo.dequantize_rows(q, s)
    # half a spacing: 2^-4 relative in the normal range, 2^-10 * s below 2^-6 * s
    bound = np.maximum(np.abs(w) * 2.0 ** -4, 2.0 ** -10 * s[:, None]) * (1 + 1e-6)
    assert (np.abs(wq - w) <= bound).all()


def test_fp8_model_matches_brute_force_with_quantized_weights():
    inputs, prompts = _bf_case(BF_CFG2)
    bf = BruteForce(inputs, fp8=True)
    ids, lps, logged = OracleModel(inputs, weights="fp8").generate(
        prompts, BF_CFG2.gen_len, log_steps=range(BF_CFG2.gen_len))
    for b in range(BF_CFG2.batch):
        bids, blps, brows = bf.generate(prompts[b], BF_CFG2.gen_len)
        assert list(ids[b]) == bids
        np.testing.assert_allclose(lps[b], blps, atol=1e-5, rtol=0)
        for k in range(BF_CFG2.gen_len):
            np.testing.assert_allclose(logged[k][b], brows[k], atol=1e-5, rtol=1e-5)
    # the quantization is visible: the exact-weight model gives other logits
    _, _, exact = OracleModel(inputs).generate(prompts, BF_CFG2.gen_len, log_steps=[0])
    assert np.abs(exact[0] - logged[0]).max() > 1e-3


def test_fp8_quantizes_after_the_lora_merge():
    """Quantizing the base weight and adding the delta afterwards (a plausible slip) is
    not what the fp8 model does."""
    inputs, _ = _bf_case(BF_CFG)
    m = OracleModel(inputs, weights="fp8")
    a, b = inputs.lora[0]["wq"]
    merged = oo.merge_lora(inputs.layers[0]["wq"], a, b, BF_CFG.lora_alpha, BF_CFG.lora_r)
    np.testing.assert_array_equal(m.layers[0]["wq"], oo.dequantize_rows(*oo.quantize_rows_e4m3(merged)))
    base_first = oo.dequantize_rows(*oo.quantize_rows_e4m3(oo.to_f32(inputs.layers[0]["wq"])))
    slip = base_first + oo.lora_delta(a, b, BF_CFG.lora_alpha, BF_CFG.lora_r)
    assert np.abs(slip - m.layers[0]["wq"]).max() > 1e-4
