"""Benchmark: OPT-style experience generation through libhe on synthetic inputs.

One step = the whole generation path on one batch: LoRA fuse, prefill of the
prompts, token-by-token greedy decode over the KV cache, LoRA unfuse, workspace
release and retake.  Default workload: OPT-13B shape, batch 128, 256-token
prompts, 256 generated tokens, bf16 weights (random N(0, 0.02) init, synthetic
prompts).  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   (the CPU oracle, timed on the host cores)

With --gpus N > 1 (launched by torchrun) every rank runs an independent replica of
the workload on its own GPU (the path has no cross-sequence exchange); the value
is the tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth.workloads import WORKLOADS, make_model, make_prompts  # noqa: E402

METRIC = "OPT-13B generated tokens/s (B=128, 256+256); decode HBM GB/s vs peak"
NOMINAL_HBM_GBS = 8000.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# Algorithmic byte and flop counts of the path (no caches, activations ignored)
# ---------------------------------------------------------------------------
def layer_weight_bytes(cfg, elem=2):
    d, f = cfg.d_model, cfg.ffn
    return (4 * d * d + 2 * d * f) * elem


def decode_step_bytes(cfg, k, B, Lp, elem=2, welem=None):
    """Bytes one decode step (token k >= 1 at position Lp + k - 1) must move.  welem:
    bytes per projection weight (1 with fp8 weights, plus a 4-byte scale per row; the
    tied LM head stays 16-bit), default elem."""
    n_keys = Lp + k
    w = cfg.n_layers * proj_weight_bytes(cfg, elem if welem is None else welem) \
        + cfg.vocab * cfg.d_model * elem
    kv_read = cfg.n_layers * 2 * B * n_keys * cfg.d_model * elem
    kv_write = cfg.n_layers * 2 * B * cfg.d_model * elem
    return w + kv_read + kv_write, w, kv_read + kv_write


def attn_decode_bytes(cfg, k, B, Lp, elem=2):
    """Bytes of one decode-attention launch (one layer): K and V rows 0..Lp+k-1."""
    return 2 * B * (Lp + k) * cfg.d_model * elem


def proj_weight_bytes(cfg, welem):
    """One layer's six projections as generation streams them (fp8: codes + row scales)."""
    if welem == 1:
        return layer_weight_bytes(cfg, 1) + (5 * cfg.d_model + cfg.ffn) * 4
    return layer_weight_bytes(cfg, welem)


def decode_gemm_bytes_per_layer(cfg, elem=2, welem=None):
    return proj_weight_bytes(cfg, elem if welem is None else welem)


def prefill_flops(cfg, B, Lp):
    d, f, L = cfg.d_model, cfg.ffn, cfg.n_layers
    tok = B * Lp
    proj = 2 * tok * (4 * d * d + 2 * d * f) * L
    attn = 2 * 2 * B * cfg.n_heads * (Lp * (Lp + 1) // 2) * cfg.head_dim * L
    head = 2 * B * d * cfg.vocab
    return proj + attn + head, proj


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# The CPU oracle as the baseline (bounded sample)
# ---------------------------------------------------------------------------
def oracle_model(inputs):
    from oracle import OracleModel
    return OracleModel(inputs)


def oracle_sample(cfg, model, prompts, decode_steps=2):
    """Times the CPU oracle on sequence 0: its prefill plus `decode_steps` decode
    steps, and scales to the rate of one full sequence (prefill + gen_len - 1 steps)."""
    p = np.asarray(prompts[:1], dtype=np.int64)
    Lp = p.shape[1]
    cache = model.new_cache(1, Lp + decode_steps + 1)
    t0 = time.perf_counter()
    x = model.forward(p, cache, 0)[:, -1:]
    tok = model.logits(x[:, 0]).argmax(-1)
    t1 = time.perf_counter()
    for k in range(1, decode_steps + 1):
        x = model.forward(tok[:, None].astype(np.int64), cache, Lp + k - 1)
        tok = model.logits(x[:, 0]).argmax(-1)
    t2 = time.perf_counter()
    t_prefill, t_step = t1 - t0, (t2 - t1) / decode_steps
    t_seq = t_prefill + (cfg.gen_len - 1) * t_step
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": cfg.gen_len / t_seq, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": (f"sequence 0 of {cfg.batch}: prefill of its {Lp}-token prompt "
                       f"({t_prefill:.2f} s) + {decode_steps} decode steps "
                       f"({t_step:.2f} s each), scaled to {cfg.gen_len} generated tokens; "
                       "fp32 numpy with its BLAS on all host cores"),
            "measured_s": t2 - t0}


# ---------------------------------------------------------------------------
def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    model = oracle_model(make_model(cfg))
    prompts = make_prompts(cfg)
    times = []
    res = None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        res = oracle_sample(cfg, model, prompts, decode_steps=1)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    value = res["value"]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * statistics.mean(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(cfg),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": res["cores"],
                             "kind": "oracle", "sample": res["sample"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def reduce_max(value: float, dist, device=None) -> float:
    """Max of a per-rank float over all ranks (plain value without a process group)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


L2_BYTES = 129 * 2 ** 20  # GB300 L2


def working_set_bytes(cfg):
    """Parameters plus the KV cache of one full generation (what a step streams)."""
    elem = 4 if cfg.dtype == "f32" else 2
    params = (cfg.n_layers * (layer_weight_bytes(cfg, elem)
                              + (4 * cfg.d_model + 2 * cfg.ffn + 4 * cfg.d_model) * elem)
              + (cfg.vocab + cfg.max_pos + cfg.pos_offset) * cfg.d_model * elem)
    kv = 2 * cfg.n_layers * cfg.batch * (cfg.prompt_len + cfg.gen_len) * cfg.d_model * elem
    return params + kv


def flushes_l2(cfg) -> bool:
    """Whether a step writes an L2-sized buffer first (working sets below 2x L2)."""
    return working_set_bytes(cfg) < 2 * L2_BYTES


def compute_dtype(cfg) -> str:
    return "f32" if cfg.dtype == "f32" else "f16"


def workload_config(cfg):
    ws = working_set_bytes(cfg)
    if cfg.dtype == "f32":
        precision = "fp32 weights, activations, KV cache and arithmetic (CUDA cores)"
    else:
        precision = ("bf16 model weights; generation reads them as fp16 (merged with LoRA "
                     "while fused), with fp16 activations and KV cache and fp32 accumulation; "
                     "LayerNorm, softmax, logits and log-probs fp32; the tied LM head reads "
                     "the bf16 embedding")
    l2 = (f"working set {ws / 1e9:.2f} GB, larger than L2: weights and KV cache stream from "
          "HBM every step" if not flushes_l2(cfg) else
          f"working set {ws / 1e6:.1f} MB fits in L2: every step first writes a 256 MiB "
          "buffer to flush L2")
    return {"workload": f"{cfg.name} greedy generation",
            "layers": cfg.n_layers, "d_model": cfg.d_model, "heads": cfg.n_heads,
            "ffn": cfg.ffn, "vocab": cfg.vocab, "batch": cfg.batch,
            "prompt_len": cfg.prompt_len, "gen_len": cfg.gen_len,
            "lora": f"r={cfg.lora_r} alpha={int(cfg.lora_alpha)} on q,k,v,out,fc1,fc2",
            "step": "fuse + prefill + decode + unfuse + release/retake workspace",
            "l2": l2, "precision": precision}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="he", choices=["he", "reference"])
    ap.add_argument("--workload", default="opt-13b", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-score", action="store_true")
    ap.add_argument("--sampling", default=None, metavar="T,TOP_P,SEED",
                    help="sampled instead of greedy generation, e.g. 0.7,0.9,1234")
    ap.add_argument("--weights", default="f16", choices=["f16", "fp8"],
                    help="projection weight format during generation (fp8: E4M3 codes with "
                         "per-row scales, decoded to fp16 on the chip)")
    ap.add_argument("--no-cuda-graph", dest="cuda_graph", action="store_false",
                    help="launch every kernel directly instead of replaying the captured "
                         "CUDA graph of the generation (enable_cuda_graph)")
    args = ap.parse_args()
    cfg = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, cfg)

    import torch
    import decode_opt_step_gb300 as he
    from synth.torch_io import model_to_device

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    hbm_peak, _tf, _tfs, peak_kind = _peaks()
    inputs = make_model(cfg)
    prompts_np = make_prompts(cfg)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        model = oracle_model(inputs)
        cpu = oracle_sample(cfg, model, prompts_np)
        del model
    w = model_to_device(inputs, dev, torch)
    del inputs
    B, Lp, Lgen = cfg.batch, cfg.prompt_len, cfg.gen_len
    eng = he.Engine(cfg, w, max_batch=B, max_seq=Lp + Lgen)
    if args.weights != "f16":
        eng.set_weight_format(args.weights)
    if args.cuda_graph:
        eng.set_cuda_graph(True)
    if args.sampling:
        t_s, p_s, seed_s = args.sampling.split(",")
        eng.set_sampling(float(t_s), float(p_s), int(seed_s))
    prompts = torch.from_numpy(prompts_np).to(dev)
    ids = torch.empty((B, Lgen), dtype=torch.int32, device=dev)
    lps = torch.empty((B, Lgen), dtype=torch.float32, device=dev)

    flush = (torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
             if flushes_l2(cfg) else None)

    def step():
        if flush is not None:
            flush.fill_(1)
        eng.fuse_lora()
        eng.generate(prompts, Lgen, out=(ids, lps))
        eng.unfuse_lora()
        eng.release_workspace()
        eng.retake_workspace()

    for _ in range(args.warmup):
        step()
    eng.check()
    # ---- timed region (device-side inputs), no per-kernel events ----
    l0 = eng.stats()["launches"]
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    phase = {"prefill_ms": 0.0, "decode_ms": 0.0, "fuse_ms": 0.0, "unfuse_ms": 0.0}
    start.record()
    for _ in range(args.steps):
        step()
        st = eng.stats()  # phase events of this step (waits for the step to finish)
        for k in phase:
            phase[k] += st[k]
    end.record()
    barrier()
    clk = clocks.stop()
    wall_ms = start.elapsed_time(end)
    launches = eng.stats()["launches"] - l0
    wall_ms = reduce_max(wall_ms, dist, dev)
    ms_per_step = wall_ms / args.steps
    tokens = B * Lgen * world
    value = tokens / (ms_per_step / 1000.0)

    # ---- roofline pass: the same steps again with events around each launch of the
    # two dominant kernel classes (events between kernels cost the overlap of
    # programmatic dependent launch, so this pass is not the headline time) ----
    eng.set_profiling(["attn_decode", "gemm"])
    kls = {"attn_decode": 0.0, "gemm": 0.0}
    kln = {"attn_decode": 0, "gemm": 0}
    for _ in range(args.steps):
        step()
        st = eng.stats()
        for k in kls:
            kls[k] += st["kclass_ms"][k]
            kln[k] += st["kclass_launches"][k]
    eng.set_profiling(())

    # ---- scoring: log-probs of the generated answers in one pass (he_score) ----
    score = None
    if not args.no_score:
        eng.fuse_lora()
        eng.generate(prompts, Lgen, out=(ids, lps))
        full = torch.cat([prompts, ids], dim=1).contiguous()
        sc = torch.empty((B, Lgen), dtype=torch.float32, device=dev)
        eng.score(full, Lp, out=sc)  # warm-up
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 2
        s0.record()
        for _ in range(reps):
            eng.score(full, Lp, out=sc)
        s1.record()
        torch.cuda.synchronize()
        sc_ms = s0.elapsed_time(s1) / reps
        lp_gap = (sc - lps).abs().max().item()
        eng.unfuse_lora()
        f_tok = B * (Lp + Lgen - 1)
        score = {"ms": sc_ms, "tokens_per_s": B * Lgen / (sc_ms / 1000.0),
                 "tflops": (prefill_flops(cfg, B, Lp + Lgen - 1)[0]
                            + 2 * B * (Lgen - 1) * cfg.d_model * cfg.vocab) / (sc_ms / 1000.0) / 1e12,
                 "tokens_in_pass": f_tok, "max_abs_vs_decode_logprobs": lp_gap}

    # ---- end to end through the host-buffer entry point ----
    e2e = None
    if not args.no_e2e:
        hp = torch.from_numpy(prompts_np).pin_memory().numpy()  # pinned host prompts
        barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            if flush is not None:
                flush.fill_(1)
            eng.fuse_lora()
            eng.generate_host(hp, Lgen)  # H2D prompts, generate, D2H ids + log-probs, sync
            eng.unfuse_lora()
            eng.release_workspace()
            eng.retake_workspace()
        barrier()
        e2e_s = reduce_max((time.perf_counter() - t0) / args.steps, dist, dev)
        e2e = {"value": tokens / e2e_s, "unit": "tokens/s",
               "h2d_bytes_per_step": B * Lp * 4, "d2h_bytes_per_step": B * Lgen * 8}

    # ---- roofline of the dominant kernel and the decode phase ----
    steps = args.steps
    welem = 1 if args.weights == "fp8" else 2
    attn_bytes = sum(attn_decode_bytes(cfg, k, B, Lp) for k in range(1, Lgen)) * cfg.n_layers
    gemm_bytes = decode_gemm_bytes_per_layer(cfg, welem=welem) * cfg.n_layers * (Lgen - 1)
    per_kernel = {}
    for name, byts in (("attn_decode", attn_bytes), ("gemm", gemm_bytes)):
        ms = kls[name] / steps
        n = kln[name] / steps
        ach = byts / (ms / 1000.0) / 1e9 if ms > 0 else None
        per_kernel[name] = {"ms_per_step": ms, "launches_per_step": n,
                            "bytes_per_launch": byts / n if n else None, "gbs": ach}
    dom = max(per_kernel, key=lambda k: per_kernel[k]["ms_per_step"])
    pk = per_kernel[dom]
    # DRAM bytes (read + write) per launch, scaled from one ncu capture of the kernel
    # (summaries under profiles/) by the ratio of measured to algorithmic bytes of the
    # captured launch: k_attn_decode at B=128, 40 heads, 384 keys (the average decode
    # launch here) and k_gemm_sk on the fc1 shape as the engine launches it (a decode
    # step of the two-layer OPT-13B-shape workload).  Set to None when the kernel changes.
    traffic_ratio = {"attn_decode": (1.007984e9 + 4.334592e6) / 1.00663296e9,
                     "gemm": (211.179264e6 + 6.607872e6) / 209.7152e6}
    if args.weights != "f16":
        traffic_ratio.pop("gemm")  # captured on the 16-bit kernel only
    traffic = (pk["bytes_per_launch"] * traffic_ratio[dom]
               if pk["bytes_per_launch"] and dom in traffic_ratio else None)
    roofline = {"bound": "hbm",
                "kernel": "k_attn_decode" if dom == "attn_decode" else "k_gemm_sk (decode projections)",
                "achieved": pk["gbs"], "peak": hbm_peak, "unit": "GB/s",
                "frac": pk["gbs"] / hbm_peak if pk["gbs"] else None, "traffic": traffic,
                "peak_kind": f"{peak_kind} HBM copy bandwidth",
                "timing": ("CUDA events around every launch of the kernel class on the engine's "
                           "stream, over a second pass of the timed steps")}
    dec_total = sum(decode_step_bytes(cfg, k, B, Lp, welem=welem)[0] for k in range(1, Lgen))
    dec_ms = phase["decode_ms"] / steps
    dec_gbs = dec_total / (dec_ms / 1000.0) / 1e9
    pf_flops, _ = prefill_flops(cfg, B, Lp)
    pf_ms = phase["prefill_ms"] / steps
    metric = METRIC if cfg.name == "opt-13b" else f"{cfg.name} generated tokens/s (B={B}, {Lp}+{Lgen})"
    if args.weights != "f16":
        metric += f" [{args.weights} projection weights]"
    line = {"metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": compute_dtype(cfg),
            "data": "synthetic (N(0,0.02) weights and LoRA factors, uniform prompt ids)",
            "config": {**workload_config(cfg), "weights": (
                           "fp16 projections (bf16 weights merged with LoRA)" if args.weights == "f16"
                           else "fp8 E4M3 projections, one fp32 scale per output row, decoded to "
                                "fp16 on the chip; the tied LM head bf16"),
                       "launch": ("one CUDA graph per generation" if args.cuda_graph
                                  else "direct launches, programmatic dependent launch"),
                       "decoding": (f"sampled (temperature, top_p, seed = {args.sampling})"
                                    if args.sampling else "greedy")},
            "clocks": clk, "gpu_launches": launches,
            "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu,
            "decode": {"ms": dec_ms, "bytes_per_step_avg": dec_total / (Lgen - 1),
                       "gbs": dec_gbs, "frac_of_measured_hbm": dec_gbs / hbm_peak,
                       "frac_of_8tbs": dec_gbs / NOMINAL_HBM_GBS,
                       "tokens_per_s": B * (Lgen - 1) / (dec_ms / 1000.0)},
            "prefill": {"ms": pf_ms, "tflops": pf_flops / (pf_ms / 1000.0) / 1e12},
            "fuse_ms": phase["fuse_ms"] / steps, "unfuse_ms": phase["unfuse_ms"] / steps,
            "score": score,
            "kernels": per_kernel}
    if rank == 0:
        if cpu is not None:
            cpu = {k: v for k, v in cpu.items() if k != "measured_s"}
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    eng.close()
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
