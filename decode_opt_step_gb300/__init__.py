"""Python binding of libhe (include/he.h): argument marshalling only.

Every step of generation runs in libhe's CUDA kernels; this module only checks
and passes pointers, sizes and the current CUDA stream.  PyTorch provides the
device memory (the engine's workspace comes from torch's caching allocator, so
a released workspace goes back to torch) and the streams.  There is no CPU or
PyTorch fallback: if libhe.so is missing or the device is not an sm_103a GPU,
construction fails with an error.
"""
from __future__ import annotations

import ctypes
from ctypes import (CFUNCTYPE, POINTER, Structure, c_char_p, c_double, c_float, c_int, c_longlong,
                    c_size_t, c_uint, c_void_p)
from pathlib import Path

import numpy as np

_LIB_PATH = Path(__file__).resolve().parent / "libhe.so"

HE_OK, HE_ERR_ARG, HE_ERR_STATE, HE_ERR_OOM = 0, -1, -2, -3
HE_ERR_CUDA, HE_ERR_UNSUPPORTED, HE_ERR_DEVICE_CHECK = -4, -5, -6
HE_DTYPE_F32, HE_DTYPE_BF16, HE_DTYPE_F16 = 0, 1, 2
HE_WEIGHTS_F16, HE_WEIGHTS_FP8 = 0, 1
HE_ATTN_PREFILL_MMA_SYNC = 1
HE_PROJ_Q, HE_PROJ_K, HE_PROJ_V, HE_PROJ_O, HE_PROJ_FC1, HE_PROJ_FC2 = range(6)
PROJ = ("wq", "wk", "wv", "wo", "w1", "w2")
BIAS = ("bq", "bk", "bv", "bo", "b1", "b2")
KCLASS = ("gemm", "attn_decode", "norm", "head", "prefill_gemm", "prefill_attn", "other", "spare")

_STATUS_NAMES = {0: "HE_OK", -1: "HE_ERR_ARG", -2: "HE_ERR_STATE", -3: "HE_ERR_OOM",
                 -4: "HE_ERR_CUDA", -5: "HE_ERR_UNSUPPORTED", -6: "HE_ERR_DEVICE_CHECK"}


class HeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class HeConfig(Structure):
    _fields_ = [("n_layers", c_int), ("d_model", c_int), ("n_heads", c_int), ("ffn", c_int),
                ("vocab", c_int), ("max_pos", c_int), ("pos_offset", c_int), ("dtype", c_int),
                ("ln_eps", c_float), ("max_batch", c_int), ("max_seq", c_int),
                ("lora_r", c_int), ("lora_alpha", c_float), ("lora_targets", c_uint)]


class HeLayerWeights(Structure):
    _fields_ = [("w", c_void_p * 6), ("b", c_void_p * 6), ("ln1_g", c_void_p),
                ("ln1_b", c_void_p), ("ln2_g", c_void_p), ("ln2_b", c_void_p),
                ("lora_a", c_void_p * 6), ("lora_b", c_void_p * 6)]


class HeWeights(Structure):
    _fields_ = [("tok_emb", c_void_p), ("pos_emb", c_void_p), ("lnf_g", c_void_p),
                ("lnf_b", c_void_p), ("layers", POINTER(HeLayerWeights))]


ALLOC_FN = CFUNCTYPE(c_void_p, c_size_t, c_void_p, c_void_p)
FREE_FN = CFUNCTYPE(None, c_void_p, c_size_t, c_void_p, c_void_p)


class HeAllocator(Structure):
    _fields_ = [("alloc", ALLOC_FN), ("free", FREE_FN), ("ctx", c_void_p)]


class HeStats(Structure):
    _fields_ = [("fuse_ms", c_double), ("prefill_ms", c_double), ("decode_ms", c_double),
                ("unfuse_ms", c_double), ("launches", c_longlong), ("generate_calls", c_longlong),
                ("workspace_bytes", c_size_t), ("kv_bytes", c_size_t), ("restore_bytes", c_size_t),
                ("kclass_ms", c_double * 8), ("kclass_launches", c_longlong * 8)]


# Every symbol include/he.h and include/he_ops.h declare, with its ctypes signature.
_SIGNATURES = {
    "he_create": (c_int, [POINTER(HeConfig), POINTER(HeWeights), POINTER(HeAllocator), c_int,
                          POINTER(c_void_p)]),
    "he_destroy": (c_int, [c_void_p]),
    "he_fuse_lora": (c_int, [c_void_p, c_void_p]),
    "he_unfuse_lora": (c_int, [c_void_p, c_void_p]),
    "he_read_fused_weight": (c_int, [c_void_p, c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "he_generate": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "he_generate_ex": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                               c_void_p, c_void_p, c_int, c_void_p, c_void_p]),
    "he_generate_host": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                                 c_void_p]),
    "he_check": (c_int, [c_void_p, c_void_p]),
    "he_release_workspace": (c_int, [c_void_p, c_void_p]),
    "he_retake_workspace": (c_int, [c_void_p, c_void_p]),
    "he_set_profiling": (c_int, [c_void_p, c_uint]),
    "he_set_cuda_graph": (c_int, [c_void_p, c_int]),
    "he_set_sampling": (c_int, [c_void_p, ctypes.c_float, ctypes.c_float, ctypes.c_uint64]),
    "he_score": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p]),
    "he_get_stats": (c_int, [c_void_p, POINTER(HeStats)]),
    "he_last_error": (c_char_p, []),
    "he_version": (c_char_p, []),
    "he_op_linear": (c_int, [c_int, c_void_p, c_int, c_void_p, c_int, c_void_p, c_int, c_int,
                             c_int, c_int, c_void_p, c_void_p]),
    "he_op_tile_weight": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p]),
    "he_op_head_greedy": (c_int, [c_int, c_void_p, c_int, c_void_p, c_int, c_int, c_int,
                                  c_void_p, c_void_p, c_void_p, c_void_p]),
    "he_op_linear_fp8": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                 c_int, c_int, c_void_p, c_void_p]),
    "he_set_weight_format": (c_int, [c_void_p, c_int]),
    "he_op_fuse_tiled": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_float, c_void_p, c_int,
                                 c_int, c_void_p]),
    "he_read_fused_fp8": (c_int, [c_void_p, c_int, c_int, c_void_p, c_size_t, c_void_p,
                                  c_void_p]),
    "he_op_attn_prefill": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                   c_int, c_int, c_int, c_int, c_void_p, c_void_p]),
    "he_op_attn_decode": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                  c_int, c_int, c_int, c_int, c_void_p, c_void_p]),
    "he_op_attn_decode_noalloc": (c_int, [c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                          c_int, c_int, c_int, c_int, c_int, c_void_p]),
}

_lib = None


def load_library(path: str | Path | None = None):
    """Loads libhe.so (built in-tree by ``decode_opt_step_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path else _LIB_PATH
    if not p.exists():
        raise RuntimeError(f"libhe.so not found at {p}: build it with "
                           "`python -m decode_opt_step_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(str(p))
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(status: int):
    if status != HE_OK:
        raise HeError(status, _lib.he_last_error().decode())


def _stream_handle(torch, stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


class Engine:
    """One OPT-style actor on one GPU: LoRA fuse/unfuse, greedy generation, workspace.

    ``cfg`` needs: n_layers, d_model, n_heads, ffn, vocab, max_pos, pos_offset, dtype
    ("f32" | "bf16"), ln_eps, lora_r, lora_alpha.  ``weights``: dict of device tensors
    tok_emb [V][d], pos_emb [max_pos+off][d], lnf_g, lnf_b and ``layers`` (list of dicts
    with wq, wk, wv, wo [d][d], w1 [ffn][d], w2 [d][ffn], their biases bq..b2,
    ln1_g/ln1_b/ln2_g/ln2_b); optional ``lora`` (list of {proj: (A [r][in], B [out][r])}).
    The tensors must stay alive while the engine exists; fuse/unfuse write w* in place.
    ``alloc_filter(nbytes) -> bool`` (torch allocator only) can refuse allocations,
    which the engine sees as an out-of-memory allocator (used to test that path).
    """

    def __init__(self, cfg, weights: dict, max_batch: int, max_seq: int, device=None,
                 allocator: str = "torch", alloc_filter=None):
        import torch
        self._torch = torch
        lib = load_library()
        self._lib = lib
        if not torch.cuda.is_available():
            raise RuntimeError("libhe needs a CUDA device")
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index or 0)
        self.dtype = cfg.dtype
        tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
        lora = weights.get("lora") or []
        targets = 0
        if lora:
            for i, name in enumerate(PROJ):
                if all(name in lf for lf in lora):
                    targets |= 1 << i
        c = HeConfig(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.ffn, cfg.vocab, cfg.max_pos,
                     cfg.pos_offset, HE_DTYPE_BF16 if cfg.dtype == "bf16" else HE_DTYPE_F32,
                     cfg.ln_eps, max_batch, max_seq, cfg.lora_r, cfg.lora_alpha, targets)
        self.cfg, self.max_batch, self.max_seq = cfg, max_batch, max_seq
        keep = []

        def ptr(t, shape=None):
            if not isinstance(t, torch.Tensor) or t.device != self.device or t.dtype != tdt:
                raise TypeError(f"expected a {tdt} tensor on {self.device}")
            if not t.is_contiguous():
                raise ValueError("weight tensors must be contiguous")
            if shape is not None and tuple(t.shape) != tuple(shape):
                raise ValueError(f"shape {tuple(t.shape)} != {tuple(shape)}")
            keep.append(t)
            return t.data_ptr()

        d, f = cfg.d_model, cfg.ffn
        shapes = {"wq": (d, d), "wk": (d, d), "wv": (d, d), "wo": (d, d), "w1": (f, d), "w2": (d, f)}
        layers = (HeLayerWeights * cfg.n_layers)()
        for li, lw in enumerate(weights["layers"]):
            L = layers[li]
            for i, (wn, bn) in enumerate(zip(PROJ, BIAS)):
                L.w[i] = ptr(lw[wn], shapes[wn])
                L.b[i] = ptr(lw[bn], (shapes[wn][0],))
                if (targets >> i) & 1:
                    a, b = lora[li][wn]
                    L.lora_a[i] = ptr(a, (cfg.lora_r, shapes[wn][1]))
                    L.lora_b[i] = ptr(b, (shapes[wn][0], cfg.lora_r))
            L.ln1_g, L.ln1_b = ptr(lw["ln1_g"], (d,)), ptr(lw["ln1_b"], (d,))
            L.ln2_g, L.ln2_b = ptr(lw["ln2_g"], (d,)), ptr(lw["ln2_b"], (d,))
        w = HeWeights(ptr(weights["tok_emb"], (cfg.vocab, d)),
                      ptr(weights["pos_emb"], (cfg.max_pos + cfg.pos_offset, d)),
                      ptr(weights["lnf_g"], (d,)), ptr(weights["lnf_b"], (d,)), layers)
        self._keep = keep
        alloc_p = None
        if allocator == "torch":
            dev_index = self.device.index

            def _alloc(nbytes, stream, _ctx):
                if alloc_filter is not None and not alloc_filter(int(nbytes)):
                    return None  # host-side allocation failure injected by the caller
                try:
                    return torch.cuda.caching_allocator_alloc(int(nbytes), dev_index,
                                                              int(stream or 0))
                except Exception:  # out of memory -> NULL -> HE_ERR_OOM
                    return None

            def _free(p, _nbytes, _stream, _ctx):
                torch.cuda.caching_allocator_delete(int(p))

            self._cb = (ALLOC_FN(_alloc), FREE_FN(_free))
            self._allocator = HeAllocator(self._cb[0], self._cb[1], None)
            alloc_p = ctypes.byref(self._allocator)
        elif allocator != "cuda":
            raise ValueError("allocator must be 'torch' or 'cuda'")
        handle = c_void_p()
        with torch.cuda.device(self.device):
            _check(lib.he_create(ctypes.byref(c), ctypes.byref(w), alloc_p, self.device.index,
                                 ctypes.byref(handle)))
        self._h = handle

    # -- calls -------------------------------------------------------------------------
    def _s(self, stream):
        return _stream_handle(self._torch, stream)

    def fuse_lora(self, stream=None):
        _check(self._lib.he_fuse_lora(self._h, self._s(stream)))

    def unfuse_lora(self, stream=None):
        _check(self._lib.he_unfuse_lora(self._h, self._s(stream)))

    def read_fused_weight(self, layer: int, proj: int, stream=None):
        """Projection `proj` (HE_PROJ_*) of `layer` as generation reads it while fused:
        the merged fp32 weight [out][in] (fp32 engines) or the flat fp16 tiled copy
        (bf16 engines, he_op_tile_weight's element order)."""
        import torch
        c = self.cfg
        rows = c.ffn if proj == HE_PROJ_FC1 else c.d_model
        cols = c.ffn if proj == HE_PROJ_FC2 else c.d_model
        if c.dtype == "f32":
            out = torch.empty((rows, cols), dtype=torch.float32, device=self.device)
        else:
            out = torch.empty(rows * cols, dtype=torch.float16, device=self.device)
        _check(self._lib.he_read_fused_weight(self._h, layer, proj, out.data_ptr(),
                                              out.numel() * out.element_size(), self._s(stream)))
        return out

    def read_fused_fp8(self, layer: int, proj: int, stream=None):
        """With fp8 weights fused: (codes, scales) of projection `proj` of `layer`: the
        E4M3 codes as uint8 in the fp8 tiled layout (flat) and the fp32 row scales."""
        import torch
        c = self.cfg
        rows = c.ffn if proj == HE_PROJ_FC1 else c.d_model
        cols = c.ffn if proj == HE_PROJ_FC2 else c.d_model
        codes = torch.empty(rows * cols, dtype=torch.uint8, device=self.device)
        scales = torch.empty(rows, dtype=torch.float32, device=self.device)
        _check(self._lib.he_read_fused_fp8(self._h, layer, proj, codes.data_ptr(), rows * cols,
                                           scales.data_ptr(), self._s(stream)))
        return codes, scales

    def set_weight_format(self, fmt: str):
        """'f16' (default) or 'fp8': the format generation reads the projections in, from
        the next fuse (or unfused generation) on (he_set_weight_format)."""
        code = {"f16": HE_WEIGHTS_F16, "fp8": HE_WEIGHTS_FP8}[fmt]
        _check(self._lib.he_set_weight_format(self._h, code))

    def release_workspace(self, stream=None):
        _check(self._lib.he_release_workspace(self._h, self._s(stream)))

    def retake_workspace(self, stream=None):
        _check(self._lib.he_retake_workspace(self._h, self._s(stream)))

    def check(self, stream=None):
        _check(self._lib.he_check(self._h, self._s(stream)))

    def set_sampling(self, temperature: float = 0.0, top_p: float = 1.0, seed: int = 0):
        """Sampled generation (temperature > 0, nucleus top_p, counter-based seed); 0 = greedy."""
        _check(self._lib.he_set_sampling(self._h, float(temperature), float(top_p),
                                         int(seed) & ((1 << 64) - 1)))

    def set_cuda_graph(self, enable: bool = True):
        """Run he_generate / he_generate_host as a captured, cached CUDA graph."""
        _check(self._lib.he_set_cuda_graph(self._h, 1 if enable else 0))

    def set_profiling(self, classes=()):
        """Time the given kernel classes (names from KCLASS, or "all"); () turns it off."""
        if classes == "all":
            mask = 0xFF
        else:
            mask = 0
            for c in classes:
                mask |= 1 << KCLASS.index(c)
        _check(self._lib.he_set_profiling(self._h, mask))

    def _prompts(self, prompts):
        torch = self._torch
        if prompts.dtype != torch.int32 or prompts.device != self.device or prompts.dim() != 2:
            raise TypeError("prompts must be a 2-D int32 tensor on the engine's device")
        return prompts.contiguous()

    def generate(self, prompts, gen_len: int, out=None, stream=None):
        """Greedy generation: returns (ids int32 [B][gen_len], logprobs fp32 [B][gen_len])."""
        torch = self._torch
        p = self._prompts(prompts)
        B, Lp = p.shape
        if out is None:
            out = (torch.empty((B, gen_len), dtype=torch.int32, device=self.device),
                   torch.empty((B, gen_len), dtype=torch.float32, device=self.device))
        ids, lps = out
        _check(self._lib.he_generate(self._h, p.data_ptr(), B, Lp, gen_len, ids.data_ptr(),
                                     lps.data_ptr(), self._s(stream)))
        return ids, lps

    def generate_ex(self, prompts, gen_len: int, force_ids=None, log_rows=(), stream=None):
        """Teacher-forced / logit-capturing generation: returns (ids, logprobs, logits)."""
        torch = self._torch
        p = self._prompts(prompts)
        B, Lp = p.shape
        ids = torch.empty((B, gen_len), dtype=torch.int32, device=self.device)
        lps = torch.empty((B, gen_len), dtype=torch.float32, device=self.device)
        fp = 0
        if force_ids is not None:
            force_ids = force_ids.to(device=self.device, dtype=torch.int32).contiguous()
            if tuple(force_ids.shape) != (B, gen_len):
                raise ValueError("force_ids must be [B][gen_len]")
            fp = force_ids.data_ptr()
        rows = np.asarray(list(log_rows), dtype=np.int32).reshape(-1, 2)
        n = rows.shape[0]
        logits = torch.empty((max(n, 1), self.cfg.vocab), dtype=torch.float32, device=self.device)
        rows_c = np.ascontiguousarray(rows)
        _check(self._lib.he_generate_ex(self._h, p.data_ptr(), B, Lp, gen_len, ids.data_ptr(),
                                        lps.data_ptr(), fp or None,
                                        rows_c.ctypes.data if n else None, n,
                                        logits.data_ptr() if n else None, self._s(stream)))
        return ids, lps, logits[:n]

    def score(self, ids, prompt_len: int, out=None, stream=None):
        """Log-probs of ids[:, prompt_len:] given their prefixes, one forward pass over
        prompt + answer (he_score): fp32 [B][L - prompt_len]."""
        torch = self._torch
        p = self._prompts(ids)
        B, L = p.shape
        if out is None:
            out = torch.empty((B, L - prompt_len), dtype=torch.float32, device=self.device)
        _check(self._lib.he_score(self._h, p.data_ptr(), B, L, prompt_len, out.data_ptr(),
                                  self._s(stream)))
        return out

    def generate_host(self, prompts: np.ndarray, gen_len: int, stream=None):
        """Host buffers in and out (copies inside the call); synchronises the stream."""
        p = np.ascontiguousarray(prompts, dtype=np.int32)
        B, Lp = p.shape
        ids = np.empty((B, gen_len), np.int32)
        lps = np.empty((B, gen_len), np.float32)
        _check(self._lib.he_generate_host(self._h, p.ctypes.data, B, Lp, gen_len, ids.ctypes.data,
                                          lps.ctypes.data, self._s(stream)))
        return ids, lps

    def stats(self) -> dict:
        s = HeStats()
        _check(self._lib.he_get_stats(self._h, ctypes.byref(s)))
        out = {k: getattr(s, k) for k, _ in HeStats._fields_ if k not in ("kclass_ms", "kclass_launches")}
        out["kclass_ms"] = {KCLASS[i]: s.kclass_ms[i] for i in range(8)}
        out["kclass_launches"] = {KCLASS[i]: s.kclass_launches[i] for i in range(8)}
        return out

    def close(self):
        if getattr(self, "_h", None):
            self._lib.he_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _dtype_code(torch, dt):
    return {torch.float32: HE_DTYPE_F32, torch.bfloat16: HE_DTYPE_BF16,
            torch.float16: HE_DTYPE_F16}[dt]


def attn_decode(q, kc, vc, n_keys: int, split: int = 1, stream=None):
    """Decode attention through he_op_attn_decode: q [B][H*hd], kc/vc [B][H][T][hd]."""
    import torch
    lib = load_library()
    B, H, T, hd = kc.shape
    ctx = torch.empty((B, H * hd), dtype=q.dtype, device=q.device)
    part = (torch.empty(B * H * split * (hd + 2), dtype=torch.float32, device=q.device)
            if split > 1 else None)
    dt = _dtype_code(torch, q.dtype)
    _check(lib.he_op_attn_decode(dt, q.data_ptr(), kc.data_ptr(), vc.data_ptr(), ctx.data_ptr(),
                                 B, H, hd, T, n_keys, split,
                                 part.data_ptr() if part is not None else None,
                                 _stream_handle(torch, stream)))
    return ctx


def attn_prefill(q, kc, vc, Lp: int, mma_sync: bool = False, dev_flags=None, stream=None):
    """Prompt attention through he_op_attn_prefill: q [B][Lp][H*hd] (pre-scaled),
    kc/vc [B][H][T][hd] holding the prompt's keys and values at positions 0..Lp-1;
    returns ctx [B][Lp][H*hd].  ``mma_sync`` selects the mma.sync kernel."""
    import torch
    lib = load_library()
    B, H, T, hd = kc.shape
    ctx = torch.empty((B, Lp, H * hd), dtype=q.dtype, device=q.device)
    _check(lib.he_op_attn_prefill(_dtype_code(torch, q.dtype), q.data_ptr(), kc.data_ptr(),
                                  vc.data_ptr(), ctx.data_ptr(), B, Lp, H, hd, T,
                                  HE_ATTN_PREFILL_MMA_SYNC if mma_sync else 0,
                                  dev_flags.data_ptr() if dev_flags is not None else None,
                                  _stream_handle(torch, stream)))
    return ctx


def attn_decode_noalloc(q, kc, vc, n_keys: int, split: int = 1, out=None, stream=None):
    """Decode attention through he_op_attn_decode_noalloc: the split partials use the
    library's built-in scratch, so nothing is allocated for them (``out`` may be
    given to avoid the output allocation as well)."""
    import torch
    lib = load_library()
    B, H, T, hd = kc.shape
    ctx = out if out is not None else torch.empty((B, H * hd), dtype=q.dtype, device=q.device)
    _check(lib.he_op_attn_decode_noalloc(_dtype_code(torch, q.dtype), q.data_ptr(), kc.data_ptr(),
                                         vc.data_ptr(), ctx.data_ptr(), B, H, hd, T, n_keys,
                                         split, _stream_handle(torch, stream)))
    return ctx


def fuse_tiled(w, lora_a=None, lora_b=None, scale: float = 0.0, stream=None):
    """he_op_fuse_tiled: W + scale * B A as fp16 in the tiled layout (flat), bf16 inputs."""
    import torch
    lib = load_library()
    N, K = w.shape
    r = 0 if lora_a is None else lora_a.shape[0]
    out = torch.empty(N * K, dtype=torch.float16, device=w.device)
    _check(lib.he_op_fuse_tiled(w.data_ptr(), lora_a.data_ptr() if r else None,
                                lora_b.data_ptr() if r else None, r, float(scale),
                                out.data_ptr(), N, K, _stream_handle(torch, stream)))
    return out


def tile_weight(w, stream=None):
    """The tiled streaming layout of a 16-bit [N][K] weight (he_op_tile_weight), flat."""
    import torch
    lib = load_library()
    if w.dtype not in (torch.bfloat16, torch.float16) or not w.is_contiguous():
        raise TypeError("w must be a contiguous bf16 or fp16 tensor")
    out = torch.empty(w.numel(), dtype=w.dtype, device=w.device)
    _check(lib.he_op_tile_weight(w.data_ptr(), out.data_ptr(), w.shape[0], w.shape[1],
                                 _stream_handle(torch, stream)))
    return out


def head_greedy(x, w, stream=None):
    """Greedy choice and its log-prob for each row of the logits x w^T (he_op_head_greedy:
    the choice is fused into the LM-head GEMM; the logits are never stored)."""
    import torch
    lib = load_library()
    M, K = x.shape
    N = w.shape[0]
    if x.dtype != w.dtype or x.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("x and w must both be bf16 or both fp16")
    if x.stride(1) != 1 or not w.is_contiguous():
        raise ValueError("x rows and w must be dense")
    R = 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128 if M <= 128 else 256
    T = (N + 127) // 128
    scratch = torch.empty(16 * M * T * 128 + (R * K + 1) // 2 + 8 + T + 4 + 4 * T * M,
                          dtype=torch.float32, device=x.device)
    ids = torch.empty(M, dtype=torch.int32, device=x.device)
    lp = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(lib.he_op_head_greedy(_dtype_code(torch, x.dtype), x.data_ptr(), x.stride(0),
                                 w.data_ptr(), M, N, K, ids.data_ptr(), lp.data_ptr(),
                                 scratch.data_ptr(), _stream_handle(torch, stream)))
    return ids, lp


def linear_fp8(x, w8_tiled, scale, N: int, K: int, split: int = 0, stream=None):
    """y = (x codes^T) * scale[n] in fp32 (he_op_linear_fp8): x fp16 [M][K], w8_tiled the
    E4M3 codes (one byte each, uint8) in the fp8 tiled layout, scale fp32 [N]."""
    import torch
    lib = load_library()
    M = x.shape[0]
    if x.dtype != torch.float16 or x.stride(1) != 1 or x.shape[1] != K:
        raise TypeError("x must be fp16 [M][K] with dense rows")
    R = 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128
    y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    scratch = torch.empty(16 * M * N + (R * K + 1) // 2 + 8 + N // 128, dtype=torch.float32,
                          device=x.device)
    _check(lib.he_op_linear_fp8(x.data_ptr(), x.stride(0), w8_tiled.data_ptr(), scale.data_ptr(),
                                y.data_ptr(), M, N, K, split, scratch.data_ptr(),
                                _stream_handle(torch, stream)))
    return y


def linear(x, w, split: int = 1, stream=None, w_tiled=None):
    """y = x w^T in fp32 through libhe's GEMM kernels (he_op_linear).  With ``w_tiled``
    (the output of tile_weight(w)) the GEMM reads the tiled layout instead of w.
    split >= 1: split-K; split == 0: stream-K on the default CTA count; split < 0:
    stream-K on -split CTAs."""
    import torch
    lib = load_library()
    M, K = x.shape
    N = w.shape[0]
    if x.dtype != w.dtype or x.dtype not in (torch.bfloat16, torch.float16, torch.float32):
        raise TypeError("x and w must have the same type: bf16, fp16 or fp32")
    if x.stride(1) != 1 or not w.is_contiguous():
        raise ValueError("x rows and w must be dense")
    y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if split <= 0:  # stream-K: up to 16 slices per tile, row-tiled x, tile counters
        R = 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128 if M <= 128 else 256
        Np = (N + 127) // 128 * 128
        scratch = torch.empty(16 * M * Np + (R * K + 1) // 2 + 4 + Np // 128,
                              dtype=torch.float32, device=x.device)
    else:
        scratch = (torch.empty((split, M, N), dtype=torch.float32, device=x.device)
                   if split > 1 else None)
    dt = _dtype_code(torch, x.dtype)
    wp, layout = (w.data_ptr(), 0) if w_tiled is None else (w_tiled.data_ptr(), 1)
    _check(lib.he_op_linear(dt, x.data_ptr(), x.stride(0), wp, layout, y.data_ptr(), M, N, K,
                            split, scratch.data_ptr() if scratch is not None else None,
                            _stream_handle(torch, stream)))
    return y
