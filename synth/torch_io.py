"""Moves synthetic model inputs (numpy, bf16 as raw uint16) onto a torch device."""
from __future__ import annotations

import numpy as np


def to_device(arr: np.ndarray, device, torch):
    if arr.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16))
        return t.to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


def model_to_device(inputs, device, torch, free_host: bool = False) -> dict:
    """{tok_emb, pos_emb, lnf_g, lnf_b, layers: [...], lora: [...]} of device tensors."""
    out = {k: to_device(v, device, torch) for k, v in inputs.globals.items()}
    out["layers"] = []
    for li, lw in enumerate(inputs.layers):
        out["layers"].append({k: to_device(v, device, torch) for k, v in lw.items()})
        if free_host:
            inputs.layers[li] = None
    out["lora"] = [{k: (to_device(a, device, torch), to_device(b, device, torch))
                    for k, (a, b) in lf.items()} for lf in inputs.lora]
    return out
