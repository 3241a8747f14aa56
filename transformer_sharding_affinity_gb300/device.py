"""Moving seeded host inputs onto the device for the C-ABI calls.

Plumbing only: PyTorch provides device memory; the values are the
generator's bf16 bit patterns (or fp32 values), copied unchanged.
"""
from __future__ import annotations

from typing import Dict

import numpy as np

UP_KEYS = ("a", "x", "Wo", "gamma", "Wg", "Wu", "Wd")
DOWN_KEYS = ("x", "gamma", "Wg", "Wu", "Wd", "gamma_next", "Wq_next", "Wk_next", "Wv_next")
ALL_KEYS = UP_KEYS + DOWN_KEYS[5:]


def host_tensor(layer: Dict[str, np.ndarray], key: str, dtype: str):
    import torch
    if dtype == "bf16":
        bits = layer[key + "_bits"]
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(layer[key], dtype=np.float32))


def to_device(layer: Dict[str, np.ndarray], dtype: str, keys=UP_KEYS, device="cuda"):
    return {k: host_tensor(layer, k, dtype).to(device) for k in keys if k in layer or k + "_bits" in layer}
