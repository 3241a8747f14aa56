"""One-call helpers over the C ABI for PyTorch users.

``s_up`` and ``s_down`` take one layer's CUDA tensors (bf16 or fp32, PyTorch
``nn.Linear`` storage), allocate the workspace and the output, enqueue the
pass on the current stream, check the device status and return S.  They only
marshal arguments; every number comes from ``libaffinity``.
"""
from __future__ import annotations

from . import binding as B


def _dims(x, HD: int, I: int, H: int, G: int, eps: float):
    import torch
    T, D = x.shape
    if HD % H:
        raise ValueError("H*d_head must be a multiple of H")
    if x.dtype == torch.bfloat16:
        dtype = B.AFF_BF16
    elif x.dtype == torch.float32:
        dtype = B.AFF_FP32
    else:
        raise TypeError("tensors must be bfloat16 or float32")
    return B.dims(T, D, H, G, HD // H, I, eps, dtype)


def s_up(a, x, Wo, gamma, Wg, Wu, Wd, H: int, G: int, mode: str = "fo", eps: float = 1e-6,
         per_head: bool = False, stream=None):
    """S_up [G, I] (and S_head [H, I] with per_head=True) for mode "fo", "add" or "loo"."""
    import torch
    if a.shape != (x.shape[0], Wo.shape[1]):
        raise ValueError("a must be [T, H*d_head] and Wo [D, H*d_head]")
    d = _dims(x, Wo.shape[1], Wg.shape[0], H, G, eps)
    m = B.MODES[mode]
    ws = torch.empty(B.workspace_size(d, m), dtype=torch.uint8, device=x.device)
    S = torch.empty(G, Wg.shape[0], device=x.device)
    Sh = torch.empty(H, Wg.shape[0], device=x.device) if per_head else None
    B.affinity_up(a, x, Wo, gamma, Wg, Wu, Wd, d, m, S, Sh, ws, stream=stream)
    st = B.device_status(ws, stream)
    if st != B.AFF_OK:
        raise B.AffinityError(st, "affinity_up", B.strerror(st))
    return (S, Sh) if per_head else S


def s_down(x, gamma, Wg, Wu, Wd, gamma_next, Wq_next, Wk_next, Wv_next, H: int, G: int, eps: float = 1e-6,
           stream=None):
    """S_down [I, G]: how much each KV group of the next layer depends on each neuron."""
    import torch
    d = _dims(x, Wq_next.shape[0], Wg.shape[0], H, G, eps)
    ws = torch.empty(B.workspace_size(d, 0, down=True), dtype=torch.uint8, device=x.device)
    S = torch.empty(Wg.shape[0], G, device=x.device)
    B.affinity_down(x, gamma, Wg, Wu, Wd, gamma_next, Wq_next, Wk_next, Wv_next, d, S, ws, stream=stream)
    st = B.device_status(ws, stream)
    if st != B.AFF_OK:
        raise B.AffinityError(st, "affinity_down", B.strerror(st))
    return S
