"""Calibration and head placement for a stack of N layers.

For each layer i the GPU pass computes S_up_i [G, I] (FO or ADD) and, for
every layer but the last, S_down_i [I, G] toward layer i+1's KV groups.  The
host helpers of the library then normalise every matrix to unit mass, take
the contiguous neuron maps, choose each layer's KV-group map by scoring every
balanced partition, and evaluate the total co-located affinity J for the
contiguous and the chosen layouts ("Affinity-Aware Sharding for Delayed Tensor
Parallelism", §3 "Objective", equation (6), and "Optimiser").

This module only sequences library calls; every number comes from
``libaffinity``.
"""
from __future__ import annotations

import dataclasses
import os
from typing import Callable, Dict, List, Optional

import numpy as np

from . import binding as B


@dataclasses.dataclass
class StackResult:
    S_up: List[np.ndarray]        # N x [G, I] fp32
    S_down: List[np.ndarray]      # N-1 x [I, G] fp32
    Shat_up: List[np.ndarray]     # unit-mass fp64
    Shat_down: List[np.ndarray]
    nu: np.ndarray                # [N, I] neuron -> device
    h_contiguous: np.ndarray      # [N, G]
    h_best: np.ndarray            # [N, G]
    J_contiguous: float
    J_best: float


def contiguous_map(n: int, L: int) -> np.ndarray:
    """Item j -> device j // (n / L) (the unpermuted Megatron layout)."""
    if n % L:
        raise ValueError("n must be a multiple of L")
    return (np.arange(n) // (n // L)).astype(np.int32)


def calibrate_stack(layer_inputs: Callable[[int], Dict[str, object]], n_layers: int, d: "B.aff_dims",
                    mode: int = B.AFF_MODE_FO, stream=None, checkpoint_dir: Optional[str] = None) -> tuple:
    """Run S_up for layers 0..N-1 and S_down for layers 0..N-2 on the GPU.

    ``layer_inputs(i)`` returns layer i's device tensors under the names of
    ``affinity_up`` / ``affinity_down`` (a, x, Wo, gamma, Wg, Wu, Wd and, for
    i < N-1, gamma_next, Wq_next, Wk_next, Wv_next: layer i+1's attention
    pre-norm gain and q/k/v projections).  Returns (S_up list, S_down list) on
    the host.

    With ``checkpoint_dir`` every finished layer is saved as
    ``layer_<i>.npz`` (written to a temporary name, then renamed), and a
    layer whose file is already there is loaded instead of recomputed, so an
    interrupted run resumes where it stopped."""
    G, I = int(d.G), int(d.I)
    state = {}

    def buffers():
        if not state:
            import torch
            ws_bytes = max(B.workspace_size(d, mode), B.workspace_size(d, mode, down=True))
            state["ws"] = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
            state["up"] = torch.empty(G, I, device="cuda")
            state["dn"] = torch.empty(I, G, device="cuda")
        return state["ws"], state["up"], state["dn"]

    S_up, S_down = [], []
    for i in range(n_layers):
        last = i + 1 == n_layers
        path = None if checkpoint_dir is None else os.path.join(checkpoint_dir, f"layer_{i:03d}.npz")
        if path is not None and os.path.exists(path):
            with np.load(path) as f:
                if f["S_up"].shape == (G, I) and (last or f["S_down"].shape == (I, G)):
                    S_up.append(f["S_up"].copy())
                    if not last:
                        S_down.append(f["S_down"].copy())
                    continue
        ws, up_dev, dn_dev = buffers()
        t = layer_inputs(i)
        B.affinity_up(t["a"], t["x"], t["Wo"], t["gamma"], t["Wg"], t["Wu"], t["Wd"], d, mode, up_dev, None, ws,
                      stream=stream)
        _status(ws, stream, f"layer {i} S_up")
        S_up.append(up_dev.cpu().numpy().copy())
        if not last:
            B.affinity_down(t["x"], t["gamma"], t["Wg"], t["Wu"], t["Wd"], t["gamma_next"], t["Wq_next"],
                            t["Wk_next"], t["Wv_next"], d, dn_dev, ws, stream=stream)
            _status(ws, stream, f"layer {i} S_down")
            S_down.append(dn_dev.cpu().numpy().copy())
        if path is not None:
            os.makedirs(checkpoint_dir, exist_ok=True)
            tmp = path + ".tmp.npz"
            arrays = {"S_up": S_up[-1]} if last else {"S_up": S_up[-1], "S_down": S_down[-1]}
            np.savez(tmp, **arrays)
            os.replace(tmp, path)
    return S_up, S_down


def _status(ws, stream, where: str) -> None:
    st = B.device_status(ws, stream)
    if st != B.AFF_OK:
        raise B.AffinityError(st, where, B.strerror(st))


def place_heads(S_up: List[np.ndarray], S_down: List[np.ndarray], L: int,
                nu: Optional[np.ndarray] = None) -> StackResult:
    """Unit-mass normalisation, contiguous neuron maps (unless given), the best
    KV-group map of every layer and J for the contiguous and chosen layouts."""
    N = len(S_up)
    if len(S_down) != N - 1:
        raise ValueError("need one S_down per layer but the last")
    G, I = S_up[0].shape
    Shat_up = [B.unit_mass(s) for s in S_up]
    Shat_down = [B.unit_mass(s) for s in S_down]
    if nu is None:
        nu = np.stack([contiguous_map(I, L)] * N)
    h_contig = np.stack([contiguous_map(G, L)] * N)
    J_contig = B.objective(Shat_up, Shat_down, h_contig, nu)
    h_best, J_best = B.best_heads(Shat_up, Shat_down, nu, L)
    return StackResult(S_up, S_down, Shat_up, Shat_down, np.asarray(nu, np.int32), h_contig, h_best, J_contig,
                       J_best)


@dataclasses.dataclass
class LayoutResult:
    h: np.ndarray        # [N, G]
    nu: np.ndarray       # [N, I]
    J: float
    sweeps: int


def optimise(Shat_up: List[np.ndarray], Shat_down: List[np.ndarray], L: int, h0: Optional[np.ndarray] = None,
             nu0: Optional[np.ndarray] = None, stream=None, **opts) -> LayoutResult:
    """Alternate the neuron step (GPU) and the head step (host) from the given
    maps -- contiguous by default -- until J stops increasing
    (``affinity_optimise_layout``).  Keyword options: max_sweeps,
    freeze_heads, freeze_neurons, minimise, layer_mask, assign."""
    import torch

    N = len(Shat_up)
    G, I = np.asarray(Shat_up[0]).shape
    if h0 is None:
        h0 = np.stack([contiguous_map(G, L)] * N)
    if nu0 is None:
        nu0 = np.stack([contiguous_map(I, L)] * N)
    ws = torch.empty(B.layout_workspace_size(N, G, I, L), dtype=torch.uint8, device="cuda")
    h, nu, J, sweeps = B.optimise_layout(Shat_up, Shat_down, L, h0, nu0, ws, stream=stream, **opts)
    return LayoutResult(h, nu, J, sweeps)


def realise_layout(w: Dict[str, object], h, nu, H: int, G: int, d_head: int, L: int, stream=None):
    """Permuted copies of one layer's weights for a balanced layout (device
    tensors, nn.Linear storage): Wq/Wk/Wv rows by KV group with their query
    heads, Wo columns by query head, Wg/Wu rows and Wd columns by neuron, all
    in order of device; device l's shard is the l-th contiguous slice.
    Returns (permuted dict, group_order, head_order, neuron_order)."""
    import torch

    go, ho, no = B.layout_orders(h, nu, H, L)
    I = int(w["Wg"].shape[0])
    D = int(w["Wg"].shape[1])
    es = w["Wg"].element_size()
    ws = torch.empty(max(256, 4 * max(H, G, I)), dtype=torch.uint8, device=w["Wg"].device)
    out = {}
    for name, order, n in (("Wq", ho, H), ("Wk", go, G), ("Wv", go, G)):
        out[name] = torch.empty_like(w[name])
        B.gather_blocks(w[name], out[name], 1, n, d_head * D * es, order, ws, stream)
    out["Wo"] = torch.empty_like(w["Wo"])
    B.gather_blocks(w["Wo"], out["Wo"], D, H, d_head * es, ho, ws, stream)
    for name in ("Wg", "Wu"):
        out[name] = torch.empty_like(w[name])
        B.gather_blocks(w[name], out[name], 1, I, D * es, no, ws, stream)
    out["Wd"] = torch.empty_like(w["Wd"])
    B.gather_blocks(w["Wd"], out["Wd"], D, I, es, no, ws, stream)
    return out, go, ho, no
