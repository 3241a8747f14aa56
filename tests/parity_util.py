"""Helpers shared by the GPU parity tests: run the C ABI on seeded inputs,
compare with the oracle under the acceptance rule (max relative error on
entries >= 1e-6 * max, identical top-8 neurons per KV group with near ties
tolerated)."""
from __future__ import annotations

import numpy as np

TOL = 2e-3          # max relative error against the fp64 oracle (bf16 operands, fp32 accumulate)
TOL_F32 = 1e-4      # fp32 path
FLOOR = 1e-6        # entries below FLOOR * max(S) are not compared
TOPK = 8
FEW_TOKENS = 64     # below this many tokens nothing averages the fp16 roundings of a single
                    # token's dot products, and the bar is taken norm-wise (see rowmax_err)


def rel_err(got: np.ndarray, ref: np.ndarray, floor_ref: float | None = None) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    top = ref.max() if floor_ref is None else floor_ref
    m = ref >= FLOOR * top
    if not m.any():
        return 0.0
    return float(np.max(np.abs(got[m] - ref[m]) / ref[m]))


def rowmax_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max_{g,k} |got - ref| / max_k ref[g, :] -- the error relative to each row's largest entry."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rmax = ref.max(axis=1, keepdims=True)
    rmax[rmax == 0] = 1.0
    return float(np.max(np.abs(got - ref) / rmax))


def topk_agrees(got_row: np.ndarray, ref_row: np.ndarray, k: int = TOPK, tie: float = TOL) -> bool:
    """Rank both rows descending (ties to the lower index).  Position by position,
    the neuron the GPU puts there must be the oracle's, or the oracle's values of
    the two neurons must be within `tie` relative of each other (a near tie)."""
    og = np.argsort(-np.asarray(got_row), kind="stable")[:k]
    orf = np.argsort(-np.asarray(ref_row), kind="stable")[:k]
    for i in range(min(k, len(og))):
        if og[i] != orf[i]:
            a, b = ref_row[og[i]], ref_row[orf[i]]
            if abs(a - b) > tie * max(abs(a), abs(b)):
                return False
    return True


def dims_of(B, shape, flags=0):
    return B.dims(shape.T, shape.D, shape.H, shape.G, shape.dh, shape.I, shape.eps,
                  B.AFF_BF16 if shape.dtype == "bf16" else B.AFF_FP32, flags)


def mode_of(B, mode: str):
    """(aff_mode, flags) for a test mode name; "add_direct" is ADD in its direct form."""
    if mode == "add_direct":
        return B.AFF_MODE_ADD, B.AFF_FLAG_ADD_DIRECT
    return B.MODES[mode], 0


def run_up(B, DV, shape, layer, mode: str, runs: int = 1, per_head: bool = True):
    import torch
    dev = DV.to_device(layer, shape.dtype)
    m, flags = mode_of(B, mode)
    d = dims_of(B, shape, flags)
    ws = torch.empty(B.workspace_size(d, m), dtype=torch.uint8, device="cuda")
    S = torch.empty(shape.G, shape.I, device="cuda")
    Sh = torch.empty(shape.H, shape.I, device="cuda") if per_head else None
    outs = []
    for _ in range(runs):
        S.fill_(float("nan"))
        if Sh is not None:
            Sh.fill_(float("nan"))
        B.affinity_up(dev["a"], dev["x"], dev["Wo"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], d,
                      m, S, Sh, ws)
        st = B.device_status(ws)
        assert st == 0, f"device status {st}: {B.strerror(st)}"
        outs.append((S.cpu().numpy().copy(), None if Sh is None else Sh.cpu().numpy().copy()))
    return outs


def run_down(B, DV, shape, layer, runs: int = 1):
    import torch
    dev = DV.to_device(layer, shape.dtype, keys=DV.DOWN_KEYS)
    d = dims_of(B, shape)
    ws = torch.empty(B.workspace_size(d, 0, down=True), dtype=torch.uint8, device="cuda")
    S = torch.empty(shape.I, shape.G, device="cuda")
    outs = []
    for _ in range(runs):
        S.fill_(float("nan"))
        B.affinity_down(dev["x"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], dev["gamma_next"], dev["Wq_next"],
                        dev["Wk_next"], dev["Wv_next"], d, S, ws)
        st = B.device_status(ws)
        assert st == 0, f"device status {st}: {B.strerror(st)}"
        outs.append(S.cpu().numpy().copy())
    return outs


def oracle_up(O, shape, layer, mode, neurons=None):
    mode = "add" if mode == "add_direct" else mode
    return O.s_up(layer["a"], layer["x"], layer["Wo"], layer["gamma"], layer["Wg"], layer["Wu"], layer["Wd"],
                  shape.H, shape.G, shape.dh, shape.eps, mode, neurons=neurons)


def oracle_down(O, shape, layer, neurons=None):
    return O.s_down(layer["x"], layer["gamma"], layer["Wg"], layer["Wu"], layer["Wd"], layer["gamma_next"],
                    layer["Wq_next"], layer["Wk_next"], layer["Wv_next"], shape.H, shape.G, shape.dh, shape.eps,
                    neurons=neurons)
