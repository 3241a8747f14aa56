"""ctypes binding of libaffinity (include/affinity.h).

Argument marshalling only: every function forwards to the C entry point of
the same name.  Device tensors are PyTorch CUDA tensors (PyTorch supplies
device memory and streams); nothing here computes any part of the scores.
Loading fails loudly if the compiled library is missing -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libaffinity.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "affinity.h")

AFF_OK = 0
AFF_ERR_INVALID_ARG = 1
AFF_ERR_UNSUPPORTED_SHAPE = 2
AFF_ERR_UNSUPPORTED_DTYPE = 3
AFF_ERR_ARCH = 4
AFF_ERR_WORKSPACE = 5
AFF_ERR_CUDA = 6
AFF_ERR_DEVICE_TIMEOUT = 7
AFF_ERR_RANGE = 8
AFF_ERR_ALIGNMENT = 9
AFF_ERR_NO_CONVERGENCE = 10

AFF_MODE_FO = 0
AFF_MODE_ADD = 1
AFF_MODE_LOO = 2
AFF_BF16 = 0
AFF_FP32 = 1
AFF_FLAG_ADD_DIRECT = 1
MODES = {"fo": AFF_MODE_FO, "add": AFF_MODE_ADD, "loo": AFF_MODE_LOO}


class aff_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("D", ctypes.c_int64), ("H", ctypes.c_int64), ("G", ctypes.c_int64),
                ("d_head", ctypes.c_int64), ("I", ctypes.c_int64), ("eps", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class aff_assign_opts(ctypes.Structure):
    _fields_ = [("dual_iters", ctypes.c_int32), ("dual_decay", ctypes.c_double), ("max_cycles", ctypes.c_int64)]


class aff_layout_opts(ctypes.Structure):
    _fields_ = [("max_sweeps", ctypes.c_int32), ("freeze_heads", ctypes.c_int32),
                ("freeze_neurons", ctypes.c_int32), ("minimise", ctypes.c_int32),
                ("layer_mask", ctypes.c_void_p), ("assign", aff_assign_opts)]


class AffinityError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: status {status}: {detail}")


_lib = None
_P = ctypes.c_void_p


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libaffinity.so (built by __graft_entry__.build()); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libaffinity.so not found at {path}: run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    st = ctypes.c_int32
    lib.affinity_workspace_size.argtypes = [ctypes.POINTER(aff_dims), ctypes.c_int32, ctypes.c_int32,
                                            ctypes.POINTER(ctypes.c_size_t)]
    lib.affinity_workspace_size.restype = st
    lib.affinity_up.argtypes = [_P] * 7 + [ctypes.POINTER(aff_dims), ctypes.c_int32, _P, _P, _P, ctypes.c_size_t, _P]
    lib.affinity_up.restype = st
    lib.affinity_up_static.argtypes = [_P] * 7 + [ctypes.POINTER(aff_dims), ctypes.c_int32, _P, _P, _P]
    lib.affinity_up_static.restype = st
    lib.affinity_down.argtypes = [_P] * 9 + [ctypes.POINTER(aff_dims), _P, _P, ctypes.c_size_t, _P]
    lib.affinity_down.restype = st
    lib.affinity_device_status.argtypes = [_P, _P]
    lib.affinity_device_status.restype = st
    lib.affinity_static_device_status.argtypes = [_P]
    lib.affinity_static_device_status.restype = st
    lib.affinity_score_partitions.argtypes = [_P, ctypes.c_int32, ctypes.c_int32, _P, ctypes.POINTER(ctypes.c_int64),
                                              ctypes.POINTER(ctypes.c_int64), _P]
    lib.affinity_score_partitions.restype = st
    lib.affinity_group_gain.argtypes = [_P, _P, _P, _P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _P]
    lib.affinity_group_gain.restype = st
    lib.affinity_objective.argtypes = [_P, _P, _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _P]
    lib.affinity_objective.restype = st
    lib.affinity_unit_mass.argtypes = [_P, ctypes.c_int64, _P]
    lib.affinity_unit_mass.restype = st
    lib.affinity_best_heads.argtypes = [_P, _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                        _P, _P]
    lib.affinity_best_heads.restype = st
    lib.affinity_combine_shards.argtypes = [_P, _P, ctypes.c_int32, ctypes.c_int64, _P]
    lib.affinity_combine_shards.restype = st
    lib.affinity_neuron_gain.argtypes = [_P, _P, _P, _P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _P, _P]
    lib.affinity_neuron_gain.restype = st
    lib.affinity_assign_neurons.argtypes = [_P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                            ctypes.POINTER(aff_assign_opts), _P, _P, _P, ctypes.c_size_t, _P]
    lib.affinity_assign_neurons.restype = st
    lib.affinity_layout_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                                   ctypes.POINTER(ctypes.c_size_t)]
    lib.affinity_layout_workspace_size.restype = st
    lib.affinity_optimise_layout.argtypes = [_P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                             ctypes.POINTER(aff_layout_opts), _P, _P, ctypes.POINTER(ctypes.c_double),
                                             ctypes.POINTER(ctypes.c_int32), _P, ctypes.c_size_t, _P]
    lib.affinity_optimise_layout.restype = st
    lib.affinity_selftest_timeout.argtypes = [_P, ctypes.c_size_t, ctypes.c_int64, _P]
    lib.affinity_selftest_timeout.restype = st
    lib.affinity_layout_orders.argtypes = [_P, _P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                           _P, _P, _P]
    lib.affinity_layout_orders.restype = st
    lib.affinity_gather_blocks.argtypes = [_P, _P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _P, _P,
                                           ctypes.c_size_t, _P]
    lib.affinity_gather_blocks.restype = st
    lib.affinity_strerror.argtypes = [ctypes.c_int32]
    lib.affinity_strerror.restype = ctypes.c_char_p
    lib.affinity_last_cuda_error.argtypes = []
    lib.affinity_last_cuda_error.restype = ctypes.c_char_p
    lib.affinity_set_timing_events.argtypes = [_P, _P]
    lib.affinity_set_timing_events.restype = st
    lib.affinity_version.argtypes = []
    lib.affinity_version.restype = ctypes.c_int32
    _lib = lib
    return lib


def strerror(status: int) -> str:
    return load().affinity_strerror(status).decode()


def _check(status: int, where: str) -> None:
    if status != AFF_OK:
        lib = load()
        detail = strerror(status)
        if status == AFF_ERR_CUDA:
            detail += " -- " + lib.affinity_last_cuda_error().decode()
        raise AffinityError(status, where, detail)


def dims(T, D, H, G, d_head, I, eps=1e-6, dtype=AFF_BF16, flags=0) -> aff_dims:
    return aff_dims(int(T), int(D), int(H), int(G), int(d_head), int(I), float(eps), int(dtype), int(flags))


def workspace_size(d: aff_dims, mode: int = AFF_MODE_FO, down: bool = False) -> int:
    n = ctypes.c_size_t(0)
    _check(load().affinity_workspace_size(ctypes.byref(d), int(mode), int(bool(down)), ctypes.byref(n)),
           "affinity_workspace_size")
    return n.value


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ws_bytes(workspace, workspace_bytes):
    if workspace_bytes is not None:
        return int(workspace_bytes)
    if hasattr(workspace, "numel"):
        return workspace.numel() * workspace.element_size()
    raise ValueError("workspace_bytes is required when the workspace is a raw address")


def affinity_up(a, x, Wo, gamma, Wg, Wu, Wd, d: aff_dims, mode: int, S_out, S_head_out, workspace,
                stream=None, workspace_bytes=None) -> None:
    """Enqueue S_up (see include/affinity.h). Tensors are CUDA tensors (or raw device addresses)."""
    nbytes = _ws_bytes(workspace, workspace_bytes)
    _check(load().affinity_up(_ptr(a), _ptr(x), _ptr(Wo), _ptr(gamma), _ptr(Wg), _ptr(Wu), _ptr(Wd),
                              ctypes.byref(d), int(mode), _ptr(S_out), _ptr(S_head_out), _ptr(workspace), nbytes,
                              _stream(stream)), "affinity_up")


def affinity_up_static(a, x, Wo, gamma, Wg, Wu, Wd, d: aff_dims, mode: int, S_out, S_head_out,
                       stream=None) -> None:
    """Enqueue S_up using the library's built-in 64 MiB scratch instead of a workspace."""
    _check(load().affinity_up_static(_ptr(a), _ptr(x), _ptr(Wo), _ptr(gamma), _ptr(Wg), _ptr(Wu), _ptr(Wd),
                                     ctypes.byref(d), int(mode), _ptr(S_out), _ptr(S_head_out), _stream(stream)),
           "affinity_up_static")


def affinity_down(x, gamma, Wg, Wu, Wd, gamma_next, Wq_next, Wk_next, Wv_next, d: aff_dims, S_out, workspace,
                  stream=None, workspace_bytes=None) -> None:
    """Enqueue S_down (see include/affinity.h)."""
    nbytes = _ws_bytes(workspace, workspace_bytes)
    _check(load().affinity_down(_ptr(x), _ptr(gamma), _ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(gamma_next),
                                _ptr(Wq_next), _ptr(Wk_next), _ptr(Wv_next), ctypes.byref(d), _ptr(S_out),
                                _ptr(workspace), nbytes, _stream(stream)), "affinity_down")


def selftest_timeout(workspace, limit_ns: int = 5_000_000, stream=None, workspace_bytes=None) -> None:
    """Enqueue a kernel whose one bounded wait must time out (affinity_selftest_timeout)."""
    _check(load().affinity_selftest_timeout(_ptr(workspace), _ws_bytes(workspace, workspace_bytes), int(limit_ns),
                                            _stream(stream)), "affinity_selftest_timeout")


def device_status(workspace, stream=None) -> int:
    """Synchronise and return (then clear) the device-latched status of the last call."""
    return int(load().affinity_device_status(_ptr(workspace), _stream(stream)))


def static_device_status(stream=None) -> int:
    """As device_status, for the array affinity_up_static uses in place of a workspace."""
    return int(load().affinity_static_device_status(_stream(stream)))


def score_partitions(C: np.ndarray):
    """Score all balanced partitions: returns (scores, count, best_index, best_assign)."""
    lib = load()
    C = np.ascontiguousarray(C, dtype=np.float64)
    G, L = C.shape
    count, best = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib.affinity_score_partitions(C.ctypes.data, G, L, None, ctypes.byref(count), ctypes.byref(best), None),
           "affinity_score_partitions")
    scores = np.empty(count.value, np.float64)
    assign = np.empty(G, np.int32)
    _check(lib.affinity_score_partitions(C.ctypes.data, G, L, scores.ctypes.data, ctypes.byref(count),
                                         ctypes.byref(best), assign.ctypes.data), "affinity_score_partitions")
    return scores, int(count.value), int(best.value), tuple(int(v) for v in assign)


def group_gain(Shat_up_i: np.ndarray, nu_i: Sequence[int], L: int, Shat_down_prev: Optional[np.ndarray] = None,
               nu_prev: Optional[Sequence[int]] = None) -> np.ndarray:
    S = np.ascontiguousarray(Shat_up_i, dtype=np.float64)
    G, I = S.shape
    nu = np.ascontiguousarray(nu_i, dtype=np.int32)
    C = np.zeros((G, L), np.float64)
    Sd = None if Shat_down_prev is None else np.ascontiguousarray(Shat_down_prev, dtype=np.float64)
    npv = None if nu_prev is None else np.ascontiguousarray(nu_prev, dtype=np.int32)
    _check(load().affinity_group_gain(S.ctypes.data, nu.ctypes.data, None if Sd is None else Sd.ctypes.data,
                                      None if npv is None else npv.ctypes.data, G, I, L, C.ctypes.data),
           "affinity_group_gain")
    return C


def objective(Shat_up: Sequence[np.ndarray], Shat_down: Sequence[np.ndarray], h: Sequence, nu: Sequence) -> float:
    N = len(Shat_up)
    G, I = np.asarray(Shat_up[0]).shape
    up = np.ascontiguousarray(np.stack([np.asarray(s, np.float64) for s in Shat_up]))
    dn = np.ascontiguousarray(np.stack([np.asarray(s, np.float64) for s in Shat_down])) if N > 1 else None
    hh = np.ascontiguousarray(np.stack([np.asarray(v, np.int32) for v in h]))
    nn = np.ascontiguousarray(np.stack([np.asarray(v, np.int32) for v in nu]))
    J = ctypes.c_double(0.0)
    _check(load().affinity_objective(up.ctypes.data, None if dn is None else dn.ctypes.data, hh.ctypes.data,
                                     nn.ctypes.data, N, G, I, ctypes.byref(J)), "affinity_objective")
    return J.value


def unit_mass(S: np.ndarray) -> np.ndarray:
    """S / sum(S) in fp64 (affinity_unit_mass); S is a host fp32 array of any shape."""
    S = np.ascontiguousarray(S, dtype=np.float32)
    out = np.empty(S.shape, np.float64)
    _check(load().affinity_unit_mass(S.ctypes.data, S.size, out.ctypes.data), "affinity_unit_mass")
    return out


def best_heads(Shat_up: Sequence[np.ndarray], Shat_down: Sequence[np.ndarray], nu: Sequence, L: int):
    """Best balanced KV-group map of every layer for fixed neuron maps (affinity_best_heads).

    Returns (h [N, G] int32, J of (h, nu))."""
    N = len(Shat_up)
    G, I = np.asarray(Shat_up[0]).shape
    up = np.ascontiguousarray(np.stack([np.asarray(s, np.float64) for s in Shat_up]))
    dn = np.ascontiguousarray(np.stack([np.asarray(s, np.float64) for s in Shat_down])) if N > 1 else None
    nn = np.ascontiguousarray(np.stack([np.asarray(v, np.int32) for v in nu]))
    h = np.empty((N, G), np.int32)
    J = ctypes.c_double(0.0)
    _check(load().affinity_best_heads(up.ctypes.data, None if dn is None else dn.ctypes.data, nn.ctypes.data, N, G,
                                      I, int(L), h.ctypes.data, ctypes.byref(J)), "affinity_best_heads")
    return h, J.value


def combine_shards(S_shards: Sequence[np.ndarray], T_shards: Sequence[int]) -> np.ndarray:
    """Token-weighted merge of S matrices from disjoint token shards (affinity_combine_shards)."""
    arrs = [np.ascontiguousarray(s, dtype=np.float32) for s in S_shards]
    shape = arrs[0].shape
    if any(a.shape != shape for a in arrs):
        raise ValueError("all shards must have the same shape")
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    T = np.ascontiguousarray(T_shards, dtype=np.int64)
    if T.shape != (len(arrs),):
        raise ValueError("one token count per shard")
    out = np.empty(shape, np.float32)
    _check(load().affinity_combine_shards(ctypes.cast(ptrs, ctypes.c_void_p), T.ctypes.data, len(arrs),
                                          arrs[0].size, out.ctypes.data), "affinity_combine_shards")
    return out


def neuron_gain(Shat_up_i, Shat_down_i, h_i, h_next, L: int, M_out, stream=None) -> None:
    """Enqueue M [I, L] (affinity_neuron_gain); Shat_* and M_out are CUDA fp64 tensors."""
    G, I = Shat_up_i.shape
    h = np.ascontiguousarray(h_i, dtype=np.int32)
    hn = None if h_next is None else np.ascontiguousarray(h_next, dtype=np.int32)
    _check(load().affinity_neuron_gain(_ptr(Shat_up_i), _ptr(Shat_down_i), h.ctypes.data,
                                       None if hn is None else hn.ctypes.data, G, I, int(L), _ptr(M_out),
                                       _stream(stream)), "affinity_neuron_gain")


def assign_opts(dual_iters: int = 0, dual_decay: float = 0.0, max_cycles: int = 0) -> aff_assign_opts:
    return aff_assign_opts(int(dual_iters), float(dual_decay), int(max_cycles))


def assign_neurons(M, L: int, nu_out, value_out, workspace, opts: Optional[aff_assign_opts] = None,
                   stream=None, workspace_bytes=None) -> None:
    """Enqueue the balanced neuron solver on M [n, I, L] (CUDA fp64) -> nu_out [n, I] int32, value_out [n] fp64."""
    n, I = (1, M.shape[0]) if M.dim() == 2 else (M.shape[0], M.shape[1])
    _check(load().affinity_assign_neurons(_ptr(M), n, I, int(L), None if opts is None else ctypes.byref(opts),
                                          _ptr(nu_out), _ptr(value_out), _ptr(workspace),
                                          _ws_bytes(workspace, workspace_bytes), _stream(stream)),
           "affinity_assign_neurons")


def layout_workspace_size(N: int, G: int, I: int, L: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().affinity_layout_workspace_size(int(N), int(G), int(I), int(L), ctypes.byref(n)),
           "affinity_layout_workspace_size")
    return n.value


def optimise_layout(Shat_up: Sequence[np.ndarray], Shat_down: Sequence[np.ndarray], L: int, h0, nu0, workspace,
                    max_sweeps: int = 0, freeze_heads: bool = False, freeze_neurons: bool = False,
                    minimise: bool = False, layer_mask=None, assign: Optional[aff_assign_opts] = None,
                    stream=None, workspace_bytes=None):
    """Alternating layout search (affinity_optimise_layout). Returns (h [N, G], nu [N, I], J, sweeps)."""
    N = len(Shat_up)
    G, I = np.asarray(Shat_up[0]).shape
    up = np.ascontiguousarray(np.stack([np.asarray(s, np.float64) for s in Shat_up]))
    dn = np.ascontiguousarray(np.stack([np.asarray(s, np.float64) for s in Shat_down])) if N > 1 else None
    h = np.ascontiguousarray(np.array(h0, dtype=np.int32).reshape(N, G))
    nu = np.ascontiguousarray(np.array(nu0, dtype=np.int32).reshape(N, I))
    mask = None if layer_mask is None else np.ascontiguousarray(layer_mask, dtype=np.uint8)
    opts = aff_layout_opts(int(max_sweeps), int(bool(freeze_heads)), int(bool(freeze_neurons)), int(bool(minimise)),
                           None if mask is None else mask.ctypes.data, assign or aff_assign_opts())
    J = ctypes.c_double(0.0)
    sweeps = ctypes.c_int32(0)
    _check(load().affinity_optimise_layout(up.ctypes.data, None if dn is None else dn.ctypes.data, N, G, I, int(L),
                                           ctypes.byref(opts), h.ctypes.data, nu.ctypes.data, ctypes.byref(J),
                                           ctypes.byref(sweeps), _ptr(workspace),
                                           _ws_bytes(workspace, workspace_bytes), _stream(stream)),
           "affinity_optimise_layout")
    return h, nu, J.value, sweeps.value


def layout_orders(h, nu, H: int, L: int):
    """(group_order [G], head_order [H], neuron_order [I]) realising a balanced layout (affinity_layout_orders)."""
    hh = np.ascontiguousarray(h, dtype=np.int32)
    nn = np.ascontiguousarray(nu, dtype=np.int32)
    go = np.empty(hh.size, np.int32)
    ho = np.empty(int(H), np.int32)
    no = np.empty(nn.size, np.int32)
    _check(load().affinity_layout_orders(hh.ctypes.data, nn.ctypes.data, hh.size, int(H), nn.size, int(L),
                                         go.ctypes.data, ho.ctypes.data, no.ctypes.data), "affinity_layout_orders")
    return go, ho, no


def gather_blocks(src, dst, rows: int, n_blocks: int, block_bytes: int, order, workspace, stream=None,
                  workspace_bytes=None) -> None:
    """Enqueue dst[r][j] = src[r][order[j]] over byte blocks (affinity_gather_blocks); order is a host array."""
    o = np.ascontiguousarray(order, dtype=np.int32)
    _check(load().affinity_gather_blocks(_ptr(src), _ptr(dst), int(rows), int(n_blocks), int(block_bytes),
                                         o.ctypes.data, _ptr(workspace), _ws_bytes(workspace, workspace_bytes),
                                         _stream(stream)), "affinity_gather_blocks")


def set_timing_events(start_event, stop_event) -> None:
    """Record torch.cuda.Event pairs around the dominant kernel of later calls (None, None stops)."""
    h0 = None if start_event is None else start_event.cuda_event
    h1 = None if stop_event is None else stop_event.cuda_event
    _check(load().affinity_set_timing_events(h0, h1), "affinity_set_timing_events")


def version() -> int:
    return int(load().affinity_version())
