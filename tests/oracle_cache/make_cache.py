"""Write the fp64 oracle's full-size results for the GPU parity tests.

TEST INFRASTRUCTURE.  This script calls only the oracle (``oracle/``) and the
seeded input generator (``workloads``, which holds none of the method's
arithmetic).  Nothing it stores comes from the CUDA path.

The oracle takes minutes per full-size layer (65,536 tokens), so the GPU
tests read its results from here instead of recomputing them.  Each file
records a SHA-256 fingerprint of the exact bf16 inputs the generator drew,
and the tests refuse a file whose fingerprint differs from the inputs they
regenerate.

Paper: "Affinity-Aware Sharding for Delayed Tensor Parallelism", §3
"Affinity scores" (S_up for FO / ADD and its exact leave-one-out sibling;
S_down for the down edge).

Usage (from the repository root):
    python tests/oracle_cache/make_cache.py            # every case
    python tests/oracle_cache/make_cache.py qwen3_fo   # named cases
"""
from __future__ import annotations

import hashlib
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import affinity_oracle as O                       # noqa: E402
from transformer_sharding_affinity_gb300 import workloads as W  # noqa: E402

UP_KEYS = ("a", "x", "Wo", "gamma", "Wg", "Wu", "Wd")
DOWN_KEYS = ("x", "gamma", "Wg", "Wu", "Wd", "gamma_next", "Wq_next", "Wk_next", "Wv_next")

# Neurons of the Llama-3-8B-shaped layer the FO oracle evaluates: a seeded
# random draw, independent of any GPU output (the whole 14,336-neuron matrix
# costs about 5e14 fp64 flop, hours on a host).
LLAMA_FO_NEURONS = 2048
LLAMA_FO_SEED = 4242


def llama_fo_neurons(I: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(LLAMA_FO_SEED))
    return np.sort(rng.choice(I, size=LLAMA_FO_NEURONS, replace=False)).astype(np.int64)


def _shape(name: str):
    if name.startswith("stack_l"):
        return W.stack_layer(int(name[len("stack_l"):]))
    return W.CONFIGS[name]


# case name -> (layer name, "up" | "down", mode, neuron subset or None)
CASES = {
    "qwen3_fo": ("qwen3_0p6b_layer", "up", "fo", None),
    "qwen3_add": ("qwen3_0p6b_layer", "up", "add", None),
    "qwen3_loo": ("qwen3_0p6b_layer", "up", "loo", None),
    "qwen3_down": ("qwen3_0p6b_layer", "down", None, None),
    "danube3_fo": ("danube3_500m_layer", "up", "fo", None),
    "danube3_add": ("danube3_500m_layer", "up", "add", None),
    "danube3_down": ("danube3_500m_layer", "down", None, None),
    "llama3_fo": ("llama3_8b_layer", "up", "fo", "llama_sample"),
    "llama3_down": ("llama3_8b_layer", "down", None, None),
    "stack_l0_fo": ("stack_l0", "up", "fo", None),
    "stack_l27_fo": ("stack_l27", "up", "fo", None),
    "stack_l0_down": ("stack_l0", "down", None, None),
    "stack_l26_down": ("stack_l26", "down", None, None),
}


def fingerprint(layer, keys) -> str:
    """SHA-256 over the bf16 bit patterns of the named inputs, in order."""
    h = hashlib.sha256()
    for k in keys:
        bits = np.ascontiguousarray(layer[k + "_bits"])
        h.update(k.encode())
        h.update(str(bits.shape).encode())
        h.update(bits.tobytes())
    return h.hexdigest()


def path_of(case: str) -> str:
    return os.path.join(HERE, case + ".npz")


def make(case: str) -> None:
    layer_name, kind, mode, subset = CASES[case]
    shape = _shape(layer_name)
    t0 = time.time()
    layer = W.make_layer(shape, with_next=(kind == "down"))
    keys = UP_KEYS if kind == "up" else DOWN_KEYS
    fp = fingerprint(layer, keys)
    neurons = llama_fo_neurons(shape.I) if subset == "llama_sample" else None
    out = dict(fingerprint=np.array(fp), layer=np.array(layer_name), kind=np.array(kind),
               mode=np.array(mode or ""), T=np.int64(shape.T),
               neurons=np.arange(shape.I, dtype=np.int64) if neurons is None else neurons)
    if kind == "up":
        S, S_head = O.s_up(layer["a"], layer["x"], layer["Wo"], layer["gamma"], layer["Wg"], layer["Wu"],
                           layer["Wd"], shape.H, shape.G, shape.dh, shape.eps, mode, neurons=neurons)
        out["S"] = np.asarray(S, np.float64)
        out["S_head"] = np.asarray(S_head, np.float64)
    else:
        S = O.s_down(layer["x"], layer["gamma"], layer["Wg"], layer["Wu"], layer["Wd"], layer["gamma_next"],
                     layer["Wq_next"], layer["Wk_next"], layer["Wv_next"], shape.H, shape.G, shape.dh, shape.eps)
        out["S"] = np.asarray(S, np.float64)
    tmp = path_of(case) + ".tmp.npz"
    np.savez_compressed(tmp, **out)
    os.replace(tmp, path_of(case))
    print(f"{case}: {time.time() - t0:.0f} s, S {out['S'].shape}, fingerprint {fp[:16]}", flush=True)


def main(argv) -> None:
    cases = argv or list(CASES)
    for c in cases:
        if c not in CASES:
            raise SystemExit(f"unknown case {c}; known: {', '.join(CASES)}")
    for c in cases:
        make(c)


if __name__ == "__main__":
    main(sys.argv[1:])
