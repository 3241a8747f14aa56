"""Dense and tensor-parallel forward pass of one pre-norm decoder layer, fp64.

TEST INFRASTRUCTURE: only ``tests/`` may import this module.  It shares no code
with the library.

Source: "Affinity-Aware Sharding for Delayed Tensor Parallelism", §3 "The
layout as a free variable".  A balanced layout (h, nu) is realised by
permuting the rows of the query, key and value projections by KV group
(each group keeps its query heads), the columns of the output projection the
same way, the rows of the gate and up projections and the columns of the
down projection by neuron, and then slicing contiguous shards.  The rotary
embedding, Qwen3's per-head q/k norms and SwiGLU act per head or per neuron,
so the dense function does not change.  The paper's §2 describes the
Megatron split used here: attention by heads, the FFN by neurons, each device
adding its partial output.

The layer: x1 = x + Attn(rmsnorm(x) * g_attn); y = x1 + FFN(rmsnorm(x1) * g_ffn),
with grouped-query causal softmax attention, rotary position embedding on q
and k (pairs (j, j + d/2), base 10000), optional per-head rms norms of q and
k with shared gains, and FFN(z) = (silu(z Wg^T) * (z Wu^T)) Wd^T.
"""
from __future__ import annotations

import numpy as np

F = np.float64


def rmsnorm(x, gain, eps=1e-6):
    x = np.asarray(x, F)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(gain, F)


def rope(x, base=10000.0):
    """x [T, n_heads, d]: rotate pairs (j, j + d/2) by angle t / base^(2j/d)."""
    T, _, d = x.shape
    half = d // 2
    inv = base ** (-np.arange(half, dtype=F) * 2.0 / d)
    ang = np.arange(T, dtype=F)[:, None] * inv[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def attention_heads(x, w, H, G, dh, heads=None):
    """Per-head attention outputs [T, len(heads), dh] of the given query heads."""
    T = x.shape[0]
    z = rmsnorm(x, w["g_attn"])
    q = (z @ np.asarray(w["Wq"], F).T).reshape(T, H, dh)
    k = (z @ np.asarray(w["Wk"], F).T).reshape(T, G, dh)
    v = (z @ np.asarray(w["Wv"], F).T).reshape(T, G, dh)
    if "qn" in w:
        q = rmsnorm(q, w["qn"])
        k = rmsnorm(k, w["kn"])
    q, k = rope(q), rope(k)
    heads = range(H) if heads is None else heads
    out = []
    mask = np.triu(np.full((T, T), -np.inf), 1)
    for h in heads:
        g = h // (H // G)
        s = q[:, h, :] @ k[:, g, :].T / np.sqrt(dh) + mask
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        out.append(p @ v[:, g, :])
    return np.stack(out, axis=1)


def layer_forward(x, w, H, G, dh):
    """Dense layer output [T, D]."""
    x = np.asarray(x, F)
    T = x.shape[0]
    o = attention_heads(x, w, H, G, dh).reshape(T, H * dh) @ np.asarray(w["Wo"], F).T
    x1 = x + o
    z = rmsnorm(x1, w["g_ffn"])
    g = z @ np.asarray(w["Wg"], F).T
    u = z @ np.asarray(w["Wu"], F).T
    act = g / (1.0 + np.exp(-g)) * u
    return x1 + act @ np.asarray(w["Wd"], F).T


def sharded_forward(x, w, H, G, dh, L):
    """The same layer on L devices: device l holds rows/columns
    [l*n/L, (l+1)*n/L) of every sharded matrix (KV groups, their query heads,
    neurons) and the partial outputs are summed."""
    x = np.asarray(x, F)
    T, D = x.shape
    Hl, Gl = H // L, G // L
    I = np.asarray(w["Wg"]).shape[0]
    Il = I // L
    o = np.zeros((T, D))
    for l in range(L):
        wl = dict(w)
        wl["Wq"] = np.asarray(w["Wq"])[l * Hl * dh:(l + 1) * Hl * dh]
        wl["Wk"] = np.asarray(w["Wk"])[l * Gl * dh:(l + 1) * Gl * dh]
        wl["Wv"] = np.asarray(w["Wv"])[l * Gl * dh:(l + 1) * Gl * dh]
        a = attention_heads(x, wl, Hl, Gl, dh).reshape(T, Hl * dh)
        o += a @ np.asarray(w["Wo"], F)[:, l * Hl * dh:(l + 1) * Hl * dh].T
    x1 = x + o
    z = rmsnorm(x1, w["g_ffn"])
    y = np.zeros((T, D))
    for l in range(L):
        sl = slice(l * Il, (l + 1) * Il)
        g = z @ np.asarray(w["Wg"], F)[sl].T
        u = z @ np.asarray(w["Wu"], F)[sl].T
        y += (g / (1.0 + np.exp(-g)) * u) @ np.asarray(w["Wd"], F)[:, sl].T
    return x1 + y


def realise(w, h, nu, H, G, dh, L):
    """Permuted weights of the layout: KV groups in order of device (stable),
    each followed by its query heads; neurons in order of device (stable)."""
    group_order = np.argsort(np.asarray(h), kind="stable")
    hpg = H // G
    head_order = np.concatenate([np.arange(g * hpg, (g + 1) * hpg) for g in group_order])
    neuron_order = np.argsort(np.asarray(nu), kind="stable")

    def rows(m, order, block):
        m = np.asarray(m)
        return m.reshape(-1, block, m.shape[1])[order].reshape(m.shape)

    out = dict(w)
    out["Wq"] = rows(w["Wq"], head_order, dh)
    out["Wk"] = rows(w["Wk"], group_order, dh)
    out["Wv"] = rows(w["Wv"], group_order, dh)
    out["Wo"] = rows(np.asarray(w["Wo"]).T, head_order, dh).T
    out["Wg"] = np.asarray(w["Wg"])[neuron_order]
    out["Wu"] = np.asarray(w["Wu"])[neuron_order]
    out["Wd"] = np.asarray(w["Wd"])[:, neuron_order]
    return out, group_order, head_order, neuron_order
