"""Layout objective and KV-group partition search, plain Python/numpy (fp64).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s oracle legs may import this module.

Source: "Affinity-Aware Sharding for Delayed Tensor Parallelism", §3
"The layout as a free variable" (balanced maps h_i: groups -> devices and
nu_i: neurons -> devices), "Objective" (unit-mass normalisation and the total
co-located affinity J, eq. 6) and "Optimiser" (scoring every labelled
balanced partition of the KV groups, G!/((G/L)!)^L of them, given the
neighbouring neuron assignments).

Readings of points the paper leaves open:
  * Partitions are enumerated lexicographically over (h(0), ..., h(G-1)) and
    the first maximum wins ties.
  * The gain of placing group g of layer i on device l, given nu_{i-1} and
    nu_i, is the part of J that depends on h_i(g):
      C[g, l] = sum_{k: nu_i(k) = l} Shat_up_i[g, k]
              + sum_{k: nu_{i-1}(k) = l} Shat_down_{i-1}[k, g]   (second term only for i > 0).
  * Contiguous layouts: group g -> g // (G/L), neuron k -> k // (I/L).
"""
from __future__ import annotations

import itertools
from math import factorial

import numpy as np


def partition_count(G: int, L: int) -> int:
    """G! / ((G/L)!)^L, the number of labelled balanced partitions ("Optimiser")."""
    if G % L:
        raise ValueError("G must be a multiple of L")
    return factorial(G) // factorial(G // L) ** L


def balanced_partitions(G: int, L: int):
    """All maps h: {0..G-1} -> {0..L-1} with exactly G/L groups per device,
    in lexicographic order of (h(0), ..., h(G-1))."""
    cap = G // L
    out = []
    h = [0] * G
    used = [0] * L

    def rec(g):
        if g == G:
            out.append(tuple(h))
            return
        for l in range(L):
            if used[l] < cap:
                used[l] += 1
                h[g] = l
                rec(g + 1)
                used[l] -= 1

    rec(0)
    return out


def score_partitions(C: np.ndarray):
    """Score every balanced partition by sum_g C[g, h(g)].

    Returns (scores [count], best_index, best_assign) with the first maximum.
    """
    C = np.asarray(C, np.float64)
    G, L = C.shape
    parts = balanced_partitions(G, L)
    scores = np.array([sum(C[g, p[g]] for g in range(G)) for p in parts], np.float64)
    best = int(np.argmax(scores))
    return scores, best, parts[best]


def unit_mass(S: np.ndarray) -> np.ndarray:
    """Shat = S / sum(S) ("Objective": each matrix normalised to unit mass)."""
    S = np.asarray(S, np.float64)
    return S / S.sum()


def contiguous_heads(G: int, L: int) -> np.ndarray:
    return np.arange(G) // (G // L)


def contiguous_neurons(I: int, L: int) -> np.ndarray:
    return np.arange(I) // (I // L)


def objective_J(S_up_hat, S_down_hat, h_maps, nu_maps) -> float:
    """Eq. (6): J = sum_i sum_{g,k: h_i(g) = nu_i(k)} Shat_up_i[g, k]
                  + sum_{i < N-1} sum_{k,g: nu_i(k) = h_{i+1}(g)} Shat_down_i[k, g].

    S_up_hat: N matrices [G, I]; S_down_hat: N-1 matrices [I, G];
    h_maps: N arrays [G]; nu_maps: N arrays [I].
    """
    N = len(S_up_hat)
    J = 0.0
    for i in range(N):
        h, nu = np.asarray(h_maps[i]), np.asarray(nu_maps[i])
        S = np.asarray(S_up_hat[i], np.float64)
        for g in range(S.shape[0]):
            for k in range(S.shape[1]):
                if h[g] == nu[k]:
                    J += S[g, k]
    for i in range(N - 1):
        nu, h_next = np.asarray(nu_maps[i]), np.asarray(h_maps[i + 1])
        S = np.asarray(S_down_hat[i], np.float64)
        for k in range(S.shape[0]):
            for g in range(S.shape[1]):
                if nu[k] == h_next[g]:
                    J += S[k, g]
    return J


def group_gain(S_up_hat_i, L, nu_i, S_down_hat_prev=None, nu_prev=None) -> np.ndarray:
    """C[g, l] for layer i given nu_i (and nu_{i-1}, Shat_down_{i-1} when i > 0)."""
    S = np.asarray(S_up_hat_i, np.float64)
    G, I = S.shape
    C = np.zeros((G, L), np.float64)
    for g in range(G):
        for k in range(I):
            C[g, nu_i[k]] += S[g, k]
    if S_down_hat_prev is not None:
        Sd = np.asarray(S_down_hat_prev, np.float64)
        for k in range(Sd.shape[0]):
            for g in range(G):
                C[g, nu_prev[k]] += Sd[k, g]
    return C


def all_balanced_maps(n: int, L: int):
    """Every balanced map of n items onto L devices (tiny n only)."""
    cap = n // L
    return [m for m in itertools.product(range(L), repeat=n)
            if all(m.count(l) == cap for l in range(L))]
