"""Neuron step of the layout search, plain numpy/scipy (fp64).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s oracle legs may import this module.  It shares no code with the
library.

Source: "Affinity-Aware Sharding for Delayed Tensor Parallelism", §3
"Optimiser".  Given the KV-group maps h_i and h_{i+1}, the gain of putting
neuron k of layer i on device l is

    M[k, l] = sum_{g: h_i(g) = l} Shat_up_i[g, k] + sum_{g: h_{i+1}(g) = l} Shat_down_i[k, g],

and the best balanced neuron map nu_i (I/L neurons per device) maximises
sum_k M[k, nu_i(k)].  The paper names this a linear assignment problem on
I/L replicated slots per device and cites the Hungarian method and the
shortest-augmenting-path solver of Crouse (2016); the oracle solves exactly
that problem with scipy's implementation of the latter.

Readings of points the paper leaves open:
  * For the last layer of a stack (no h_{i+1}) only the S_up term enters.
  * Ties between equally good maps are not resolved the same way as the
    GPU solver; comparisons use the objective value, and the map itself only
    where the optimum is unique.
"""
from __future__ import annotations

import itertools

import numpy as np
from scipy.optimize import linear_sum_assignment


def neuron_gain(Shat_up_i, h_i, L, Shat_down_i=None, h_next=None) -> np.ndarray:
    """M [I, L] from the unit-mass S_up_i [G, I] (and S_down_i [I, G] with h_{i+1})."""
    S = np.asarray(Shat_up_i, np.float64)
    G, I = S.shape
    M = np.zeros((I, L), np.float64)
    for g in range(G):
        M[:, h_i[g]] += S[g]
    if Shat_down_i is not None:
        Sd = np.asarray(Shat_down_i, np.float64)
        for g in range(G):
            M[:, h_next[g]] += Sd[:, g]
    return M


def best_balanced_neurons(M):
    """Exact maximiser of sum_k M[k, nu(k)] over maps with I/L neurons per device.

    Slot j of the replicated assignment belongs to device j // (I/L).
    Returns (nu [I] int, objective)."""
    M = np.asarray(M, np.float64)
    I, L = M.shape
    if I % L:
        raise ValueError("I must be a multiple of L")
    cap = I // L
    cost = -np.repeat(M, cap, axis=1)          # [I, I]: column j is a slot on device j // cap
    rows, cols = linear_sum_assignment(cost)
    nu = np.empty(I, np.int64)
    nu[rows] = cols // cap
    return nu, float(M[np.arange(I), nu].sum())


def assignment_value(M, nu) -> float:
    M = np.asarray(M, np.float64)
    return float(M[np.arange(M.shape[0]), np.asarray(nu)].sum())


def brute_force_best(M):
    """Every balanced map of a tiny M (exhaustive); returns (best value, all optimal maps)."""
    M = np.asarray(M, np.float64)
    I, L = M.shape
    cap = I // L
    best, arg = -np.inf, []
    for m in itertools.product(range(L), repeat=I):
        if any(m.count(l) != cap for l in range(L)):
            continue
        v = assignment_value(M, m)
        if v > best + 1e-15:
            best, arg = v, [m]
        elif abs(v - best) <= 1e-15:
            arg.append(m)
    return best, arg


def device_cycle_gains(M, nu):
    """Gain of every simple cycle of devices under single-neuron moves.

    Moving neuron k from device a to device b changes the objective by
    M[k, b] - M[k, a]; a cycle a1 -> a2 -> ... -> a1 moves one neuron out of
    each device on it, keeping every device's count.  Returns the largest
    cycle gain using, on each edge, the best neuron of its source device.
    A balanced map is optimal exactly when this is <= 0 (no improving
    exchange cycle)."""
    M = np.asarray(M, np.float64)
    I, L = M.shape
    nu = np.asarray(nu)
    w = np.full((L, L), -np.inf)
    for a in range(L):
        ks = np.nonzero(nu == a)[0]
        for b in range(L):
            if a != b and len(ks):
                w[a, b] = np.max(M[ks, b] - M[ks, a])
    best = -np.inf
    for r in range(2, L + 1):
        for cyc in itertools.permutations(range(L), r):
            if cyc[0] != min(cyc):
                continue
            best = max(best, sum(w[cyc[i], cyc[(i + 1) % r]] for i in range(r)))
    return best
