"""Pins of the neuron-step oracle ("Affinity-Aware Sharding for Delayed Tensor
Parallelism", §3 "Optimiser"): the gain M against the objective J of
equation (6), the exact solver against exhaustive search, and the
exchange-cycle optimality certificate against both."""
import itertools

import numpy as np
import pytest

from oracle import assignment as A
from oracle import partitions as P


def _unit(rng, shape):
    return P.unit_mass(rng.random(shape))


def test_gain_differences_are_objective_differences():
    """With everything else fixed, J(nu_0) - J(nu_0') equals the difference of
    sum_k M_0[k, nu_0(k)]: M carries exactly the nu_0-dependent part of J."""
    rng = np.random.default_rng(1)
    G, I, L = 8, 24, 4
    ups = [_unit(rng, (G, I)) for _ in range(2)]
    dn = [_unit(rng, (I, G))]
    h = [rng.permutation(P.contiguous_heads(G, L)) for _ in range(2)]
    nu1 = rng.permutation(P.contiguous_neurons(I, L))
    M = A.neuron_gain(ups[0], h[0], L, dn[0], h[1])
    base = rng.permutation(P.contiguous_neurons(I, L))
    for _ in range(10):
        other = rng.permutation(P.contiguous_neurons(I, L))
        dJ = P.objective_J(ups, dn, h, [base, nu1]) - P.objective_J(ups, dn, h, [other, nu1])
        dV = A.assignment_value(M, base) - A.assignment_value(M, other)
        np.testing.assert_allclose(dJ, dV, rtol=1e-12, atol=1e-15)


def test_gain_row_sums_do_not_depend_on_the_head_maps():
    rng = np.random.default_rng(2)
    G, I, L = 8, 40, 4
    up, dn = _unit(rng, (G, I)), _unit(rng, (I, G))
    ref = up.sum(0) + dn.sum(1)
    for _ in range(5):
        h0, h1 = rng.permutation(P.contiguous_heads(G, L)), rng.permutation(P.contiguous_heads(G, L))
        np.testing.assert_allclose(A.neuron_gain(up, h0, L, dn, h1).sum(1), ref, rtol=1e-13)
    # last layer: only the S_up term
    np.testing.assert_allclose(A.neuron_gain(up, h0, L).sum(1), up.sum(0), rtol=1e-13)


@pytest.mark.parametrize("I,L,seed", [(8, 2, 0), (8, 4, 1), (9, 3, 2), (12, 3, 3), (10, 2, 4)])
def test_exact_solver_matches_exhaustive_search(I, L, seed):
    M = np.random.default_rng(seed).random((I, L))
    nu, v = A.best_balanced_neurons(M)
    best, maps = A.brute_force_best(M)
    np.testing.assert_allclose(v, best, rtol=1e-14)
    assert tuple(nu) in maps
    assert all(np.bincount(nu, minlength=L) == I // L)


@pytest.mark.parametrize("I,L,seed", [(8, 2, 5), (8, 4, 6), (9, 3, 7)])
def test_cycle_certificate_separates_optimal_from_suboptimal_maps(I, L, seed):
    """The certificate is <= 0 on every exhaustive optimum and > 0 on every
    balanced map that is worse (checked over all balanced maps)."""
    M = np.random.default_rng(seed).random((I, L))
    best, _ = A.brute_force_best(M)
    cap = I // L
    for m in itertools.product(range(L), repeat=I):
        if any(m.count(l) != cap for l in range(L)):
            continue
        gain = A.device_cycle_gains(M, m)
        if A.assignment_value(M, m) >= best - 1e-13:
            assert gain <= 1e-13
        else:
            assert gain > 0


def test_exact_solver_passes_the_certificate_at_layer_size():
    rng = np.random.default_rng(8)
    G, I, L = 8, 768, 4
    M = A.neuron_gain(_unit(rng, (G, I)), rng.permutation(P.contiguous_heads(G, L)), L,
                      _unit(rng, (I, G)), rng.permutation(P.contiguous_heads(G, L)))
    nu, v = A.best_balanced_neurons(M)
    assert A.device_cycle_gains(M, nu) <= 1e-15
    assert all(np.bincount(nu, minlength=L) == I // L)
    # never worse than the contiguous map or a random balanced map
    assert v >= A.assignment_value(M, P.contiguous_neurons(I, L)) - 1e-15
    assert v >= A.assignment_value(M, rng.permutation(P.contiguous_neurons(I, L))) - 1e-15


def test_separable_preferences_give_the_closed_form():
    """Neuron k gains 1 only on device k mod L: every neuron gets its device, value I."""
    I, L = 64, 4
    M = np.zeros((I, L))
    M[np.arange(I), np.arange(I) % L] = 1.0
    nu, v = A.best_balanced_neurons(M)
    assert v == I
    np.testing.assert_array_equal(nu, np.arange(I) % L)
