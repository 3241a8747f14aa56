"""GPU layout search against the oracle ("Affinity-Aware Sharding for Delayed
Tensor Parallelism", §3 "Optimiser"): the neuron gain bit for bit, the
balanced neuron solver against the Hungarian-type exact solver and the
exchange-cycle certificate, and the alternating search against the oracle's
two steps at its fixed point."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import assignment as A  # noqa: E402
from oracle import partitions as P  # noqa: E402
from transformer_sharding_affinity_gb300 import binding as B  # noqa: E402
from transformer_sharding_affinity_gb300 import stack as ST  # noqa: E402

pytestmark = pytest.mark.gpu


def _unit(rng, shape):
    return P.unit_mass(rng.random(shape))


def _gain(up, dn, h, hn, L):
    G, I = up.shape
    M = torch.empty(I, L, dtype=torch.float64, device="cuda")
    d_up = torch.from_numpy(np.ascontiguousarray(up)).cuda()
    d_dn = None if dn is None else torch.from_numpy(np.ascontiguousarray(dn)).cuda()
    B.neuron_gain(d_up, d_dn, h, hn, L, M)
    return M.cpu().numpy()


def _solve(M_np, L, opts=None, expect_status=0):
    M = torch.from_numpy(np.ascontiguousarray(M_np)).cuda()
    n, I = (1, M_np.shape[0]) if M_np.ndim == 2 else M_np.shape[:2]
    nu = torch.empty(n, I, dtype=torch.int32, device="cuda")
    val = torch.empty(n, dtype=torch.float64, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    B.assign_neurons(M, L, nu, val, ws, opts)
    st = B.device_status(ws)
    assert st == expect_status, f"device status {st}: {B.strerror(st)}"
    return nu.cpu().numpy(), val.cpu().numpy()


def _layer_gain(rng, G, I, L, last=False):
    up = _unit(rng, (G, I))
    h = rng.permutation(P.contiguous_heads(G, L))
    if last:
        return A.neuron_gain(up, h, L)
    return A.neuron_gain(up, h, L, _unit(rng, (I, G)), rng.permutation(P.contiguous_heads(G, L)))


@pytest.mark.parametrize("last", [False, True])
def test_neuron_gain_is_bit_exact(last):
    rng = np.random.default_rng(3)
    G, I, L = 8, 3072, 4
    up, dn = _unit(rng, (G, I)), _unit(rng, (I, G))
    h, hn = rng.permutation(P.contiguous_heads(G, L)), rng.permutation(P.contiguous_heads(G, L))
    got = _gain(up, None if last else dn, h, None if last else hn, L)
    ref = A.neuron_gain(up, h, L) if last else A.neuron_gain(up, h, L, dn, hn)
    assert np.array_equal(got.view(np.uint64), ref.view(np.uint64))


@pytest.mark.parametrize("I,L,G", [(3072, 4, 8), (4096, 4, 8), (96, 8, 16), (48, 3, 6), (64, 2, 4), (8, 1, 2)])
def test_assign_matches_the_exact_solver(I, L, G):
    rng = np.random.default_rng(I + L)
    M = _layer_gain(rng, G, I, L)
    nu, val = _solve(M, L)
    nu = nu[0]
    ref_nu, ref_val = A.best_balanced_neurons(M)
    assert np.all(np.bincount(nu, minlength=L) == I // L)
    np.testing.assert_allclose(val[0], ref_val, rtol=1e-12)
    np.testing.assert_allclose(val[0], A.assignment_value(M, nu), rtol=1e-13)
    assert A.device_cycle_gains(M, nu) <= 1e-15
    if not np.array_equal(nu, ref_nu):   # only possible when two maps tie to rounding
        np.testing.assert_allclose(A.assignment_value(M, nu), A.assignment_value(M, ref_nu), rtol=1e-13)


def test_assign_at_llama_width_passes_the_certificate():
    rng = np.random.default_rng(11)
    I, L = 14336, 4
    M = _layer_gain(rng, 8, I, L)
    nu, val = _solve(M, L)
    nu = nu[0]
    assert np.all(np.bincount(nu, minlength=L) == I // L)
    assert A.device_cycle_gains(M, nu) <= 1e-15
    assert val[0] >= A.assignment_value(M, P.contiguous_neurons(I, L))


def test_assign_batched_equals_single_and_is_deterministic():
    rng = np.random.default_rng(5)
    Ms = np.stack([_layer_gain(rng, 8, 768, 4, last=(i == 2)) for i in range(3)])
    nu_b, val_b = _solve(Ms, 4)
    nu_b2, val_b2 = _solve(Ms, 4)
    assert np.array_equal(nu_b, nu_b2) and np.array_equal(val_b.view(np.uint64), val_b2.view(np.uint64))
    for i in range(3):
        nu_s, val_s = _solve(Ms[i], 4)
        assert np.array_equal(nu_s[0], nu_b[i]) and val_s[0] == val_b[i]


def test_assign_from_a_poor_start_still_reaches_the_optimum():
    """One dual step leaves the work to the fix-up and the exchange cycles."""
    rng = np.random.default_rng(6)
    M = _layer_gain(rng, 8, 1024, 4)
    nu, val = _solve(M, 4, B.assign_opts(dual_iters=1))
    _, ref_val = A.best_balanced_neurons(M)
    np.testing.assert_allclose(val[0], ref_val, rtol=1e-12)
    assert A.device_cycle_gains(M, nu[0]) <= 1e-15


def test_assign_reports_the_cycle_cap():
    rng = np.random.default_rng(7)
    M = _layer_gain(rng, 8, 3072, 4)
    nu, _ = _solve(M, 4, B.assign_opts(dual_iters=1, max_cycles=1), expect_status=B.AFF_ERR_NO_CONVERGENCE)
    assert np.all(np.bincount(nu[0], minlength=4) == 3072 // 4)


def _stack(rng, N, G, I):
    return [_unit(rng, (G, I)) for _ in range(N)], [_unit(rng, (I, G)) for _ in range(N - 1)]


def _assert_fixed_point(up, dn, L, h, nu, minimise=False):
    """Neither step of the oracle improves the returned layout."""
    N = len(up)
    sgn = -1.0 if minimise else 1.0
    for i in range(N):
        M = sgn * (A.neuron_gain(up[i], h[i], L, dn[i], h[i + 1]) if i + 1 < N else A.neuron_gain(up[i], h[i], L))
        _, best = A.best_balanced_neurons(M)
        np.testing.assert_allclose(A.assignment_value(M, nu[i]), best, rtol=1e-12)
        C = sgn * P.group_gain(up[i], L, nu[i], dn[i - 1] if i else None, nu[i - 1] if i else None)
        scores, _, _ = P.score_partitions(C)
        np.testing.assert_allclose(sum(C[g, h[i][g]] for g in range(len(h[i]))), scores.max(), rtol=1e-12)


def test_optimise_layout_reaches_a_fixed_point_of_both_steps():
    rng = np.random.default_rng(9)
    N, G, I, L = 4, 8, 256, 4
    up, dn = _stack(rng, N, G, I)
    res = ST.optimise(up, dn, L)
    J0 = P.objective_J(up, dn, [P.contiguous_heads(G, L)] * N, [P.contiguous_neurons(I, L)] * N)
    np.testing.assert_allclose(res.J, P.objective_J(up, dn, list(res.h), list(res.nu)), rtol=1e-12)
    assert res.J > J0 and 1 <= res.sweeps <= 16
    for i in range(N):
        assert np.all(np.bincount(res.nu[i], minlength=L) == I // L)
        assert np.all(np.bincount(res.h[i], minlength=L) == G // L)
    _assert_fixed_point(up, dn, L, res.h, res.nu)


def test_optimise_layout_options():
    rng = np.random.default_rng(10)
    N, G, I, L = 3, 8, 128, 4
    up, dn = _stack(rng, N, G, I)
    hc, nc = np.stack([P.contiguous_heads(G, L)] * N), np.stack([P.contiguous_neurons(I, L)] * N)
    J0 = P.objective_J(up, dn, list(hc), list(nc))
    r = ST.optimise(up, dn, L, freeze_heads=True)
    assert np.array_equal(r.h, hc) and r.J >= J0
    r = ST.optimise(up, dn, L, freeze_neurons=True)
    assert np.array_equal(r.nu, nc) and r.J >= J0
    r = ST.optimise(up, dn, L, minimise=True)
    assert r.J < J0
    np.testing.assert_allclose(r.J, P.objective_J(up, dn, list(r.h), list(r.nu)), rtol=1e-12)
    _assert_fixed_point(up, dn, L, r.h, r.nu, minimise=True)
    mask = np.array([1, 0, 1], np.uint8)
    r = ST.optimise(up, dn, L, layer_mask=mask)
    assert np.array_equal(r.h[1], hc[1]) and np.array_equal(r.nu[1], nc[1]) and r.J >= J0
