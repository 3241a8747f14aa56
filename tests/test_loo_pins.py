"""Pins of the oracle's leave-one-out score ("Affinity-Aware Sharding for
Delayed Tensor Parallelism", §3 "Affinity scores": exact leave-one-out
ablation of the pre-activations, which differs from ADD only by the change of
the norm's rms when a head is removed)."""
import numpy as np
import pytest

from oracle import affinity_oracle as O


def _layer(seed, T=24, D=32, H=4, G=2, dh=8, I=40):
    rng = np.random.default_rng(seed)
    return dict(a=rng.standard_normal((T, H * dh)), x=rng.standard_normal((T, D)),
                Wo=0.2 * rng.standard_normal((D, H * dh)), gamma=1 + 0.1 * rng.standard_normal(D),
                Wg=0.2 * rng.standard_normal((I, D)), Wu=0.2 * rng.standard_normal((I, D)),
                Wd=0.2 * rng.standard_normal((D, I))), (H, G, dh)


def _up(l, hg, mode, eps=1e-6, **kw):
    H, G, dh = hg
    return O.s_up(l["a"], l["x"], l["Wo"], l["gamma"], l["Wg"], l["Wu"], l["Wd"], H, G, dh, eps, mode, **kw)


@pytest.mark.parametrize("s", [1e-4, 1e-5])
def test_small_heads_follow_the_first_order_expansion(s):
    """With the heads' writes c_h scaled by s -> 0, the rms of x - c_h moves by
    -(x . c_h) / (D r) to first order, so
      g_k - g_k^(-h) = p_h . w^g_k - g_k (x . c_h) / (D r^2) + O(s^2)
    (likewise for u), i.e. LOO / s^2 -> E_t[(pg - g kappa)^2 + (pu - u kappa)^2]
    with kappa = (x . c_h) / (D r^2): ADD plus the first-order rms term."""
    l, hg = _layer(1)
    H, G, dh = hg
    T, D = l["x"].shape
    n, r = O.normalised_input(l["x"], l["gamma"], 1e-6)
    g, u = n @ l["Wg"].T, n @ l["Wu"].T
    lin = np.zeros((H, l["Wg"].shape[0]))
    for h in range(H):
        cols = slice(h * dh, (h + 1) * dh)
        c = l["a"][:, cols] @ l["Wo"][:, cols].T
        p = l["gamma"] * c / r[:, None]
        kappa = np.sum(l["x"] * c, axis=1) / (D * r * r)
        dg = p @ l["Wg"].T - g * kappa[:, None]
        du = p @ l["Wu"].T - u * kappa[:, None]
        lin[h] = np.mean(dg * dg + du * du, axis=0)
    l["a"] = l["a"] * s
    _, loo = _up(l, hg, "loo")
    np.testing.assert_allclose(loo / (s * s), lin, rtol=200 * s)
    _, add = _up(l, hg, "add")
    assert np.max(np.abs(loo / add - 1)) > 1e-2       # the rms term is first order, not negligible here


def test_removing_the_whole_residual_leaves_the_full_preactivation_energy():
    """One head whose write is the entire residual: without it the FFN input is
    zero, so LOO = E_t[g_k^2 + u_k^2]."""
    l, _ = _layer(2, H=1, G=1, dh=16)
    l["x"] = l["a"] @ l["Wo"].T
    _, loo = _up(l, (1, 1, 16), "loo")
    n, _ = O.normalised_input(l["x"], l["gamma"], 1e-6)
    g, u = n @ l["Wg"].T, n @ l["Wu"].T
    np.testing.assert_allclose(loo[0], np.mean(g * g + u * u, axis=0), rtol=1e-12)


def test_loo_is_invariant_to_scaling_the_residual_and_the_heads_together():
    l, hg = _layer(3)
    _, ref = _up(l, hg, "loo", eps=0.0)
    l["a"], l["x"] = 3.7 * l["a"], 3.7 * l["x"]
    _, got = _up(l, hg, "loo", eps=0.0)
    np.testing.assert_allclose(got, ref, rtol=1e-11)


def test_loo_group_sum_blocking_and_neuron_subsets():
    l, hg = _layer(4)
    S, Sh = _up(l, hg, "loo")
    S2, _ = _up(l, hg, "loo", token_block=5)
    np.testing.assert_allclose(S2, S, rtol=1e-12)
    np.testing.assert_allclose(Sh.reshape(2, 2, -1).sum(1), S, rtol=1e-13)
    idx = np.array([3, 17, 39])
    Ss, _ = _up(l, hg, "loo", neurons=idx)
    np.testing.assert_allclose(Ss, S[:, idx], rtol=1e-12)
    # it is a different score from ADD once the heads are not small
    _, add = _up(l, hg, "add")
    assert np.max(np.abs(Sh / add - 1)) > 1e-2
