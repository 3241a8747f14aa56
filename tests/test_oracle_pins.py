"""Pins for the fp64 oracle: each test checks it against something other than
itself -- a finite difference, an explicit scalar loop, a closed form, an
exact invariance, or a value the paper prints.  CPU only.

Paper: "Affinity-Aware Sharding for Delayed Tensor Parallelism", §3
("Affinity scores", eq. 5; "Objective", eq. 6; "Optimiser").
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import affinity_oracle as O
from oracle import partitions as P

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "paper_values.json")))


def _layer(rng, T=5, D=6, H=4, G=2, dh=3, I=7, scale=0.4):
    return dict(
        a=rng.normal(0, 1, (T, H * dh)), x=rng.normal(0, 1, (T, D)),
        Wo=rng.normal(0, scale, (D, H * dh)), gamma=1 + rng.normal(0, 0.1, D),
        Wg=rng.normal(0, scale, (I, D)), Wu=rng.normal(0, scale, (I, D)),
        Wd=rng.normal(0, scale, (D, I)),
        gamma_next=1 + rng.normal(0, 0.1, D), Wq_next=rng.normal(0, scale, (H * dh, D)),
        Wk_next=rng.normal(0, scale, (G * dh, D)), Wv_next=rng.normal(0, scale, (G * dh, D)),
        H=H, G=G, dh=dh)


def _up(L, mode, eps=1e-6, **kw):
    return O.s_up(L["a"], L["x"], L["Wo"], L["gamma"], L["Wg"], L["Wu"], L["Wd"],
                  L["H"], L["G"], L["dh"], eps, mode, **kw)


def _down(L, eps=1e-6, **kw):
    return O.s_down(L["x"], L["gamma"], L["Wg"], L["Wu"], L["Wd"], L["gamma_next"],
                    L["Wq_next"], L["Wk_next"], L["Wv_next"], L["H"], L["G"], L["dh"], eps, **kw)


def _msilu(z):
    return z / (1.0 + math.exp(-z)) if z > -700 else 0.0


def _msig(z):
    return 1.0 / (1.0 + math.exp(-z))


# ---------------------------------------------------------------- elementwise

def test_sigmoid_against_tanh_form():
    z = np.linspace(-15, 15, 2001)        # tanh form loses digits for very negative z
    ref = 0.5 * (1.0 + np.tanh(z / 2.0))
    np.testing.assert_allclose(O.sigmoid(z), ref, rtol=1e-9)
    zn = np.linspace(-700, -15, 500)         # sigmoid(z) (1 + e^-z) = 1
    np.testing.assert_allclose(O.sigmoid(zn) * (1.0 + np.exp(-zn)), 1.0, rtol=1e-14)
    assert O.sigmoid(np.array([0.0]))[0] == 0.5
    big = O.sigmoid(np.array([-800.0, 800.0]))
    assert big[0] == 0.0 and big[1] == 1.0


def test_silu_prime_is_derivative_of_silu():
    z = np.linspace(-12, 12, 241)
    h = 1e-5
    fd = np.array([(_msilu(v + h) - _msilu(v - h)) / (2 * h) for v in z])
    np.testing.assert_allclose(O.silu_prime(z), fd, rtol=1e-8, atol=1e-10)
    assert O.silu_prime(np.array([0.0]))[0] == 0.5
    np.testing.assert_allclose(O.silu(z), [_msilu(v) for v in z], rtol=1e-14)


def test_rms_closed_form():
    eps = 1e-6
    assert O.rms(np.array([[3.0, 4.0]]), eps)[0] == pytest.approx(math.sqrt(12.5 + eps), rel=1e-15)
    assert O.rms(np.full((1, 64), -2.5), 0.0)[0] == pytest.approx(2.5, rel=1e-15)


# ---------------------------------------------------------------- head pieces / eq. 5

def test_head_pieces_sum_to_normalised_input():
    """With x = sum_h a_h W_o^(h) (no other writer), sum_h p_h equals the
    normalised input gamma*x/r.  x is built with one full matmul a @ Wo^T."""
    rng = np.random.default_rng(1)
    L = _layer(rng, T=6, D=9, H=6, G=3, dh=4)
    x = L["a"] @ L["Wo"].T
    n, r = O.normalised_input(x, L["gamma"], 1e-6)
    p = O.head_pieces(L["a"], L["Wo"], L["gamma"], r, L["H"], L["dh"])
    np.testing.assert_allclose(p.sum(axis=1), n, rtol=1e-12, atol=1e-14)


def test_delta_is_first_order_removal_of_head_piece():
    """Delta_hk (eq. 5) = -d/deps of silu(g_k(eps)) u_k(eps) at eps = 0, where
    eps of head h's write a_h W_o^(h) is taken out of x with r held fixed.
    Computed here by central differences from scratch (scalar math)."""
    rng = np.random.default_rng(2)
    L = _layer(rng, T=4, D=6, H=4, G=2, dh=3, I=5, scale=0.5)
    eps_rms, e = 1e-6, 1e-5
    D_or = O.delta(L["a"], L["x"], L["Wo"], L["gamma"], L["Wg"], L["Wu"], L["H"], L["dh"], eps_rms)
    T, H, dh, I = 4, 4, 3, 5
    for t in range(T):
        r = math.sqrt(sum(v * v for v in L["x"][t]) / 6 + eps_rms)
        for h in range(H):
            c = L["a"][t, h * dh:(h + 1) * dh] @ L["Wo"][:, h * dh:(h + 1) * dh].T   # head h's write
            for k in range(I):
                def f(s):
                    n = L["gamma"] * (L["x"][t] - s * c) / r
                    return _msilu(float(n @ L["Wg"][k])) * float(n @ L["Wu"][k])
                fd = (f(-e) - f(e)) / (2 * e)
                assert D_or[t, h, k] == pytest.approx(fd, rel=2e-7, abs=1e-11)


def test_single_head_homogeneity():
    """H = G = 1 and x = a W_o: the head piece is the whole normalised input,
    so g = p.w^g, u = p.w^u and Delta = d/ds [silu(s g) (s u)] at s = 1."""
    rng = np.random.default_rng(3)
    T, D, dh, I = 5, 7, 7, 6
    a = rng.normal(0, 1, (T, dh))
    Wo = rng.normal(0, 0.5, (D, dh))
    gamma = 1 + rng.normal(0, 0.1, D)
    Wg, Wu = rng.normal(0, 0.5, (I, D)), rng.normal(0, 0.5, (I, D))
    x = a @ Wo.T
    Dl = O.delta(a, x, Wo, gamma, Wg, Wu, 1, dh, 1e-6)
    for t in range(T):
        r = math.sqrt(float(x[t] @ x[t]) / D + 1e-6)
        n = gamma * x[t] / r
        for k in range(I):
            g, u = float(n @ Wg[k]), float(n @ Wu[k])
            h = 1e-5
            fd = ((_msilu((1 + h) * g) * (1 + h) * u) - (_msilu((1 - h) * g) * (1 - h) * u)) / (2 * h)
            assert Dl[t, 0, k] == pytest.approx(fd, rel=1e-7, abs=1e-12)


# ---------------------------------------------------------------- explicit loops

def _loops_up(L, mode, eps):
    a, x, Wo, gm, Wg, Wu, Wd = (L[k] for k in ("a", "x", "Wo", "gamma", "Wg", "Wu", "Wd"))
    H, G, dh = L["H"], L["G"], L["dh"]
    T, D = x.shape
    I = Wg.shape[0]
    S_head = [[0.0] * I for _ in range(H)]
    for t in range(T):
        r = math.sqrt(sum(x[t, d] ** 2 for d in range(D)) / D + eps)
        n = [gm[d] * x[t, d] / r for d in range(D)]
        for h in range(H):
            p = [gm[d] * sum(a[t, h * dh + j] * Wo[d, h * dh + j] for j in range(dh)) / r for d in range(D)]
            for k in range(I):
                g = sum(n[d] * Wg[k, d] for d in range(D))
                u = sum(n[d] * Wu[k, d] for d in range(D))
                pg = sum(p[d] * Wg[k, d] for d in range(D))
                pu = sum(p[d] * Wu[k, d] for d in range(D))
                if mode == "fo":
                    s = _msig(g)
                    dl = s * (1 + g * (1 - s)) * u * pg + g * s * pu
                    S_head[h][k] += dl * dl / T
                else:
                    S_head[h][k] += (pg * pg + pu * pu) / T
    if mode == "fo":
        for h in range(H):
            for k in range(I):
                S_head[h][k] *= sum(Wd[d, k] ** 2 for d in range(D))
    hpg = H // G
    S = [[sum(S_head[h][k] for h in range(g * hpg, (g + 1) * hpg)) for k in range(I)] for g in range(G)]
    return np.array(S), np.array(S_head)


@pytest.mark.parametrize("mode", ["fo", "add"])
def test_s_up_matches_scalar_loops(mode):
    rng = np.random.default_rng(4)
    L = _layer(rng, T=3, D=4, H=4, G=2, dh=2, I=3, scale=0.6)
    S, Sh = _up(L, mode, token_block=2)
    S_ref, Sh_ref = _loops_up(L, mode, 1e-6)
    np.testing.assert_allclose(S, S_ref, rtol=1e-12)
    np.testing.assert_allclose(Sh, Sh_ref, rtol=1e-12)


def test_add_equals_quadratic_forms_of_the_second_moment():
    """ADD per head is a mean of squared linear forms in a_h/r, so it equals
    m^T E_t[(a_h/r)(a_h/r)^T] m with m = W_o^(h)^T diag(gamma) w for every gate and
    up row w (the form the GPU evaluates by default).  Built here from the
    second moment of each head's slice of a and the folded rows, with no per-token
    p_h; the oracle forms p_h per token."""
    rng = np.random.default_rng(12)
    L = _layer(rng, T=40, D=10, H=4, G=2, dh=5, I=9)
    eps = 1e-6
    S, Sh = _up(L, "add", eps=eps)
    a, x, Wo, gm, Wg, Wu = (L[k] for k in ("a", "x", "Wo", "gamma", "Wg", "Wu"))
    H, G, dh = L["H"], L["G"], L["dh"]
    T = x.shape[0]
    r = np.sqrt((x * x).mean(axis=1) + eps)
    Sh_ref = np.zeros_like(Sh)
    for h in range(H):
        at = a[:, h * dh:(h + 1) * dh] / r[:, None]
        C = at.T @ at / T                                   # d_head x d_head second moment
        Woh = Wo[:, h * dh:(h + 1) * dh]                    # D x d_head
        for Wrow in (Wg, Wu):
            M = Wrow @ (gm[:, None] * Woh)                  # I x d_head folded rows
            Sh_ref[h] += np.einsum("ki,ij,kj->k", M, C, M)
    np.testing.assert_allclose(Sh, Sh_ref, rtol=1e-12)
    np.testing.assert_allclose(S, Sh_ref.reshape(G, H // G, -1).sum(1), rtol=1e-12)
    # and the second moment is positive semi-definite, so every entry is >= 0
    assert np.all(Sh >= 0)


def test_s_down_matches_scalar_loops():
    rng = np.random.default_rng(5)
    L = _layer(rng, T=3, D=4, H=4, G=2, dh=2, I=3, scale=0.6)
    eps = 1e-6
    x, gm, Wg, Wu, Wd = L["x"], L["gamma"], L["Wg"], L["Wu"], L["Wd"]
    gp, Wq, Wk, Wv = L["gamma_next"], L["Wq_next"], L["Wk_next"], L["Wv_next"]
    T, D = x.shape
    I, H, G, dh = 3, 4, 2, 2
    c = [0.0] * I
    for t in range(T):
        r = math.sqrt(sum(v * v for v in x[t]) / D + eps)
        n = [gm[d] * x[t, d] / r for d in range(D)]
        al = [_msilu(sum(n[d] * Wg[k, d] for d in range(D))) * sum(n[d] * Wu[k, d] for d in range(D))
              for k in range(I)]
        xp = [x[t, d] + sum(al[k] * Wd[d, k] for k in range(I)) for d in range(D)]
        rp = math.sqrt(sum(v * v for v in xp) / D + eps)
        for k in range(I):
            c[k] += al[k] ** 2 / rp ** 2 / T
    ref = np.zeros((I, G))
    for k in range(I):
        for g in range(G):
            rows = [Wq[(g * (H // G)) * dh + i] for i in range((H // G) * dh)] + \
                   [Wk[g * dh + i] for i in range(dh)] + [Wv[g * dh + i] for i in range(dh)]
            b2 = sum(sum(row[d] * gp[d] * Wd[d, k] for d in range(D)) ** 2 for row in rows)
            ref[k, g] = c[k] * b2
    np.testing.assert_allclose(_down(L, token_block=2), ref, rtol=1e-12)


# ---------------------------------------------------------------- exact laws

def test_scaling_laws():
    rng = np.random.default_rng(6)
    L = _layer(rng, T=8, D=6, H=4, G=2, dh=3, I=5)
    c = 1.7
    fo, _ = _up(L, "fo", eps=0.0)
    ad, _ = _up(L, "add", eps=0.0)

    def up(mode, **chg):
        return _up(dict(L, **chg), mode, eps=0.0)[0]

    np.testing.assert_allclose(up("fo", a=c * L["a"]), c * c * fo, rtol=1e-12)
    np.testing.assert_allclose(up("add", a=c * L["a"]), c * c * ad, rtol=1e-12)
    np.testing.assert_allclose(up("fo", Wd=c * L["Wd"]), c * c * fo, rtol=1e-12)
    np.testing.assert_allclose(up("add", Wd=c * L["Wd"]), ad, rtol=1e-12)
    np.testing.assert_allclose(up("fo", x=c * L["x"]), fo / (c * c), rtol=1e-12)
    np.testing.assert_allclose(up("add", x=c * L["x"]), ad / (c * c), rtol=1e-12)
    np.testing.assert_allclose(up("add", gamma=c * L["gamma"]), c * c * ad, rtol=1e-12)
    # S_down: scaling the next layer's q/k/v rows scales ||b||^2 by c^2
    dn = _down(L, eps=0.0)
    dn2 = _down(dict(L, Wq_next=c * L["Wq_next"], Wk_next=c * L["Wk_next"], Wv_next=c * L["Wv_next"]), eps=0.0)
    np.testing.assert_allclose(dn2, c * c * dn, rtol=1e-12)


def test_permutation_equivariance():
    """Permuting neurons (rows of Wg/Wu, columns of Wd) permutes S_up's columns
    and S_down's rows; permuting KV groups (head blocks of a and Wo; q/k/v row
    blocks of the next layer) permutes S_up's rows and S_down's columns
    (§3 'The layout as a free variable')."""
    rng = np.random.default_rng(7)
    L = _layer(rng, T=6, D=5, H=6, G=3, dh=2, I=7)
    H, G, dh = 6, 3, 2
    pn = rng.permutation(7)
    Ln = dict(L, Wg=L["Wg"][pn], Wu=L["Wu"][pn], Wd=L["Wd"][:, pn])
    for mode in ("fo", "add"):
        np.testing.assert_allclose(_up(Ln, mode)[0], _up(L, mode)[0][:, pn], rtol=1e-12)
    np.testing.assert_allclose(_down(Ln), _down(L)[pn], rtol=1e-12)
    pg = rng.permutation(G)
    hpg = H // G
    head_order = np.concatenate([np.arange(g * hpg, (g + 1) * hpg) for g in pg])
    cols = np.concatenate([np.arange(h * dh, (h + 1) * dh) for h in head_order])
    Lg = dict(L, a=L["a"][:, cols], Wo=L["Wo"][:, cols])
    for mode in ("fo", "add"):
        np.testing.assert_allclose(_up(Lg, mode)[0], _up(L, mode)[0][pg], rtol=1e-12)
    kv = np.concatenate([np.arange(g * dh, (g + 1) * dh) for g in pg])
    Ld = dict(L, Wq_next=L["Wq_next"][cols], Wk_next=L["Wk_next"][kv], Wv_next=L["Wv_next"][kv])
    np.testing.assert_allclose(_down(Ld), _down(L)[:, pg], rtol=1e-12)


def test_group_sum_and_one_head_per_group():
    rng = np.random.default_rng(8)
    L = _layer(rng, T=5, D=5, H=6, G=2, dh=2, I=4)
    S, Sh = _up(L, "fo")
    np.testing.assert_allclose(S, Sh.reshape(2, 3, 4).sum(1), rtol=1e-14)
    S6, Sh6 = _up(dict(L, G=6), "fo")
    np.testing.assert_allclose(S6, Sh6, rtol=0)
    np.testing.assert_allclose(Sh6, Sh, rtol=1e-14)


def test_special_cases():
    rng = np.random.default_rng(9)
    L = _layer(rng, T=6, D=5, H=4, G=2, dh=2, I=4)
    S0, _ = _up(dict(L, Wu=np.zeros_like(L["Wu"])), "fo")
    assert np.all(S0 == 0.0)                                  # u = 0 and p.w^u = 0
    Sa, _ = _up(dict(L, Wu=np.zeros_like(L["Wu"])), "add")
    n, r = O.normalised_input(L["x"], L["gamma"], 1e-6)
    p = O.head_pieces(L["a"], L["Wo"], L["gamma"], r, 4, 2)
    gate_only = ((p @ L["Wg"].T) ** 2).mean(0)                # E_t[(p_h.w^g_k)^2]
    np.testing.assert_allclose(Sa, gate_only.reshape(2, 2, 4).sum(1), rtol=1e-12)
    for mode in ("fo", "add"):
        assert np.all(_up(dict(L, a=np.zeros_like(L["a"])), mode)[0] == 0.0)
    assert np.all(_up(dict(L, Wd=np.zeros_like(L["Wd"])), "fo")[0] == 0.0)
    # Wd = 0: x' = x, so c_k = E_t[alpha_k^2 / r^2]; and every b_gk = 0
    c = O.down_token_weights(L["x"], L["gamma"], L["Wg"], L["Wu"], np.zeros_like(L["Wd"]), 1e-6)
    alpha = O.silu(n @ L["Wg"].T) * (n @ L["Wu"].T)
    np.testing.assert_allclose(c, (alpha ** 2 / (r * r)[:, None]).mean(0), rtol=1e-13)
    assert np.all(_down(dict(L, Wd=np.zeros_like(L["Wd"]))) == 0.0)


def test_neuron_subset_and_token_blocking():
    rng = np.random.default_rng(10)
    L = _layer(rng, T=37, D=6, H=4, G=2, dh=3, I=9)
    idx = np.array([7, 0, 3])
    for mode in ("fo", "add"):
        full, _ = _up(L, mode, token_block=512)
        np.testing.assert_allclose(_up(L, mode, neurons=idx)[0], full[:, idx], rtol=1e-13)
        np.testing.assert_allclose(_up(L, mode, token_block=5)[0], full, rtol=1e-13)
    np.testing.assert_allclose(_down(L, neurons=idx, token_block=4), _down(L)[idx], rtol=1e-13)


# ---------------------------------------------------------------- partitions and J

def test_partition_count_matches_paper():
    gv = GOLDEN["partition_count"]
    assert P.partition_count(gv["G"], gv["L"]) == gv["count"]
    parts = P.balanced_partitions(gv["G"], gv["L"])
    assert len(parts) == gv["count"] == len(set(parts))


@pytest.mark.parametrize("G,L", [(2, 1), (2, 2), (4, 2), (6, 3), (6, 2), (8, 2), (8, 4)])
def test_partition_enumeration_brute_force(G, L):
    brute = P.all_balanced_maps(G, L)          # itertools.product is lexicographic
    assert P.balanced_partitions(G, L) == brute
    assert len(brute) == P.partition_count(G, L)


def test_score_partitions_brute_force():
    rng = np.random.default_rng(11)
    C = rng.random((8, 4))
    scores, best, assign = P.score_partitions(C)
    brute = [sum(C[g, m[g]] for g in range(8)) for m in P.all_balanced_maps(8, 4)]
    np.testing.assert_allclose(scores, brute, rtol=0, atol=0)
    assert best == int(np.argmax(brute)) and assign == P.all_balanced_maps(8, 4)[best]
    C2 = np.ones((4, 2))                       # all tied: the first (lexicographic) wins
    assert P.score_partitions(C2)[1] == 0


def _random_stack(rng, N, G, I):
    ups = [P.unit_mass(rng.random((G, I))) for _ in range(N)]
    downs = [P.unit_mass(rng.random((I, G))) for _ in range(N - 1)]
    return ups, downs


def test_random_layout_expectation_exact():
    """Averaged over every balanced layout, J = (2N-1)/L ('Objective')."""
    rng = np.random.default_rng(12)
    for N, G, I, L in [(2, 2, 2, 2), (3, 2, 4, 2), (2, 3, 3, 3)]:
        ups, downs = _random_stack(rng, N, G, I)
        hm, nm = P.all_balanced_maps(G, L), P.all_balanced_maps(I, L)
        import itertools
        tot, cnt = 0.0, 0
        for hs in itertools.product(hm, repeat=N):
            for ns in itertools.product(nm, repeat=N):
                J = P.objective_J(ups, downs, hs, ns)
                assert -1e-12 <= J <= 2 * N - 1 + 1e-12
                tot += J
                cnt += 1
        assert tot / cnt == pytest.approx((2 * N - 1) / L, rel=1e-12)


def test_random_layout_expectation_paper_values():
    for c in GOLDEN["random_layout_expectation"]["cases"]:
        assert 2 * c["N"] - 1 == c["edges"]
        assert (2 * c["N"] - 1) / c["L"] == c["expected_J"]


def test_single_device_scores_every_edge():
    rng = np.random.default_rng(13)
    ups, downs = _random_stack(rng, 3, 4, 6)
    J = P.objective_J(ups, downs, [np.zeros(4, int)] * 3, [np.zeros(6, int)] * 3)
    assert J == pytest.approx(5.0, rel=1e-14)


def test_group_gain_reproduces_J_differences():
    """Changing only h_i changes J by exactly the change of sum_g C[g, h_i(g)]."""
    rng = np.random.default_rng(14)
    N, G, I, L = 3, 4, 8, 2
    ups, downs = _random_stack(rng, N, G, I)
    hs = [np.array(P.contiguous_heads(G, L)) for _ in range(N)]
    ns = [rng.permutation(P.contiguous_neurons(I, L)) for _ in range(N)]
    for i in range(N):
        C = P.group_gain(ups[i], L, ns[i], downs[i - 1] if i else None, ns[i - 1] if i else None)
        parts = P.balanced_partitions(G, L)
        base_h = list(hs)
        Js, Cs = [], []
        for p in parts:
            base_h[i] = np.array(p)
            Js.append(P.objective_J(ups, downs, base_h, ns))
            Cs.append(sum(C[g, p[g]] for g in range(G)))
        np.testing.assert_allclose(np.array(Js) - Js[0], np.array(Cs) - Cs[0], atol=1e-13)
