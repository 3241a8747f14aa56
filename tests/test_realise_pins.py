"""Pins of the layer-forward oracle used to check layout realisation
("Affinity-Aware Sharding for Delayed Tensor Parallelism", §3 "The layout as
a free variable"; §2 for the Megatron split): rotary and attention special
cases, the dense function unchanged by any balanced layout, and the L-device
split summing to the dense layer."""
import numpy as np
import pytest

from oracle import layer_forward as LF
from oracle import partitions as P


def _weights(rng, D, H, G, dh, I, qk_norm=True):
    w = {"g_attn": 1 + 0.1 * rng.standard_normal(D), "g_ffn": 1 + 0.1 * rng.standard_normal(D),
         "Wq": 0.1 * rng.standard_normal((H * dh, D)), "Wk": 0.1 * rng.standard_normal((G * dh, D)),
         "Wv": 0.1 * rng.standard_normal((G * dh, D)), "Wo": 0.1 * rng.standard_normal((D, H * dh)),
         "Wg": 0.1 * rng.standard_normal((I, D)), "Wu": 0.1 * rng.standard_normal((I, D)),
         "Wd": 0.1 * rng.standard_normal((D, I))}
    if qk_norm:
        w["qn"] = 1 + 0.1 * rng.standard_normal(dh)
        w["kn"] = 1 + 0.1 * rng.standard_normal(dh)
    return w


def test_rope_is_a_rotation_with_relative_phase():
    rng = np.random.default_rng(0)
    T, d = 9, 8
    v = rng.standard_normal(d)
    x = np.tile(v, (T, 1, 1))
    r = LF.rope(x)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(v), rtol=1e-13)
    # <R_t v, R_s v> depends on t - s only
    dots = r[:, 0, :] @ r[:, 0, :].T
    for lag in range(1, 4):
        np.testing.assert_allclose(np.diag(dots, lag), dots[0, lag], rtol=1e-12)
    np.testing.assert_allclose(r[0, 0], v, rtol=0, atol=0)   # position 0 is the identity


def test_single_token_attention_returns_its_value():
    rng = np.random.default_rng(1)
    D, H, G, dh = 16, 4, 2, 8
    w = _weights(rng, D, H, G, dh, 8, qk_norm=False)
    x = rng.standard_normal((1, D))
    out = LF.attention_heads(x, w, H, G, dh)
    v = (LF.rmsnorm(x, w["g_attn"]) @ w["Wv"].T).reshape(1, G, dh)
    for h in range(H):
        np.testing.assert_allclose(out[0, h], v[0, h // (H // G)], rtol=1e-13)


@pytest.mark.parametrize("L,seed", [(2, 2), (4, 3)])
def test_any_balanced_layout_keeps_the_dense_function(L, seed):
    rng = np.random.default_rng(seed)
    T, D, H, G, dh, I = 12, 32, 8, 4, 8, 64
    w = _weights(rng, D, H, G, dh, I)
    x = rng.standard_normal((T, D))
    ref = LF.layer_forward(x, w, H, G, dh)
    h = rng.permutation(P.contiguous_heads(G, L))
    nu = rng.permutation(P.contiguous_neurons(I, L))
    wp, go, ho, no = LF.realise(w, h, nu, H, G, dh, L)
    np.testing.assert_allclose(LF.layer_forward(x, wp, H, G, dh), ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(LF.sharded_forward(x, wp, H, G, dh, L), ref, rtol=1e-12, atol=1e-12)
    # device l's shard holds exactly its groups (with their heads) and its neurons
    for l in range(L):
        assert set(go[l * G // L:(l + 1) * G // L]) == set(np.nonzero(h == l)[0])
        assert set(no[l * I // L:(l + 1) * I // L]) == set(np.nonzero(nu == l)[0])
        assert set(ho[l * H // L:(l + 1) * H // L]) == {hh for g in np.nonzero(h == l)[0]
                                                         for hh in range(g * H // G, (g + 1) * H // G)}


def test_a_mismatched_permutation_changes_the_function():
    """Permuting Wo's head blocks differently from Wq's breaks equivalence,
    so the check above can fail."""
    rng = np.random.default_rng(4)
    T, D, H, G, dh, I, L = 8, 16, 4, 2, 8, 16, 2
    w = _weights(rng, D, H, G, dh, I)
    x = rng.standard_normal((T, D))
    wp, _, _, _ = LF.realise(w, np.array([1, 0]), np.arange(I) // (I // L), H, G, dh, L)
    bad = dict(wp)
    bad["Wo"] = w["Wo"]
    assert np.max(np.abs(LF.layer_forward(x, bad, H, G, dh) - LF.layer_forward(x, w, H, G, dh))) > 1e-3


def test_attention_is_causal():
    """Changing later tokens leaves every earlier token's attention output unchanged."""
    rng = np.random.default_rng(5)
    T, D, H, G, dh = 7, 16, 4, 2, 8
    w = _weights(rng, D, H, G, dh, 8)
    x = rng.standard_normal((T, D))
    y = x.copy()
    y[4:] = rng.standard_normal((T - 4, D))
    a, b = LF.attention_heads(x, w, H, G, dh), LF.attention_heads(y, w, H, G, dh)
    np.testing.assert_allclose(a[:4], b[:4], rtol=1e-14, atol=1e-14)
    assert np.max(np.abs(a[4:] - b[4:])) > 1e-3


def test_equal_scores_average_the_causal_prefix():
    """With W_q = 0 every score is 0, so each token's output is the mean of the values
    of the tokens up to it (its KV group's values)."""
    rng = np.random.default_rng(6)
    T, D, H, G, dh = 6, 16, 4, 2, 8
    w = _weights(rng, D, H, G, dh, 8)
    w["Wq"] = np.zeros_like(w["Wq"])
    x = rng.standard_normal((T, D))
    out = LF.attention_heads(x, w, H, G, dh)
    v = (LF.rmsnorm(x, w["g_attn"]) @ w["Wv"].T).reshape(T, G, dh)
    for h in range(H):
        g = h // (H // G)
        for t in range(T):
            np.testing.assert_allclose(out[t, h], v[:t + 1, g].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_attention_against_scalar_loops():
    """Grouped-query causal softmax attention, written out with scalar loops on a tiny
    layer (no q/k norms): scores q.k / sqrt(d), masked above the diagonal, softmax over
    the keys, the values of query head h's KV group h // (H / G)."""
    import math
    rng = np.random.default_rng(7)
    T, D, H, G, dh = 5, 6, 4, 2, 4
    w = _weights(rng, D, H, G, dh, 8, qk_norm=False)
    x = rng.standard_normal((T, D))
    z = LF.rmsnorm(x, w["g_attn"])
    q = LF.rope((z @ w["Wq"].T).reshape(T, H, dh))
    k = LF.rope((z @ w["Wk"].T).reshape(T, G, dh))
    v = (z @ w["Wv"].T).reshape(T, G, dh)
    out = LF.attention_heads(x, w, H, G, dh)
    for h in range(H):
        g = h // (H // G)
        for t in range(T):
            sc = [sum(q[t, h, i] * k[s, g, i] for i in range(dh)) / math.sqrt(dh) for s in range(t + 1)]
            m = max(sc)
            e = [math.exp(c - m) for c in sc]
            tot = sum(e)
            for i in range(dh):
                ref = sum(e[s] / tot * v[s, g, i] for s in range(t + 1))
                assert abs(out[t, h, i] - ref) <= 1e-12 * (1 + abs(ref))


def test_ffn_against_scalar_loops():
    """With W_o = 0 the attention adds nothing, and the layer is x + FFN(rmsnorm(x) g):
    SwiGLU written out with scalar loops, rms over the row with eps = 1e-6."""
    import math
    rng = np.random.default_rng(8)
    T, D, H, G, dh, I = 3, 5, 2, 1, 4, 6
    w = _weights(rng, D, H, G, dh, I, qk_norm=False)
    w["Wo"] = np.zeros_like(w["Wo"])
    x = rng.standard_normal((T, D))
    y = LF.layer_forward(x, w, H, G, dh)
    for t in range(T):
        r = math.sqrt(sum(x[t, d] ** 2 for d in range(D)) / D + 1e-6)
        z = [x[t, d] / r * w["g_ffn"][d] for d in range(D)]
        act = []
        for i in range(I):
            gi = sum(z[d] * w["Wg"][i, d] for d in range(D))
            ui = sum(z[d] * w["Wu"][i, d] for d in range(D))
            act.append(gi / (1.0 + math.exp(-gi)) * ui)
        for j in range(D):
            ref = x[t, j] + sum(act[i] * w["Wd"][j, i] for i in range(I))
            assert abs(y[t, j] - ref) <= 1e-12 * (1 + abs(ref))
