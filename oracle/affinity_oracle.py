"""fp64 CPU oracle for the head/neuron affinity scores S_up and S_down.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The library never calls it, and it shares no code with the CUDA path.

Source: "Affinity-Aware Sharding for Delayed Tensor Parallelism" (de Reynal,
2026), §3 "Method: affinity-aware layouts", paragraph "Affinity scores",
equation (5), and the two sentences after it that define the FO score, the
ADD score and S_down.  Both the first-page text rendering and the arXiv HTML
rendering of the paper were read; the latter gives the inline formulas
cleanly but drops the display of eq. (5), which the former keeps.

Everything is written the way the paper states it, in float64, with no
algebraic refolding: the head piece p_h is formed explicitly in R^D for
every token before it is dotted with a neuron's gate/up row.  The only
liberty taken is that the token average E_t is accumulated over blocks of
tokens (a loop over t), which changes the rounding order and nothing else.

Readings of points the paper leaves open:
  * r = rms(x) = sqrt(mean_d x_d^2 + eps) with eps an explicit argument.
  * Head h belongs to KV group floor(h / (H/G)) (contiguous, the usual
    grouped-query order); both FO and ADD are summed over a group's heads.
  * E_t is the plain mean over all T tokens.
  * For S_down, r' is the rms of the residual after this FFN,
    x' = x + sum_k alpha_k w^d_k, with the same eps; W^qkv_g stacks the
    query rows of g's heads, then g's key rows, then g's value rows.

Array layout (PyTorch nn.Linear storage):
  a [T, H*dh], x [T, D], Wo [D, H*dh], gamma [D], Wg/Wu [I, D], Wd [D, I],
  gamma_next [D], Wq_next [H*dh, D], Wk_next/Wv_next [G*dh, D].
"""
from __future__ import annotations

import numpy as np

F = np.float64


def rms(x: np.ndarray, eps: float) -> np.ndarray:
    """r = rms(x) over the last axis ("Affinity scores": r = rms(x))."""
    x = np.asarray(x, F)
    return np.sqrt(np.mean(x * x, axis=-1) + eps)


def sigmoid(z: np.ndarray) -> np.ndarray:
    """Logistic function 1 / (1 + e^-z), evaluated without overflow."""
    z = np.asarray(z, F)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    e = np.exp(z[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z), the SwiGLU gate nonlinearity."""
    z = np.asarray(z, F)
    return z * sigmoid(z)


def silu_prime(z: np.ndarray) -> np.ndarray:
    """d silu / dz = s + z s (1 - s) with s = sigmoid(z)."""
    z = np.asarray(z, F)
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def normalised_input(x: np.ndarray, gamma: np.ndarray, eps: float):
    """The FFN's normalised input n = gamma * x / r and r = rms(x) ("Affinity scores")."""
    x = np.asarray(x, F)
    r = rms(x, eps)
    return np.asarray(gamma, F) * x / r[:, None], r


def head_pieces(a: np.ndarray, Wo: np.ndarray, gamma: np.ndarray, r: np.ndarray,
                H: int, dh: int) -> np.ndarray:
    """p_h = gamma * (a_h W_o^(h)) / r for every token and head -> [T, H, D].

    ("Affinity scores": the normalised FFN input decomposes over heads as
    sum_h p_h + rest.)  W_o^(h) is head h's slice of the output projection:
    with Wo stored [D, H*dh], (a_h W_o^(h))_d = sum_j a[t, h*dh + j] * Wo[d, h*dh + j].
    """
    a = np.asarray(a, F)
    Wo = np.asarray(Wo, F)
    gamma = np.asarray(gamma, F)
    T = a.shape[0]
    D = Wo.shape[0]
    p = np.empty((T, H, D), F)
    for h in range(H):
        cols = slice(h * dh, (h + 1) * dh)
        p[:, h, :] = gamma * (a[:, cols] @ Wo[:, cols].T) / r[:, None]
    return p


def delta(a, x, Wo, gamma, Wg, Wu, H, dh, eps, neurons=None) -> np.ndarray:
    """Eq. (5): Delta_hk = silu'(g_k) u_k (p_h . w^g_k) + silu(g_k) (p_h . w^u_k).

    The first-order change of neuron k's output silu(g_k) u_k when head h's
    piece p_h is removed from its pre-activations (the rms held fixed).
    Returns [T, H, K] for the selected neurons (all by default).  Meant for
    small inputs: it materialises every (t, h, k) value.
    """
    Wg = np.asarray(Wg, F)
    Wu = np.asarray(Wu, F)
    if neurons is not None:
        Wg, Wu = Wg[neurons], Wu[neurons]
    n, r = normalised_input(x, gamma, eps)
    g = n @ Wg.T                      # g_k = n . w^g_k
    u = n @ Wu.T                      # u_k = n . w^u_k
    p = head_pieces(a, Wo, gamma, r, H, dh)
    pg = p @ Wg.T                     # p_h . w^g_k   [T, H, K]
    pu = p @ Wu.T                     # p_h . w^u_k
    return silu_prime(g)[:, None, :] * u[:, None, :] * pg + silu(g)[:, None, :] * pu


def group_of_head(H: int, G: int) -> np.ndarray:
    """KV group of each query head: contiguous blocks of H/G heads."""
    if H % G:
        raise ValueError("H must be a multiple of G")
    return np.arange(H) // (H // G)


def sum_over_groups(S_head: np.ndarray, H: int, G: int) -> np.ndarray:
    """S_up[g, k] = sum over the query heads h of KV group g of S_head[h, k]."""
    grp = group_of_head(H, G)
    out = np.zeros((G,) + S_head.shape[1:], F)
    for h in range(H):
        out[grp[h]] += S_head[h]
    return out


def s_up(a, x, Wo, gamma, Wg, Wu, Wd, H, G, dh, eps, mode="fo", neurons=None,
         token_block=512):
    """S_up for one layer, FO, ADD or LOO ("Affinity scores" paragraph of §3).

    FO:  S_hk = E_t[Delta_hk^2] * ||w^d_k||^2 (eq. 5 for Delta; w^d_k the
         down-projection column), then summed over each KV group's heads.
    ADD: S_hk = E_t[(p_h . w^g_k)^2 + (p_h . w^u_k)^2], summed likewise.
    LOO: the exact leave-one-out change of the pre-activations,
         S_hk = E_t[(g_k - g_k^(-h))^2 + (u_k - u_k^(-h))^2], where g^(-h),
         u^(-h) are recomputed from the residual with head h's write
         c_h = a_h W_o^(h) removed, x - c_h, including its new rms (the
         paper's ablation score that differs from ADD only by the rms change).

    ``neurons`` restricts the columns (the definition evaluated for those k
    only).  Returns (S_up [G, K], S_head [H, K]).
    """
    if mode not in ("fo", "add", "loo"):
        raise ValueError(mode)
    a = np.asarray(a, F)
    x = np.asarray(x, F)
    Wg = np.asarray(Wg, F)
    Wu = np.asarray(Wu, F)
    Wd = np.asarray(Wd, F)
    if neurons is not None:
        Wg, Wu, Wd = Wg[neurons], Wu[neurons], Wd[:, neurons]
    T = x.shape[0]
    K = Wg.shape[0]
    acc = np.zeros((H, K), F)
    Wo_ = np.asarray(Wo, F)
    for t0 in range(0, T, token_block):
        ts = slice(t0, min(T, t0 + token_block))
        n, r = normalised_input(x[ts], gamma, eps)
        if mode == "loo":
            g = n @ Wg.T
            u = n @ Wu.T
            for h in range(H):
                cols = slice(h * dh, (h + 1) * dh)
                c = a[ts, cols] @ Wo_[:, cols].T              # head h's write into the residual
                n_rm, _ = normalised_input(x[ts] - c, gamma, eps)
                dg = g - n_rm @ Wg.T
                du = u - n_rm @ Wu.T
                acc[h] += np.sum(dg * dg + du * du, axis=0)
            continue
        p = head_pieces(a[ts], Wo, gamma, r, H, dh)       # [Tb, H, D]
        pg = p @ Wg.T                                      # [Tb, H, K]
        pu = p @ Wu.T
        if mode == "fo":
            g = n @ Wg.T
            u = n @ Wu.T
            d = silu_prime(g)[:, None, :] * u[:, None, :] * pg + silu(g)[:, None, :] * pu
            acc += np.sum(d * d, axis=0)
        else:
            acc += np.sum(pg * pg + pu * pu, axis=0)
    S_head = acc / T
    if mode == "fo":
        S_head = S_head * np.sum(Wd * Wd, axis=0)[None, :]   # ||w^d_k||^2
    return sum_over_groups(S_head, H, G), S_head


def qkv_rows_of_group(Wq_next, Wk_next, Wv_next, H, G, dh, g) -> np.ndarray:
    """W^qkv_g: the next layer's query rows of g's heads, then g's key and value rows."""
    hpg = H // G
    q = np.asarray(Wq_next, F)[g * hpg * dh:(g + 1) * hpg * dh]
    k = np.asarray(Wk_next, F)[g * dh:(g + 1) * dh]
    v = np.asarray(Wv_next, F)[g * dh:(g + 1) * dh]
    return np.concatenate([q, k, v], axis=0)


def down_write_norms(Wd, gamma_next, Wq_next, Wk_next, Wv_next, H, G, dh, neurons=None):
    """||b_gk||^2 with b_gk = W^qkv_g (gamma' * w^d_k) ("Affinity scores", down edge).

    Returns [K, G].
    """
    Wd = np.asarray(Wd, F)
    if neurons is not None:
        Wd = Wd[:, neurons]
    gw = np.asarray(gamma_next, F)[:, None] * Wd            # gamma' * w^d_k, [D, K]
    out = np.empty((Wd.shape[1], G), F)
    for g in range(G):
        b = qkv_rows_of_group(Wq_next, Wk_next, Wv_next, H, G, dh, g) @ gw   # [rows, K]
        out[:, g] = np.sum(b * b, axis=0)
    return out


def down_token_weights(x, gamma, Wg, Wu, Wd, eps, neurons=None, token_block=512):
    """c_k = E_t[alpha_k^2 / r'^2] ("Affinity scores", down edge).

    alpha_k = silu(g_k) u_k is neuron k's activation; r' = rms(x') is the
    next layer's pre-norm rms, x' = x + sum_k alpha_k w^d_k (all neurons).
    Returns [K] for the selected neurons.
    """
    x = np.asarray(x, F)
    Wg = np.asarray(Wg, F)
    Wu = np.asarray(Wu, F)
    Wd = np.asarray(Wd, F)
    T = x.shape[0]
    sel = np.arange(Wg.shape[0]) if neurons is None else np.asarray(neurons)
    acc = np.zeros(len(sel), F)
    for t0 in range(0, T, token_block):
        ts = slice(t0, min(T, t0 + token_block))
        n, _ = normalised_input(x[ts], gamma, eps)
        alpha = silu(n @ Wg.T) * (n @ Wu.T)                  # [Tb, I]
        xp = x[ts] + alpha @ Wd.T                             # x' = x + sum_k alpha_k w^d_k
        rp = rms(xp, eps)
        acc += np.sum(alpha[:, sel] ** 2 / (rp * rp)[:, None], axis=0)
    return acc / T


def s_down(x, gamma, Wg, Wu, Wd, gamma_next, Wq_next, Wk_next, Wv_next, H, G, dh, eps,
           neurons=None, token_block=512):
    """S_down[k, g] = E_t[alpha_k^2 / r'^2] * ||b_gk||^2 ("Affinity scores", down edge).

    Returns [K, G].
    """
    c = down_token_weights(x, gamma, Wg, Wu, Wd, eps, neurons, token_block)
    b2 = down_write_norms(Wd, gamma_next, Wq_next, Wk_next, Wv_next, H, G, dh, neurons)
    return c[:, None] * b2
