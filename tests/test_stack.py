"""The 28-layer Qwen3-shaped stack: S_up (FO) of every layer and S_down of
every layer but the last on the GPU, then unit mass, contiguous neuron maps,
the best of the 2520 balanced KV-group partitions per layer and the objective
J ("Affinity-Aware Sharding for Delayed Tensor Parallelism", §3 "Objective",
equation (6), "Optimiser").  The host sequence is checked against the oracle
on CPU; the GPU run adds matrix-wide parity on the first and last layers
against the cached fp64 oracle."""
import numpy as np
import pytest

from oracle import partitions as P
from transformer_sharding_affinity_gb300 import stack as ST

from parity_util import TOL, rel_err, topk_agrees


def _check_host_sequence(res, L):
    """Every number of place_heads against the oracle's partition functions."""
    N = len(res.S_up)
    G, I = res.S_up[0].shape
    ups = [P.unit_mass(s.astype(np.float64)) for s in res.S_up]
    downs = [P.unit_mass(s.astype(np.float64)) for s in res.S_down]
    for a, b in zip(res.Shat_up + res.Shat_down, ups + downs):
        np.testing.assert_allclose(a, b, rtol=1e-13)
    nu = [P.contiguous_neurons(I, L)] * N
    hc = [P.contiguous_heads(G, L)] * N
    np.testing.assert_array_equal(res.nu, np.stack(nu))
    np.testing.assert_array_equal(res.h_contiguous, np.stack(hc))
    np.testing.assert_allclose(res.J_contiguous, P.objective_J(ups, downs, hc, nu), rtol=1e-12)
    for i in range(N):
        C = P.group_gain(ups[i], L, nu[i], downs[i - 1] if i else None, nu[i - 1] if i else None)
        _, _, best = P.score_partitions(C)
        assert tuple(res.h_best[i]) == tuple(best), f"layer {i}"
    np.testing.assert_allclose(res.J_best, P.objective_J(ups, downs, list(res.h_best), nu), rtol=1e-12)
    assert 0.0 <= res.J_contiguous <= res.J_best <= 2 * N - 1


def test_place_heads_host_sequence():
    rng = np.random.default_rng(12)
    N, G, I, L = 5, 8, 96, 4
    S_up = [rng.gamma(0.5, size=(G, I)).astype(np.float32) for _ in range(N)]
    S_down = [rng.gamma(0.5, size=(I, G)).astype(np.float32) for _ in range(N - 1)]
    res = ST.place_heads(S_up, S_down, L)
    _check_host_sequence(res, L)


def test_place_heads_uniform_scores_give_the_expectation():
    """Uniform S makes every layout score (2N-1)/L; the first partition wins."""
    N, G, I, L = 4, 8, 64, 4
    res = ST.place_heads([np.ones((G, I), np.float32)] * N, [np.ones((I, G), np.float32)] * (N - 1), L)
    np.testing.assert_allclose([res.J_contiguous, res.J_best], (2 * N - 1) / L, rtol=1e-12)
    np.testing.assert_array_equal(res.h_best, res.h_contiguous)


@pytest.mark.gpu
@pytest.mark.slow
def test_qwen3_stack_28_layers(record_property, tmp_path):
    torch = pytest.importorskip("torch")
    from transformer_sharding_affinity_gb300 import binding as B
    from transformer_sharding_affinity_gb300 import device as DV
    from transformer_sharding_affinity_gb300 import workloads as W

    shape0 = W.stack_layer(0)
    d = B.dims(shape0.T, shape0.D, shape0.H, shape0.G, shape0.dh, shape0.I, shape0.eps, B.AFF_BF16)
    N, L = W.STACK_LAYERS, 4
    keep = {}

    def layer_inputs(i):
        layer = W.make_layer(W.stack_layer(i), with_next=i + 1 < N)
        if i in (0, N - 2, N - 1):
            keep[i] = layer
        return DV.to_device(layer, "bf16", keys=DV.ALL_KEYS if i + 1 < N else DV.UP_KEYS)

    S_up, S_down = ST.calibrate_stack(layer_inputs, N, d, checkpoint_dir=str(tmp_path))
    assert len(S_up) == N and len(S_down) == N - 1
    for S in S_up + S_down:
        assert np.all(np.isfinite(S)) and S.min() >= 0.0 and S.max() > 0.0
    torch.cuda.synchronize()

    # matrix-wide parity of the first and last layers' S_up (FO) and of the first and
    # last S_down against the cached fp64 oracle (tests/oracle_cache/)
    from oracle_cache.make_cache import DOWN_KEYS, UP_KEYS, fingerprint, path_of
    checks = [(0, "up", "stack_l0_fo"), (N - 1, "up", f"stack_l{N - 1}_fo"),
              (0, "down", "stack_l0_down"), (N - 2, "down", f"stack_l{N - 2}_down")]
    for i, kind, case in checks:
        ref = np.load(path_of(case))
        layer = keep[i]
        assert str(ref["fingerprint"]) == fingerprint(layer, UP_KEYS if kind == "up" else DOWN_KEYS), case
        S_gpu = S_up[i] if kind == "up" else S_down[i]
        S_ref = ref["S"]
        e = rel_err(S_gpu, S_ref)
        record_property(f"layer{i}_{kind}_max_rel_err", e)
        assert e <= TOL, f"layer {i} S_{kind}: max rel err {e:.3e}"
        for g in range(W.stack_layer(i).G):
            got, want = (S_gpu[g], S_ref[g]) if kind == "up" else (S_gpu[:, g], S_ref[:, g])
            assert topk_agrees(got, want), f"layer {i} S_{kind}: top-8 of group {g} differs"
    rng = np.random.default_rng(28)
    shape = W.stack_layer(0)

    # resume: only the layers whose checkpoints are gone are recomputed, bit for bit
    for i in (0, N - 1):
        (tmp_path / f"layer_{i:03d}.npz").unlink()
    recomputed = []

    def counted(i):
        recomputed.append(i)
        return layer_inputs(i)
    up2, dn2 = ST.calibrate_stack(counted, N, d, checkpoint_dir=str(tmp_path))
    assert recomputed == [0, N - 1]
    for a, b in zip(up2 + dn2, S_up + S_down):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))

    res = ST.place_heads(S_up, S_down, L)
    _check_host_sequence(res, L)
    assert res.h_best.shape == (N, shape.G)
    # a uniformly random balanced layout scores (2N - 1) / L in expectation ("Objective")
    from transformer_sharding_affinity_gb300 import binding as Bb
    J = [Bb.objective(res.Shat_up, res.Shat_down, [rng.permutation(P.contiguous_heads(shape.G, L)) for _ in range(N)],
                      [rng.permutation(P.contiguous_neurons(shape.I, L)) for _ in range(N)]) for _ in range(200)]
    record_property("J_random_mean", float(np.mean(J)))
    assert abs(np.mean(J) - (2 * N - 1) / L) < 4 * np.std(J) / np.sqrt(len(J)) + 1e-9
    record_property("J_contiguous", res.J_contiguous)
    record_property("J_best_heads", res.J_best)

    # the alternating search from the contiguous layout: J never falls below
    # the head-only optimum, and the first layer's neuron map is the exact
    # best balanced map given the result's head maps
    from oracle import assignment as A
    lay = ST.optimise(res.Shat_up, res.Shat_down, L)
    record_property("J_optimised", lay.J)
    record_property("sweeps", lay.sweeps)
    np.testing.assert_allclose(lay.J, P.objective_J(res.Shat_up, res.Shat_down, list(lay.h), list(lay.nu)),
                               rtol=1e-12)
    assert lay.J >= res.J_best - 1e-12 and lay.J <= 2 * N - 1
    M0 = A.neuron_gain(res.Shat_up[0], lay.h[0], L, res.Shat_down[0], lay.h[1])
    _, best0 = A.best_balanced_neurons(M0)
    np.testing.assert_allclose(A.assignment_value(M0, lay.nu[0]), best0, rtol=1e-12)


def test_calibrate_stack_resumes_from_checkpoints(tmp_path):
    """Layers already on disk are loaded, not recomputed: with every layer
    saved, the call needs no GPU and never asks for inputs."""
    from transformer_sharding_affinity_gb300 import binding as B
    rng = np.random.default_rng(21)
    N, G, I = 3, 4, 16
    saved_up = [rng.random((G, I)).astype(np.float32) for _ in range(N)]
    saved_dn = [rng.random((I, G)).astype(np.float32) for _ in range(N - 1)]
    for i in range(N):
        arrays = {"S_up": saved_up[i]} if i == N - 1 else {"S_up": saved_up[i], "S_down": saved_dn[i]}
        np.savez(tmp_path / f"layer_{i:03d}.npz", **arrays)

    def no_inputs(i):
        raise AssertionError(f"layer {i} was recomputed")

    d = B.dims(64, 32, 4, G, 8, I)
    up, dn = ST.calibrate_stack(no_inputs, N, d, checkpoint_dir=str(tmp_path))
    for a, b in zip(up + dn, saved_up + saved_dn):
        assert np.array_equal(a, b)
