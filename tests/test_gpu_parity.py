"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs, every entry and the top-8 ranking per KV group, on small
and medium shapes (the full-size layers are in test_gpu_full_size.py).  Paper:
"Affinity-Aware Sharding for Delayed Tensor Parallelism", §3 "Affinity scores"."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import affinity_oracle as O
from transformer_sharding_affinity_gb300 import binding as B
from transformer_sharding_affinity_gb300 import device as DV
from transformer_sharding_affinity_gb300 import workloads as W

from parity_util import (FEW_TOKENS, TOL, TOL_F32, oracle_down, oracle_up, rel_err, rowmax_err, run_down, run_up,
                         topk_agrees)

pytestmark = pytest.mark.gpu

S = W.LayerShape
SMALL = [
    S("tiles", T=384, D=256, H=4, G=2, dh=64, I=256, dtype="bf16", w_std=0.05, x_dist="normal_outliers", seed=11),
    S("ragged_T", T=333, D=192, H=4, G=2, dh=96, I=384, dtype="bf16", w_std=0.05, x_dist="normal_outliers", seed=12),
    S("ragged_I", T=129, D=128, H=2, G=1, dh=128, I=200, dtype="bf16", w_std=0.05, x_dist="normal", seed=13),
    S("dh16", T=256, D=64, H=4, G=2, dh=16, I=128, dtype="bf16", w_std=0.05, x_dist="normal", seed=14),
    S("one_token", T=1, D=64, H=2, G=2, dh=32, I=136, dtype="bf16", w_std=0.05, x_dist="normal", seed=15),
    S("mqa", T=200, D=128, H=8, G=1, dh=24, I=64, dtype="bf16", w_std=0.05, x_dist="normal_outliers", seed=16),
    S("wide_head", T=160, D=520, H=2, G=2, dh=256, I=264, dtype="bf16", w_std=0.03, x_dist="student_t4", seed=17),
    S("many_heads", T=140, D=128, H=32, G=8, dh=8, I=128, dtype="bf16", w_std=0.05, x_dist="normal", seed=18),
]
MEDIUM = S("qwen_slice", T=4096, D=1024, H=16, G=8, dh=128, I=512, dtype="bf16", w_std=0.02,
           x_dist="normal_outliers", seed=21)


def _assert_up(shape, mode, tol=TOL, record=None):
    layer = W.make_layer(shape)
    (S_gpu, Sh_gpu), = run_up(B, DV, shape, layer, mode)
    S_ref, Sh_ref = oracle_up(O, shape, layer, mode)
    err = rowmax_err if shape.T < FEW_TOKENS else rel_err
    e = err(S_gpu, S_ref)
    eh = err(Sh_gpu, Sh_ref)
    if record:
        record(f"{shape.name}_{mode}_max_rel_err", e)
    assert e <= tol and eh <= tol, f"{shape.name} {mode}: max rel err S {e:.3e}, S_head {eh:.3e}"
    for g in range(shape.G):
        assert topk_agrees(S_gpu[g], S_ref[g]), f"{shape.name} {mode}: top-8 of group {g} differs"
    # the group sum of the per-head output is the grouped output
    hpg = shape.H // shape.G
    np.testing.assert_allclose(Sh_gpu.reshape(shape.G, hpg, shape.I).sum(1), S_gpu, rtol=2e-6, atol=0)
    return e


@pytest.mark.parametrize("mode", ["fo", "add", "add_direct", "loo"])
@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_up_small(shape, mode):
    _assert_up(shape, mode)


@pytest.mark.parametrize("mode", ["fo", "add"])
def test_up_tiny_fp32(mode, record_property):
    _assert_up(W.CONFIGS["tiny"], mode, tol=TOL_F32, record=record_property)


@pytest.mark.parametrize("mode", ["fo", "add", "add_direct", "loo"])
def test_up_medium(mode, record_property):
    _assert_up(MEDIUM, mode, record=record_property)


def test_loo_is_deterministic_and_differs_from_add():
    shape = MEDIUM.scaled(T=2048)
    layer = W.make_layer(shape)
    outs = run_up(B, DV, shape, layer, "loo", runs=2)
    assert np.array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))
    (S_add, _), = run_up(B, DV, shape, layer, "add")
    assert np.max(np.abs(outs[0][0] / S_add - 1)) > 1e-2


def test_add_second_moment_form():
    """ADD through each head's second moment: bit-for-bit repeatable, a = 0 gives
    exactly 0, and it agrees with the direct contraction (both are checked
    against the oracle elsewhere; here against each other on a 4096-token slice)."""
    layer = W.make_layer(MEDIUM)
    outs = run_up(B, DV, MEDIUM, layer, "add", runs=2)
    assert np.array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))
    assert np.array_equal(outs[0][1].view(np.uint32), outs[1][1].view(np.uint32))
    (S_dir, Sh_dir), = run_up(B, DV, MEDIUM, layer, "add_direct")
    assert rel_err(outs[0][0], S_dir) <= TOL and rel_err(outs[0][1], Sh_dir) <= TOL
    z = dict(layer)
    z["a"] = np.zeros_like(layer["a"])
    z["a_bits"] = np.zeros_like(layer["a_bits"])
    (S0, Sh0), = run_up(B, DV, MEDIUM, z, "add")
    assert np.all(S0 == 0.0) and np.all(Sh0 == 0.0)


def test_add_many_quadratic_form_units():
    """16 heads x 2048 neurons: 512 quadratic-form units, more than two per SM of a
    152-SM part, and 16 x 16 Gram units.  Sampled neurons against the oracle over
    all tokens, both ADD forms, and bit-identical repeats."""
    shape = S("many_units", T=1536, D=256, H=16, G=8, dh=64, I=2048, dtype="bf16", w_std=0.05,
              x_dist="normal_outliers", seed=24)
    layer = W.make_layer(shape)
    rng = np.random.default_rng(8)
    for mode in ("add", "add_direct"):
        outs = run_up(B, DV, shape, layer, mode, runs=2)
        S_gpu, Sh_gpu = outs[0]
        assert np.array_equal(S_gpu.view(np.uint32), outs[1][0].view(np.uint32))
        idx = _candidates(S_gpu, rng, top=8, n_random=48)
        S_ref, Sh_ref = oracle_up(O, shape, layer, mode, neurons=idx)
        assert rel_err(S_gpu[:, idx], S_ref) <= TOL, mode
        assert rel_err(Sh_gpu[:, idx], Sh_ref) <= TOL, mode
        for g in range(shape.G):
            assert topk_agrees(S_gpu[g, idx], S_ref[g]), f"{mode}: top-8 of group {g} differs"


def test_add_fold_split_leaves_results_unchanged(monkeypatch):
    """ADD in the second-moment form may run some fold units before the Gram pass
    (beside 1/r) and the rest after it; each unit writes its own M16 tile, so S is
    bit-identical however the units are split (none early, some, all)."""
    shape = S("fold_split", T=1536, D=256, H=16, G=8, dh=64, I=2048, dtype="bf16", w_std=0.05,
              x_dist="normal_outliers", seed=25)
    layer = W.make_layer(shape)
    outs = []
    for early in ("0", "37", "100000"):
        monkeypatch.setenv("AFFINITY_FOLD_EARLY", early)
        outs.append(run_up(B, DV, shape, layer, "add")[0])
    for S_, Sh_ in outs[1:]:
        assert np.array_equal(S_.view(np.uint32), outs[0][0].view(np.uint32))
        assert np.array_equal(Sh_.view(np.uint32), outs[0][1].view(np.uint32))


def test_up_deterministic():
    layer = W.make_layer(MEDIUM)
    outs = run_up(B, DV, MEDIUM, layer, "fo", runs=3)
    for S_, Sh_ in outs[1:]:
        assert np.array_equal(S_.view(np.uint32), outs[0][0].view(np.uint32))
        assert np.array_equal(Sh_.view(np.uint32), outs[0][1].view(np.uint32))


def test_up_zero_heads_and_gate_only():
    """a = 0 gives S_up = 0 exactly; Wu = 0 gives FO = 0 (the oracle's special cases)."""
    shape = SMALL[0]
    layer = W.make_layer(shape)
    z = dict(layer)
    z["a"] = np.zeros_like(layer["a"])
    z["a_bits"] = np.zeros_like(layer["a_bits"])
    (S0, _), = run_up(B, DV, shape, z, "fo")
    assert np.all(S0 == 0.0)
    u = dict(layer)
    u["Wu"] = np.zeros_like(layer["Wu"])
    u["Wu_bits"] = np.zeros_like(layer["Wu_bits"])
    (S1, _), = run_up(B, DV, shape, u, "fo")
    assert np.all(S1 == 0.0)


def test_up_permutation_equivariance():
    """Permuting neurons permutes S_up's columns (bit-exact when whole 128-neuron
    tiles are permuted, within tolerance otherwise)."""
    shape = MEDIUM.scaled(T=1024)
    layer = W.make_layer(shape)
    (S_ref, _), = run_up(B, DV, shape, layer, "fo")
    perm = np.concatenate([np.arange(256, 384), np.arange(0, 128), np.arange(384, 512), np.arange(128, 256)])
    p = dict(layer)
    for k in ("Wg", "Wu"):
        p[k] = layer[k][perm]
        p[k + "_bits"] = layer[k + "_bits"][perm]
    p["Wd"] = layer["Wd"][:, perm]
    p["Wd_bits"] = np.ascontiguousarray(layer["Wd_bits"][:, perm])
    (S_p, _), = run_up(B, DV, shape, p, "fo")
    assert np.array_equal(S_p, S_ref[:, perm])


@pytest.mark.parametrize("shape", SMALL[:4] + [W.CONFIGS["tiny"]], ids=[s.name for s in SMALL[:4]] + ["tiny"])
def test_down_small(shape, record_property):
    layer = W.make_layer(shape, with_next=True)
    S_gpu, = run_down(B, DV, shape, layer)
    S_ref = oracle_down(O, shape, layer)
    tol = TOL_F32 if shape.dtype == "fp32" else TOL
    e = rel_err(S_gpu, S_ref)
    record_property(f"{shape.name}_down_max_rel_err", e)
    assert e <= tol, f"{shape.name} down: max rel err {e:.3e}"


def test_down_medium_deterministic():
    shape = MEDIUM.scaled(T=2048)
    layer = W.make_layer(shape, with_next=True)
    outs = run_down(B, DV, shape, layer, runs=2)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    S_ref = oracle_down(O, shape, layer)
    e = rel_err(outs[0], S_ref)
    assert e <= TOL, f"down medium: max rel err {e:.3e}"


def _candidates(S_gpu, rng, top=16, n_random=48):
    G, I = S_gpu.shape
    cand = set()
    for g in range(G):
        cand.update(np.argsort(-S_gpu[g], kind="stable")[:top].tolist())
    cand.update(rng.choice(I, size=min(n_random, I), replace=False).tolist())
    return np.array(sorted(cand))


_SWEEP = [W.random_small_shape(np.random.default_rng(1000 + i), name=f"rand{i}") for i in range(12)]


@pytest.mark.parametrize("shape", _SWEEP, ids=[s.name for s in _SWEEP])
def test_up_random_shapes(shape):
    """Seeded random small shapes (ragged T, D, d_head and I; 1-12 heads in
    1-4 groups): every mode against the oracle."""
    for mode in ("fo", "add", "add_direct", "loo"):
        _assert_up(shape, mode)


@pytest.mark.parametrize("shape", _SWEEP[:6], ids=[s.name for s in _SWEEP[:6]])
def test_down_random_shapes(shape):
    layer = W.make_layer(shape, with_next=True)
    S_gpu, = run_down(B, DV, shape, layer)
    S_ref = oracle_down(O, shape, layer)
    err = rowmax_err(S_gpu.T, S_ref.T) if shape.T < FEW_TOKENS else rel_err(S_gpu, S_ref)
    assert err <= TOL, f"{shape.name} down: {err:.3e}"
