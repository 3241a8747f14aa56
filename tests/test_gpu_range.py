"""Inputs outside fp16's range: every finite bf16 input is accepted.

The bf16 path contracts fp16 copies of its operands on the tensor cores.  Each
copy is scaled by a power of two chosen on the device from the tensor's
largest magnitude (or a bound on it), and the fp32 results are scaled back, so
head outputs, gains and weights far outside fp16's range give the same scores
as the fp64 oracle on the same inputs ("Affinity-Aware Sharding for Delayed
Tensor Parallelism", §3 "Affinity scores": p_h = gamma (a_h W_o^(h)) / r is
defined for any activations; its §5.6 reports massive activations).  A
non-finite input is still reported as AFF_ERR_RANGE."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import affinity_oracle as O  # noqa: E402
from transformer_sharding_affinity_gb300 import binding as B  # noqa: E402
from transformer_sharding_affinity_gb300 import device as DV  # noqa: E402
from transformer_sharding_affinity_gb300 import workloads as W  # noqa: E402

from parity_util import TOL, dims_of, mode_of, oracle_up, rel_err, rowmax_err, run_up, topk_agrees  # noqa: E402

pytestmark = pytest.mark.gpu

SHAPE = W.LayerShape("range", T=384, D=256, H=4, G=2, dh=64, I=256, dtype="bf16", w_std=0.05,
                     x_dist="normal_outliers", seed=51)
STREAMED = W.LayerShape("range_dh96", T=300, D=192, H=4, G=2, dh=96, I=264, dtype="bf16", w_std=0.05,
                        x_dist="normal_outliers", seed=52)


def _set(layer, key, values):
    """Replace one input by exactly representable bf16 values (float view and bit pattern)."""
    bits = W.bf16_bits(np.asarray(values, np.float32))
    layer[key + "_bits"] = bits
    layer[key] = (bits.astype(np.uint32) << 16).view(np.float32)


def _scaled(layer, key, power):
    out = dict(layer)
    _set(out, key, layer[key] * np.float32(2.0 ** power))   # a power of two: exact in bf16 here
    return out


def _one_huge_head_output(layer):
    out = dict(layer)
    a = layer["a"].copy()
    a[5, 7] = 999424.0            # a bf16 value; a / r is far beyond fp16's 65504
    _set(out, "a", a)
    return out


# Each case moves staged operands far outside fp16's range (|v| < 65504, normal
# above 2^-14) while the SwiGLU operating point g, u keeps its ordinary size:
# scaling the gate/up weights up and the gain down by the same power of two
# leaves g, u and every p_h.w unchanged but overflows W16 and underflows n16.
CASES = {
    "one_huge_head_output": _one_huge_head_output,
    "huge_head_outputs": lambda L: _scaled(L, "a", 17),
    "tiny_head_outputs": lambda L: _scaled(L, "a", -40),
    "huge_gate_up_weights_tiny_gain": lambda L: _scaled(_scaled(_scaled(L, "Wg", 22), "Wu", 22), "gamma", -22),
    "huge_gain_tiny_gate_up_weights": lambda L: _scaled(_scaled(_scaled(L, "Wg", -14), "Wu", -14), "gamma", 14),
    "huge_Wo_tiny_head_outputs": lambda L: _scaled(_scaled(L, "Wo", 20), "a", -20),
    "tiny_Wo": lambda L: _scaled(L, "Wo", -34),
}
MODES = ["fo", "add", "add_direct", "loo"]
# One head output a million times the others makes that head's scores the
# contribution of a single token: nothing averages the fixed fp16 rounding of
# the folded rows there, so those entries are held to the few-token bar (the
# error relative to each row's largest entry), as for layers of under 64 tokens.
FEW_TOKEN_CASES = {"one_huge_head_output"}


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", list(CASES), ids=list(CASES))
def test_out_of_fp16_range_inputs_match_the_oracle(case, mode, record_property):
    for shape in (SHAPE, STREAMED):
        layer = CASES[case](W.make_layer(shape))
        (S_gpu, Sh_gpu), = run_up(B, DV, shape, layer, mode)   # asserts a clean device status
        S_ref, Sh_ref = oracle_up(O, shape, layer, mode)
        assert np.isfinite(S_gpu).all() and np.isfinite(Sh_gpu).all()
        err = rowmax_err if case in FEW_TOKEN_CASES else rel_err
        e, eh = err(S_gpu, S_ref), err(Sh_gpu, Sh_ref)
        record_property(f"{shape.name}_{case}_{mode}_max_rel_err", e)
        assert e <= TOL and eh <= TOL, f"{shape.name} {case} {mode}: max rel err S {e:.3e}, S_head {eh:.3e}"
        for g in range(shape.G):
            assert topk_agrees(S_gpu[g], S_ref[g]), f"{shape.name} {case} {mode}: top-8 of group {g} differs"


@pytest.mark.parametrize("mode", MODES)
def test_scaling_leaves_ordinary_inputs_bit_identical_across_runs(mode):
    outs = run_up(B, DV, SHAPE, W.make_layer(SHAPE), mode, runs=2)
    assert np.array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))


@pytest.mark.parametrize("mode", MODES)
def test_non_finite_input_is_reported(mode):
    """An infinite head output has no finite score: the call reports AFF_ERR_RANGE,
    and the same workspace computes the next call normally."""
    layer = W.make_layer(SHAPE)
    bad = dict(layer)
    bad["a_bits"] = layer["a_bits"].copy()
    bad["a_bits"][5, 7] = 0x7F80          # bf16 +inf
    m, flags = mode_of(B, mode)
    d = dims_of(B, SHAPE, flags)
    ws = torch.empty(B.workspace_size(d, m), dtype=torch.uint8, device="cuda")
    S = torch.empty(SHAPE.G, SHAPE.I, device="cuda")
    dev = DV.to_device(bad, "bf16")
    B.affinity_up(dev["a"], dev["x"], dev["Wo"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], d, m, S, None, ws)
    assert B.device_status(ws) == B.AFF_ERR_RANGE
    dev = DV.to_device(layer, "bf16")
    B.affinity_up(dev["a"], dev["x"], dev["Wo"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], d, m, S, None, ws)
    assert B.device_status(ws) == B.AFF_OK
    S_ref, _ = oracle_up(O, SHAPE, layer, mode)
    assert rel_err(S.cpu().numpy(), S_ref) <= TOL
