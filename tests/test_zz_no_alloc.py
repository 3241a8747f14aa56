"""affinity_up_static -- the entry point for callers that cannot allocate
device memory -- against affinity_up on the same inputs, two calls in a row.

Kept in a file of its own that pytest collects last, so that a run stopping
at its first failure has already run every other test; it also passes on
its own in a fresh process."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from transformer_sharding_affinity_gb300 import binding as B
from transformer_sharding_affinity_gb300 import device as DV
from transformer_sharding_affinity_gb300 import workloads as W

from parity_util import TOL, dims_of, rel_err, run_up

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 64 << 20


def _static(shape, layer, mode):
    dev = DV.to_device(layer, shape.dtype)
    d = dims_of(B, shape)
    S = torch.full((shape.G, shape.I), float("nan"), device="cuda")
    Sh = torch.full((shape.H, shape.I), float("nan"), device="cuda")
    B.affinity_up_static(dev["a"], dev["x"], dev["Wo"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], d,
                         B.MODES[mode], S, Sh)
    torch.cuda.synchronize()
    return S.cpu().numpy(), Sh.cpu().numpy()


def test_static_scratch_matches_workspace_entry_point():
    # a larger call first, then a smaller one that sits on the first call's leftovers
    first = W.LayerShape("nx_a", T=1536, D=512, H=8, G=4, dh=64, I=640, dtype="bf16", w_std=0.03,
                         x_dist="normal_outliers", seed=31)
    second = W.LayerShape("nx_b", T=333, D=192, H=4, G=2, dh=96, I=264, dtype="bf16", w_std=0.05,
                          x_dist="normal_outliers", seed=32)
    for shape, mode in ((first, "fo"), (second, "fo"), (second, "add")):
        d = dims_of(B, shape)
        assert B.workspace_size(d, B.MODES[mode]) <= SCRATCH_LIMIT
        layer = W.make_layer(shape)
        S_s, Sh_s = _static(shape, layer, mode)
        (S_w, Sh_w), = run_up(B, DV, shape, layer, mode)
        assert np.isfinite(S_s).all() and np.isfinite(Sh_s).all()
        assert rel_err(S_s, S_w) <= TOL and rel_err(Sh_s, Sh_w) <= TOL, shape.name


def test_static_scratch_refuses_shapes_over_the_limit():
    shape = W.CONFIGS["qwen3_0p6b_layer"]
    d = dims_of(B, shape)
    assert B.workspace_size(d, B.AFF_MODE_FO) > SCRATCH_LIMIT
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    S = torch.empty(1, device="cuda")
    with pytest.raises(B.AffinityError) as e:
        B.affinity_up_static(x, x, x, x, x, x, x, d, B.AFF_MODE_FO, S, None)
    assert e.value.status == B.AFF_ERR_WORKSPACE
