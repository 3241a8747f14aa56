"""affinity_up_static -- the entry point for callers that cannot allocate
device memory -- against affinity_up on the same inputs, two calls in a row.

Callers that cannot allocate are, for example, a plugin whose host framework
owns every device allocation and hands out no scratch, or a process whose
memory pool already holds the whole device.  The static entry point runs the
same kernels on a scratch array compiled into the library, so its output must
equal affinity_up's bit for bit; device-side errors are read from that array
with affinity_static_device_status.

Kept in a file of its own that pytest collects last, so that a run stopping
at its first failure has already run every other test; it also passes on
its own in a fresh process."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from transformer_sharding_affinity_gb300 import binding as B
from transformer_sharding_affinity_gb300 import device as DV
from transformer_sharding_affinity_gb300 import workloads as W

from parity_util import dims_of, mode_of, run_up

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 64 << 20


def _static(shape, layer, mode):
    dev = DV.to_device(layer, shape.dtype)
    m, flags = mode_of(B, mode)
    d = dims_of(B, shape, flags)
    S = torch.full((shape.G, shape.I), float("nan"), device="cuda")
    Sh = torch.full((shape.H, shape.I), float("nan"), device="cuda")
    B.affinity_up_static(dev["a"], dev["x"], dev["Wo"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], d, m, S, Sh)
    st = B.static_device_status()
    assert st == B.AFF_OK, f"static device status {st}: {B.strerror(st)}"
    return S.cpu().numpy(), Sh.cpu().numpy()


def _bits(v):
    return np.ascontiguousarray(v, np.float32).view(np.uint32)


def test_static_scratch_matches_workspace_entry_point():
    # a larger call first, then smaller ones that sit on the earlier calls' leftovers
    first = W.LayerShape("nx_a", T=1536, D=512, H=8, G=4, dh=64, I=640, dtype="bf16", w_std=0.03,
                         x_dist="normal_outliers", seed=31)
    second = W.LayerShape("nx_b", T=333, D=192, H=4, G=2, dh=96, I=264, dtype="bf16", w_std=0.05,
                          x_dist="normal_outliers", seed=32)
    for shape, mode in ((first, "fo"), (second, "fo"), (second, "add"), (first, "loo"), (second, "add_direct")):
        m, flags = mode_of(B, mode)
        assert B.workspace_size(dims_of(B, shape, flags), m) <= SCRATCH_LIMIT
        layer = W.make_layer(shape)
        (S_w, Sh_w), = run_up(B, DV, shape, layer, mode)
        for _ in range(2):   # two calls in a row on the same static scratch
            S_s, Sh_s = _static(shape, layer, mode)
            assert np.array_equal(_bits(S_s), _bits(S_w)), f"{shape.name} {mode}: S differs"
            assert np.array_equal(_bits(Sh_s), _bits(Sh_w)), f"{shape.name} {mode}: S_head differs"


@pytest.mark.parametrize("mode", ["fo", "add"])
def test_static_scratch_reports_device_errors(mode):
    """A non-finite head output reaches the fp16 operands; the kernels latch
    AFF_ERR_RANGE in the static array's status word, affinity_static_device_status
    reports it once and clears it, and the next call is clean."""
    shape = W.LayerShape("nx_c", T=256, D=128, H=4, G=2, dh=64, I=256, dtype="bf16", w_std=0.05,
                         x_dist="normal", seed=33)
    layer = W.make_layer(shape)
    bad = dict(layer)
    bad["a_bits"] = layer["a_bits"].copy()
    bad["a_bits"][5, 7] = 0x7F80          # bf16 +inf
    m, flags = mode_of(B, mode)
    d = dims_of(B, shape, flags)
    dev = DV.to_device(bad, "bf16")
    S = torch.empty(shape.G, shape.I, device="cuda")
    B.affinity_up_static(dev["a"], dev["x"], dev["Wo"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], d, m, S, None)
    assert B.static_device_status() == B.AFF_ERR_RANGE
    assert B.static_device_status() == B.AFF_OK          # read once, then cleared
    S_s, _ = _static(shape, layer, mode)
    (S_w, _), = run_up(B, DV, shape, layer, mode)
    assert np.array_equal(_bits(S_s), _bits(S_w))


def test_static_scratch_refuses_shapes_over_the_limit():
    shape = W.CONFIGS["qwen3_0p6b_layer"]
    d = dims_of(B, shape)
    assert B.workspace_size(d, B.AFF_MODE_FO) > SCRATCH_LIMIT
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    S = torch.empty(1, device="cuda")
    with pytest.raises(B.AffinityError) as e:
        B.affinity_up_static(x, x, x, x, x, x, x, d, B.AFF_MODE_FO, S, None)
    assert e.value.status == B.AFF_ERR_WORKSPACE
