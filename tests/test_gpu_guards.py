"""Failure detection and memory guards on the GPU.

* A kernel whose only wait can never be satisfied must give up after its
  limit, latch AFF_ERR_DEVICE_TIMEOUT in the workspace and leave the context
  usable (the path every bounded pipeline wait takes on a stall).
* Canary bytes just past the declared workspace and past each output must
  be untouched by every mode of the pass."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import affinity_oracle as O  # noqa: E402
from transformer_sharding_affinity_gb300 import binding as B  # noqa: E402
from transformer_sharding_affinity_gb300 import device as DV  # noqa: E402
from transformer_sharding_affinity_gb300 import workloads as W  # noqa: E402

from parity_util import TOL, dims_of, mode_of, oracle_up, rel_err  # noqa: E402

pytestmark = pytest.mark.gpu

SHAPE = W.LayerShape("guard", T=300, D=192, H=4, G=2, dh=96, I=264, dtype="bf16", w_std=0.05,
                     x_dist="normal_outliers", seed=31)
CANARY = 0x5A
TAIL = 65536


def test_bounded_wait_times_out_and_the_context_stays_usable():
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    B.selftest_timeout(ws, limit_ns=5_000_000)
    assert B.device_status(ws) == B.AFF_ERR_DEVICE_TIMEOUT
    assert B.device_status(ws) == B.AFF_OK          # reading the status clears it
    layer = W.make_layer(SHAPE)
    dev = DV.to_device(layer, "bf16")
    d = dims_of(B, SHAPE)
    ws = torch.empty(B.workspace_size(d, B.AFF_MODE_FO), dtype=torch.uint8, device="cuda")
    S = torch.empty(SHAPE.G, SHAPE.I, device="cuda")
    B.affinity_up(dev["a"], dev["x"], dev["Wo"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], d, B.AFF_MODE_FO, S,
                  None, ws)
    assert B.device_status(ws) == B.AFF_OK
    S_ref, _ = oracle_up(O, SHAPE, layer, "fo")
    assert rel_err(S.cpu().numpy(), S_ref) <= TOL


@pytest.mark.parametrize("mode", ["fo", "add", "add_direct", "loo", "down"])
def test_nothing_is_written_past_the_workspace_or_the_outputs(mode):
    layer = W.make_layer(SHAPE, with_next=(mode == "down"))
    down = mode == "down"
    m, flags = (0, 0) if down else mode_of(B, mode)
    d = dims_of(B, SHAPE, flags)
    keys = DV.DOWN_KEYS if down else DV.UP_KEYS
    dev = DV.to_device(layer, "bf16", keys=keys)
    n = B.workspace_size(d, m, down=down)
    buf = torch.full((n + TAIL,), CANARY, dtype=torch.uint8, device="cuda")
    ws = buf[:n]
    out_n = SHAPE.G * SHAPE.I
    out = torch.full((out_n + TAIL // 4,), -7.0, device="cuda")
    head = torch.full((SHAPE.H * SHAPE.I + TAIL // 4,), -7.0, device="cuda")
    if down:
        B.affinity_down(dev["x"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], dev["gamma_next"], dev["Wq_next"],
                        dev["Wk_next"], dev["Wv_next"], d, out[:out_n], ws)
    else:
        B.affinity_up(dev["a"], dev["x"], dev["Wo"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], d,
                      m, out[:out_n], head[:SHAPE.H * SHAPE.I], ws)
    assert B.device_status(ws) == B.AFF_OK
    assert torch.all(buf[n:] == CANARY).item(), "bytes past the workspace were written"
    assert torch.all(out[out_n:] == -7.0).item(), "floats past S_out were written"
    if not down:
        assert torch.all(head[SHAPE.H * SHAPE.I:] == -7.0).item(), "floats past S_head_out were written"
    assert torch.isfinite(out[:out_n]).all().item()


def test_one_call_helpers_match_the_abi():
    from transformer_sharding_affinity_gb300 import scores
    layer = W.make_layer(SHAPE, with_next=True)
    dev = DV.to_device(layer, "bf16", keys=DV.ALL_KEYS)
    S, Sh = scores.s_up(dev["a"], dev["x"], dev["Wo"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], SHAPE.H,
                        SHAPE.G, "fo", SHAPE.eps, per_head=True)
    S_ref, _ = oracle_up(O, SHAPE, layer, "fo")
    assert rel_err(S.cpu().numpy(), S_ref) <= TOL
    np.testing.assert_allclose(Sh.cpu().numpy().reshape(SHAPE.G, -1, SHAPE.I).sum(1), S.cpu().numpy(), rtol=2e-6)
    Sd = scores.s_down(dev["x"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], dev["gamma_next"], dev["Wq_next"],
                       dev["Wk_next"], dev["Wv_next"], SHAPE.H, SHAPE.G, SHAPE.eps)
    Sd_ref = O.s_down(layer["x"], layer["gamma"], layer["Wg"], layer["Wu"], layer["Wd"], layer["gamma_next"],
                      layer["Wq_next"], layer["Wk_next"], layer["Wv_next"], SHAPE.H, SHAPE.G, SHAPE.dh, SHAPE.eps)
    assert rel_err(Sd.cpu().numpy(), Sd_ref) <= TOL


def test_the_pass_can_be_captured_in_a_cuda_graph():
    """affinity_up is stream-ordered with no host synchronisation, so it can be
    captured (including its side-stream fork / join) and replayed; replays
    are bit-identical to direct calls and follow new inputs written in place."""
    layer = W.make_layer(SHAPE)
    dev = DV.to_device(layer, "bf16")
    d = dims_of(B, SHAPE)
    ws = torch.empty(B.workspace_size(d, B.AFF_MODE_FO), dtype=torch.uint8, device="cuda")
    S = torch.empty(SHAPE.G, SHAPE.I, device="cuda")

    def call():
        B.affinity_up(dev["a"], dev["x"], dev["Wo"], dev["gamma"], dev["Wg"], dev["Wu"], dev["Wd"], d,
                      B.AFF_MODE_FO, S, None, ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()                                    # warm-up outside capture (first-use setup)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    direct = S.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    S.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert B.device_status(ws) == B.AFF_OK
    assert torch.equal(S, direct)
    # new activations in the same buffers: the replay computes them
    other = W.make_layer(SHAPE.scaled(seed=SHAPE.seed + 1))
    dev["a"].copy_(DV.host_tensor(other, "a", "bf16").cuda())
    dev["x"].copy_(DV.host_tensor(other, "x", "bf16").cuda())
    g.replay()
    torch.cuda.synchronize()
    ref = dict(layer)
    ref["a"], ref["x"] = other["a"], other["x"]
    S_ref, _ = oracle_up(O, SHAPE, ref, "fo")
    assert rel_err(S.cpu().numpy(), S_ref) <= TOL
