"""Layout realisation on the GPU ("Affinity-Aware Sharding for Delayed Tensor
Parallelism", §3 "The layout as a free variable"): the permuted weights equal
the oracle's bit for bit, and the dense and L-device forward passes of the
permuted layer reproduce the original layer."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import layer_forward as LF  # noqa: E402
from oracle import partitions as P  # noqa: E402
from transformer_sharding_affinity_gb300 import stack as ST  # noqa: E402
from transformer_sharding_affinity_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu
NAMES = ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")


def _weights(rng, D, H, G, dh, I, bf16):
    w = {"g_attn": 1 + 0.1 * rng.standard_normal(D), "g_ffn": 1 + 0.1 * rng.standard_normal(D),
         "qn": 1 + 0.1 * rng.standard_normal(dh), "kn": 1 + 0.1 * rng.standard_normal(dh)}
    shapes = {"Wq": (H * dh, D), "Wk": (G * dh, D), "Wv": (G * dh, D), "Wo": (D, H * dh), "Wg": (I, D),
              "Wu": (I, D), "Wd": (D, I)}
    for k, s in shapes.items():
        v = (0.1 * rng.standard_normal(s)).astype(np.float32)
        w[k] = W.bf16_round(v) if bf16 else v
    return w


def _to_dev(w, bf16):
    out = {}
    for k in NAMES:
        if bf16:
            out[k] = torch.from_numpy(W.bf16_bits(w[k]).view(np.int16)).view(torch.bfloat16).cuda()
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(w[k])).cuda()
    return out


def _to_host(t):
    if t.dtype == torch.bfloat16:
        return (t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    return t.cpu().numpy()


@pytest.mark.parametrize("L,bf16", [(2, True), (4, False), (4, True)])
def test_realised_layer_matches_the_oracle_and_keeps_the_function(L, bf16):
    rng = np.random.default_rng(L + 10 * bf16)
    T, D, H, G, dh, I = 16, 64, 8, 4, 16, 128
    w = _weights(rng, D, H, G, dh, I, bf16)
    h = rng.permutation(P.contiguous_heads(G, L)).astype(np.int32)
    nu = rng.permutation(P.contiguous_neurons(I, L)).astype(np.int32)
    dev, go, ho, no = ST.realise_layout(_to_dev(w, bf16), h, nu, H, G, dh, L)
    ref, rgo, rho, rno = LF.realise(w, h, nu, H, G, dh, L)
    np.testing.assert_array_equal(go, rgo)
    np.testing.assert_array_equal(ho, rho)
    np.testing.assert_array_equal(no, rno)
    got = dict(w)
    for k in NAMES:
        got[k] = _to_host(dev[k])
        assert np.array_equal(got[k].view(np.uint32), np.asarray(ref[k], np.float32).view(np.uint32)), k
    x = rng.standard_normal((T, D))
    dense = LF.layer_forward(x, w, H, G, dh)
    np.testing.assert_allclose(LF.layer_forward(x, got, H, G, dh), dense, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(LF.sharded_forward(x, got, H, G, dh, L), dense, rtol=1e-12, atol=1e-12)


def test_realise_at_qwen3_shape_is_a_pure_permutation():
    rng = np.random.default_rng(7)
    D, H, G, dh, I, L = 1024, 16, 8, 128, 3072, 4
    w = _weights(rng, D, H, G, dh, I, True)
    h = rng.permutation(P.contiguous_heads(G, L)).astype(np.int32)
    nu = rng.permutation(P.contiguous_neurons(I, L)).astype(np.int32)
    dev, _, _, _ = ST.realise_layout(_to_dev(w, True), h, nu, H, G, dh, L)
    ref, _, _, _ = LF.realise(w, h, nu, H, G, dh, L)
    for k in NAMES:
        assert np.array_equal(_to_host(dev[k]).view(np.uint32), np.asarray(ref[k], np.float32).view(np.uint32)), k
