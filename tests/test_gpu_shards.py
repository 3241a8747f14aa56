"""Token shards on the GPU: affinity_up / affinity_down run on two disjoint
token ranges of one layer in one process, and the library's exchange step
(affinity_combine_shards, a token-weighted mean in shard order) merges them.

Every affinity entry is a token mean times a per-neuron factor ("Affinity-
Aware Sharding for Delayed Tensor Parallelism", §3 "Affinity scores"), so the
merged matrices equal the single call on all tokens up to the rounding of the
final sums, and the oracle within the acceptance tolerance.  The multi-process
form of the same merge is tested with gloo ranks in test_shards_gloo.py."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import affinity_oracle as O
from transformer_sharding_affinity_gb300 import binding as B
from transformer_sharding_affinity_gb300 import device as DV
from transformer_sharding_affinity_gb300 import workloads as W

from parity_util import TOL, oracle_down, oracle_up, rel_err, run_down, run_up

pytestmark = pytest.mark.gpu

SHAPE = W.LayerShape("shards", T=4096, D=1024, H=16, G=8, dh=128, I=512, dtype="bf16", w_std=0.02,
                     x_dist="normal_outliers", seed=41)
# a split on the 512-token chunk grid of the head passes, and a ragged one
SPLITS = [1536, 1000]
# Merged against the single call: the head passes' 512-token partial sums are the
# same on the chunk grid, so only the final fp32 roundings differ (a few ulps).
# The second-moment ADD form sums each head's Gram matrix over token chunks sized
# from T, so a shard moves the chunk boundaries: fp32 reordering of the sums.
MERGE_RTOL = {"fo": 2e-6, "loo": 2e-6, "add": 2e-5}


def _token_slice(layer, lo, hi):
    part = dict(layer)
    for k in ("a", "x"):
        part[k] = layer[k][lo:hi]
        part[k + "_bits"] = layer[k + "_bits"][lo:hi]
    return part


@pytest.mark.parametrize("split", SPLITS)
@pytest.mark.parametrize("mode", ["fo", "add", "loo"])
def test_up_two_token_shards_merge(mode, split):
    layer = W.make_layer(SHAPE)
    (S_all, Sh_all), = run_up(B, DV, SHAPE, layer, mode)
    shards, heads, counts = [], [], []
    for lo, hi in ((0, split), (split, SHAPE.T)):
        shape = SHAPE.scaled(T=hi - lo)
        (S, Sh), = run_up(B, DV, shape, _token_slice(layer, lo, hi), mode)
        shards.append(S)
        heads.append(Sh)
        counts.append(hi - lo)
    S_m = B.combine_shards(shards, counts)
    Sh_m = B.combine_shards(heads, counts)
    if split % 512 == 0:
        np.testing.assert_allclose(S_m, S_all, rtol=MERGE_RTOL[mode], atol=0)
        np.testing.assert_allclose(Sh_m, Sh_all, rtol=MERGE_RTOL[mode], atol=0)
    S_ref, Sh_ref = oracle_up(O, SHAPE, layer, mode)
    assert rel_err(S_m, S_ref) <= TOL and rel_err(Sh_m, Sh_ref) <= TOL


@pytest.mark.parametrize("split", SPLITS)
def test_down_two_token_shards_merge(split):
    layer = W.make_layer(SHAPE, with_next=True)
    S_all, = run_down(B, DV, SHAPE, layer)
    shards, counts = [], []
    for lo, hi in ((0, split), (split, SHAPE.T)):
        (S,) = run_down(B, DV, SHAPE.scaled(T=hi - lo), _token_slice(layer, lo, hi))
        shards.append(S)
        counts.append(hi - lo)
    S_m = B.combine_shards(shards, counts)
    if split % 256 == 0:
        np.testing.assert_allclose(S_m, S_all, rtol=MERGE_RTOL["fo"], atol=0)
    assert rel_err(S_m, oracle_down(O, SHAPE, layer)) <= TOL
