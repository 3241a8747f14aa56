"""Token-sharded calibration across two processes (``gloo`` on CPU).

Each rank computes S_up (FO and ADD) and S_down on its own contiguous shard of
the calibration tokens -- with the oracle, since this host has no GPU -- and
the library's exchange step merges the shards.  The merged matrices must
equal the oracle on all tokens ("Affinity-Aware Sharding for Delayed Tensor
Parallelism", §3 "Affinity scores": every entry is a token mean times a
per-neuron factor) and be bit-identical on both ranks."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from oracle import affinity_oracle as O  # noqa: E402
from transformer_sharding_affinity_gb300 import shards  # noqa: E402
from transformer_sharding_affinity_gb300 import workloads as W  # noqa: E402

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard_scores(shape, layer, lo, hi):
    sl = lambda t: t[lo:hi]  # noqa: E731
    out = {}
    for mode in ("fo", "add"):
        S, Sh = O.s_up(sl(layer["a"]), sl(layer["x"]), layer["Wo"], layer["gamma"], layer["Wg"], layer["Wu"],
                       layer["Wd"], shape.H, shape.G, shape.dh, shape.eps, mode)
        out[mode] = S
        out[mode + "_head"] = Sh
    out["down"] = O.s_down(sl(layer["x"]), layer["gamma"], layer["Wg"], layer["Wu"], layer["Wd"],
                           layer["gamma_next"], layer["Wq_next"], layer["Wk_next"], layer["Wv_next"], shape.H,
                           shape.G, shape.dh, shape.eps)
    return out


def _rank_main(rank, port, T, outdir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        shape = W.CONFIGS["tiny"].scaled(T=T)
        layer = W.make_layer(shape, with_next=True)
        lo, hi = shards.token_range(T, rank, WORLD)
        local = _shard_scores(shape, layer, lo, hi)
        merged = {k: shards.allgather_combine(torch.from_numpy(v.astype(np.float32)), hi - lo)
                  for k, v in local.items()}
        np.savez(os.path.join(outdir, f"rank{rank}.npz"), **merged)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("T", [256, 301])
def test_two_rank_token_shards_merge_to_the_full_pass(tmp_path, T):
    mp.start_processes(_rank_main, args=(_free_port(), T, str(tmp_path)), nprocs=WORLD, join=True,
                       start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npz")
    r1 = np.load(tmp_path / "rank1.npz")
    shape = W.CONFIGS["tiny"].scaled(T=T)
    layer = W.make_layer(shape, with_next=True)
    full = _shard_scores(shape, layer, 0, T)
    for k, ref in full.items():
        assert np.array_equal(r0[k].view(np.uint32), r1[k].view(np.uint32)), f"{k}: ranks disagree"
        # fp32 shard values merged in fp64: a few fp32 ulps from the full-set value
        np.testing.assert_allclose(r0[k], ref, rtol=1e-6, atol=0, err_msg=k)


def test_token_range_covers_every_token_once():
    for T in (0, 1, 7, 256, 1001):
        for world in (1, 2, 3, 8):
            ranges = [shards.token_range(T, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == T
            for (a, b), (c, d) in zip(ranges, ranges[1:]):
                assert b == c
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shards.token_range(10, 2, 2)
