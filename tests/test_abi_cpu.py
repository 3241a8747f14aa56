"""The C ABI without a GPU: the library loads and exports every entry point
include/affinity.h declares, argument validation returns the documented codes
before touching a device, and the host-only helpers (partition scoring, group
gain, objective J) agree with the oracle exactly."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import partitions as P
from transformer_sharding_affinity_gb300 import binding as B
from transformer_sharding_affinity_gb300 import build as BUILD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        BUILD.build()
    return B.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "affinity.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"AFF_API\s+[\w\s\*]+?\b(affinity_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/affinity.h but not exported"


def test_version_and_strerror(lib):
    assert B.version() >= 100
    for code in range(0, 10):
        assert len(B.strerror(code)) > 0
    assert B.strerror(123) == "unknown status"


def _d(**kw):
    base = dict(T=256, D=64, H=4, G=2, d_head=16, I=128, eps=1e-6, dtype=B.AFF_BF16)
    base.update(kw)
    return B.dims(**base)


def _ws(d, mode=0, down=0):
    n = ctypes.c_size_t(0)
    st = B.load().affinity_workspace_size(ctypes.byref(d), mode, down, ctypes.byref(n))
    return st, n.value


def test_workspace_size(lib):
    st, n_fo = _ws(_d())
    assert st == B.AFF_OK and n_fo > 0 and n_fo % 1024 == 0
    st, n_add = _ws(_d(flags=B.AFF_FLAG_ADD_DIRECT), 1)
    assert st == B.AFF_OK and 0 < n_add < n_fo          # ADD needs no operating point / Wd norms
    st, n_add_m = _ws(_d(), 1)                           # second-moment form: 128 x 128 per head and chunk
    assert st == B.AFF_OK and n_add_m > 0 and n_add_m % 1024 == 0
    st, n_dn = _ws(_d(), 0, 1)
    assert st == B.AFF_OK and n_dn > 0
    st, n_big = _ws(_d(T=65536, D=1024, H=16, G=8, d_head=128, I=3072))
    assert st == B.AFF_OK and n_big > 400 * 2**20
    st, n_f32 = _ws(_d(dtype=B.AFF_FP32))
    assert st == B.AFF_OK and n_f32 > 0


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), B.AFF_ERR_INVALID_ARG),
    (dict(I=-1), B.AFF_ERR_INVALID_ARG),
    (dict(H=3, G=2), B.AFF_ERR_UNSUPPORTED_SHAPE),
    (dict(D=60), B.AFF_ERR_UNSUPPORTED_SHAPE),
    (dict(d_head=12), B.AFF_ERR_UNSUPPORTED_SHAPE),
    (dict(I=100), B.AFF_ERR_UNSUPPORTED_SHAPE),
    (dict(H=256, G=1), B.AFF_ERR_UNSUPPORTED_SHAPE),
    (dict(dtype=7), B.AFF_ERR_UNSUPPORTED_DTYPE),
    (dict(eps=float("nan")), B.AFF_ERR_INVALID_ARG),
    (dict(eps=-1.0), B.AFF_ERR_INVALID_ARG),
])
def test_bad_dims(lib, kw, code):
    assert _ws(_d(**kw))[0] == code


def test_flag_constant_matches_header(lib):
    src = open(os.path.join(ROOT, "include", "affinity.h")).read()
    m = re.search(r"#define\s+AFF_FLAG_ADD_DIRECT\s+(\d+)u", src)
    assert m and int(m.group(1)) == B.AFF_FLAG_ADD_DIRECT


def test_add_forms_size_their_own_workspace(lib):
    """The second-moment ADD form keeps one d_head x d_head matrix per head (and
    per token chunk) instead of the direct form's per-chunk neuron partials."""
    d = _d(T=65536, D=1024, H=16, G=8, d_head=128, I=3072)
    st, moment = _ws(d, B.AFF_MODE_ADD)
    d.flags = B.AFF_FLAG_ADD_DIRECT
    st2, direct = _ws(d, B.AFF_MODE_ADD)
    assert st == st2 == B.AFF_OK and moment < direct
    # d_head > 128 has no second-moment form: the flag changes nothing
    w = _d(T=4096, D=512, H=2, G=2, d_head=256, I=264)
    a = _ws(w, B.AFF_MODE_ADD)
    w.flags = B.AFF_FLAG_ADD_DIRECT
    assert _ws(w, B.AFF_MODE_ADD) == a


def test_fp32_relaxes_alignment_constraints(lib):
    assert _ws(_d(D=60, d_head=12, I=100, dtype=B.AFF_FP32))[0] == B.AFF_OK


def test_flags_and_mode_are_checked(lib):
    d = _d()
    d.flags = B.AFF_FLAG_ADD_DIRECT
    assert _ws(d, B.AFF_MODE_ADD)[0] == B.AFF_OK
    for bad in (2, 1 << 31, B.AFF_FLAG_ADD_DIRECT | 4):
        d.flags = bad
        assert _ws(d)[0] == B.AFF_ERR_INVALID_ARG
    assert _ws(_d(), 5)[0] == B.AFF_ERR_INVALID_ARG


def _up(lib, d, ptrs, mode=0, ws=1 << 20, ws_bytes=1 << 40, S=1 << 20):
    return lib.affinity_up(*ptrs, ctypes.byref(d), mode, S, None, ws, ws_bytes, None)


def test_up_argument_errors_before_any_launch(lib):
    d = _d()
    good = [0x10000 * (i + 1) for i in range(7)]
    assert _up(lib, d, [None] + good[1:]) == B.AFF_ERR_INVALID_ARG
    assert _up(lib, d, good, S=None) == B.AFF_ERR_INVALID_ARG
    assert _up(lib, d, good[:6] + [None]) == B.AFF_ERR_INVALID_ARG            # FO reads Wd
    assert _up(lib, d, good[:1] + [good[1] + 8] + good[2:]) == B.AFF_ERR_ALIGNMENT
    assert _up(lib, d, good, ws=None) == B.AFF_ERR_WORKSPACE
    assert _up(lib, d, good, ws=(1 << 20) + 128) == B.AFF_ERR_WORKSPACE       # 256-byte alignment
    assert _up(lib, d, good, ws_bytes=1024) == B.AFF_ERR_WORKSPACE
    assert _up(lib, d, good, mode=3) == B.AFF_ERR_INVALID_ARG
    bad = _d(T=0)
    assert _up(lib, bad, good) == B.AFF_ERR_INVALID_ARG


def test_up_without_a_device_reports_arch(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    d = _d()
    good = [0x10000 * (i + 1) for i in range(7)]
    assert _up(lib, d, good) == B.AFF_ERR_ARCH


def test_down_argument_errors(lib):
    d = _d()
    good = [0x10000 * (i + 1) for i in range(9)]
    f = lib.affinity_down
    assert f(*([None] + good[1:]), ctypes.byref(d), 1 << 20, 1 << 20, 1 << 40, None) == B.AFF_ERR_INVALID_ARG
    assert f(*good, ctypes.byref(d), None, 1 << 20, 1 << 40, None) == B.AFF_ERR_INVALID_ARG
    assert f(*good, ctypes.byref(d), (1 << 20) + 4, 1 << 20, 1 << 40, None) == B.AFF_ERR_ALIGNMENT
    assert f(*good, ctypes.byref(d), 1 << 20, 1 << 20, 16, None) == B.AFF_ERR_WORKSPACE


# ---------------------------------------------------------------- host helpers vs the oracle

@pytest.mark.parametrize("G,L", [(8, 4), (8, 2), (6, 3), (4, 4), (4, 1), (12, 4), (10, 5)])
def test_score_partitions_matches_oracle(lib, G, L):
    rng = np.random.default_rng(G * 100 + L)
    C = rng.random((G, L))
    scores, count, best, assign = B.score_partitions(C)
    assert count == P.partition_count(G, L)
    o_scores, o_best, o_assign = P.score_partitions(C)
    np.testing.assert_array_equal(scores, o_scores)
    assert best == o_best and assign == tuple(o_assign)


def test_score_partitions_paper_count_and_ties(lib):
    scores, count, best, assign = B.score_partitions(np.zeros((8, 4)))
    assert count == 2520 and best == 0 and assign == (0, 0, 1, 1, 2, 2, 3, 3)
    for G, L in [(0, 1), (8, 3), (4, 8), (17, 1)]:
        cnt, bi = ctypes.c_int64(0), ctypes.c_int64(0)
        C = np.zeros((max(G, 1), max(L, 1)))
        assert lib.affinity_score_partitions(C.ctypes.data, G, L, None, ctypes.byref(cnt), ctypes.byref(bi),
                                             None) == B.AFF_ERR_INVALID_ARG
    C = np.zeros((16, 8))   # 16!/2^8 ~ 8e10 partitions: refused
    assert lib.affinity_score_partitions(C.ctypes.data, 16, 8, None, ctypes.byref(cnt), ctypes.byref(bi),
                                         None) == B.AFF_ERR_UNSUPPORTED_SHAPE


def test_group_gain_and_objective_match_oracle(lib):
    rng = np.random.default_rng(3)
    N, G, I, L = 4, 8, 64, 4
    ups = [P.unit_mass(rng.random((G, I))) for _ in range(N)]
    downs = [P.unit_mass(rng.random((I, G))) for _ in range(N - 1)]
    hs = [rng.permutation(P.contiguous_heads(G, L)) for _ in range(N)]
    ns = [rng.permutation(P.contiguous_neurons(I, L)) for _ in range(N)]
    np.testing.assert_allclose(B.objective(ups, downs, hs, ns), P.objective_J(ups, downs, hs, ns), rtol=1e-13)
    for i in range(N):
        got = B.group_gain(ups[i], ns[i], L, downs[i - 1] if i else None, ns[i - 1] if i else None)
        ref = P.group_gain(ups[i], L, ns[i], downs[i - 1] if i else None, ns[i - 1] if i else None)
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-16)
    bad = np.array(ns[0])
    bad[0] = L
    with pytest.raises(B.AffinityError):
        B.group_gain(ups[0], bad, L)


def test_unit_mass_matches_oracle(lib):
    rng = np.random.default_rng(4)
    S = rng.random((8, 96)).astype(np.float32)
    np.testing.assert_allclose(B.unit_mass(S), P.unit_mass(S.astype(np.float64)), rtol=1e-14)
    assert abs(B.unit_mass(S).sum() - 1.0) < 1e-12
    for bad in (np.zeros((2, 3), np.float32), np.full((2, 2), np.inf, np.float32)):
        with pytest.raises(B.AffinityError):
            B.unit_mass(bad)


def test_best_heads_is_the_brute_force_optimum(lib):
    """With nu fixed, the per-layer partition choice maximises J over every
    combination of balanced head maps (brute force over all N-tuples)."""
    import itertools
    rng = np.random.default_rng(6)
    N, G, I, L = 3, 4, 12, 2
    ups = [P.unit_mass(rng.random((G, I))) for _ in range(N)]
    downs = [P.unit_mass(rng.random((I, G))) for _ in range(N - 1)]
    ns = [rng.permutation(P.contiguous_neurons(I, L)) for _ in range(N)]
    h, J = B.best_heads(ups, downs, ns, L)
    maps = P.balanced_partitions(G, L)
    best = max(P.objective_J(ups, downs, list(hs), ns) for hs in itertools.product(maps, repeat=N))
    np.testing.assert_allclose(J, best, rtol=1e-13)
    np.testing.assert_allclose(J, P.objective_J(ups, downs, list(h), ns), rtol=1e-13)
    # per layer it is the oracle's partition choice on the oracle's gain
    for i in range(N):
        C = P.group_gain(ups[i], L, ns[i], downs[i - 1] if i else None, ns[i - 1] if i else None)
        assert tuple(h[i]) == tuple(P.score_partitions(C)[2])


def test_combine_shards_is_the_token_weighted_mean(lib):
    rng = np.random.default_rng(8)
    S = [rng.random((4, 10)).astype(np.float32) for _ in range(3)]
    T = [100, 0, 37]
    got = B.combine_shards(S, T)
    ref = (100 * S[0].astype(np.float64) + 37 * S[2]) / 137
    np.testing.assert_allclose(got, ref, rtol=1e-7)
    np.testing.assert_array_equal(B.combine_shards([S[0]], [5]), S[0])
    for bad_T in ([0, 0, 0], [1, -1, 1]):
        with pytest.raises(B.AffinityError):
            B.combine_shards(S, bad_T)


# ---------------------------------------------------------------- layout search: validation before any device use

def test_layout_search_argument_checks(lib):
    P_ = ctypes.c_void_p
    fake = P_(1 << 20)          # never dereferenced: every check below fails before a device is touched
    h = np.zeros(8, np.int32)
    h4 = (np.arange(8) // 2).astype(np.int32)
    assert lib.affinity_neuron_gain(fake, None, h4.ctypes.data, None, 8, 64, 9, fake, None) == \
        B.AFF_ERR_UNSUPPORTED_SHAPE
    assert lib.affinity_neuron_gain(fake, None, h4.ctypes.data, None, 17, 64, 4, fake, None) == B.AFF_ERR_INVALID_ARG
    bad = h4.copy()
    bad[0] = 4
    assert lib.affinity_neuron_gain(fake, None, bad.ctypes.data, None, 8, 64, 4, fake, None) == B.AFF_ERR_INVALID_ARG
    assert lib.affinity_neuron_gain(fake, fake, h4.ctypes.data, None, 8, 64, 4, fake, None) == B.AFF_ERR_INVALID_ARG
    assert lib.affinity_neuron_gain(fake, None, h4.ctypes.data, None, 8, 64, 4, fake, None) == B.AFF_ERR_ARCH

    def assign(I, L, ws=fake, nbytes=256):
        return lib.affinity_assign_neurons(fake, 1, I, L, None, fake, fake, ws, nbytes, None)
    assert assign(66, 4) == B.AFF_ERR_UNSUPPORTED_SHAPE
    assert assign(49152 + 4, 4) == B.AFF_ERR_UNSUPPORTED_SHAPE
    assert assign(64, 9) == B.AFF_ERR_UNSUPPORTED_SHAPE
    assert assign(64, 4, nbytes=128) == B.AFF_ERR_WORKSPACE
    assert assign(64, 4, ws=P_((1 << 20) + 8)) == B.AFF_ERR_WORKSPACE
    assert assign(64, 4) == B.AFF_ERR_ARCH

    n = B.layout_workspace_size(28, 8, 3072, 4)
    assert n >= 28 * 8 * 3072 * 8 * 2 + 28 * 3072 * 4 * 8
    with pytest.raises(B.AffinityError):
        B.layout_workspace_size(2, 6, 64, 4)      # G % L != 0
    N, G, I, L = 2, 8, 64, 4
    up = np.full((N, G, I), 1.0 / (G * I))
    dn = np.full((N - 1, I, G), 1.0 / (G * I))
    hh = np.stack([h4] * N).astype(np.int32)
    nn = np.stack([(np.arange(I) // (I // L)).astype(np.int32)] * N)
    J, sw = ctypes.c_double(0), ctypes.c_int32(0)
    ws_n = B.layout_workspace_size(N, G, I, L)

    def opt(hmap, numap, nbytes=ws_n):
        return lib.affinity_optimise_layout(up.ctypes.data, dn.ctypes.data, N, G, I, L, None, hmap.ctypes.data,
                                            numap.ctypes.data, ctypes.byref(J), ctypes.byref(sw), fake, nbytes, None)
    unbalanced = hh.copy()
    unbalanced[0, 0] = 1
    assert opt(unbalanced, nn) == B.AFF_ERR_INVALID_ARG
    assert opt(hh, nn, nbytes=ws_n - 1) == B.AFF_ERR_WORKSPACE
    assert opt(hh, nn) == B.AFF_ERR_ARCH
    assert h.sum() == 0


def test_layout_orders_match_the_oracle_and_gather_checks(lib):
    from oracle import layer_forward as LF
    rng = np.random.default_rng(13)
    G, H, I, L, dh = 8, 16, 96, 4, 4
    h = rng.permutation(P.contiguous_heads(G, L)).astype(np.int32)
    nu = rng.permutation(P.contiguous_neurons(I, L)).astype(np.int32)
    go, ho, no = B.layout_orders(h, nu, H, L)
    w = {k: np.zeros((1, 1)) for k in ()}
    shapes = {"Wq": (H * dh, 8), "Wk": (G * dh, 8), "Wv": (G * dh, 8), "Wo": (8, H * dh), "Wg": (I, 8),
              "Wu": (I, 8), "Wd": (8, I)}
    w = {k: rng.standard_normal(s) for k, s in shapes.items()}
    _, rgo, rho, rno = LF.realise(w, h, nu, H, G, dh, L)
    np.testing.assert_array_equal(go, rgo)
    np.testing.assert_array_equal(ho, rho)
    np.testing.assert_array_equal(no, rno)
    bad = h.copy()
    bad[0] = (bad[0] + 1) % L
    with pytest.raises(B.AffinityError):
        B.layout_orders(bad, nu, H, L)
    fake = ctypes.c_void_p(1 << 20)
    other = ctypes.c_void_p(1 << 24)
    o = np.array([0, 2, 2, 1], np.int32)       # not a permutation
    assert lib.affinity_gather_blocks(fake, other, 1, 4, 16, o.ctypes.data, fake, 256, None) == \
        B.AFF_ERR_INVALID_ARG
    o = np.array([0, 2, 3, 1], np.int32)
    assert lib.affinity_gather_blocks(fake, fake, 1, 4, 16, o.ctypes.data, other, 256, None) == \
        B.AFF_ERR_INVALID_ARG                   # in and out overlap
    assert lib.affinity_gather_blocks(fake, other, 1, 4, 16, o.ctypes.data, other, 8, None) == B.AFF_ERR_WORKSPACE
    assert lib.affinity_gather_blocks(fake, other, 1, 4, 16, o.ctypes.data, ctypes.c_void_p(1 << 28), 256,
                                      None) == B.AFF_ERR_ARCH


def test_loo_mode_is_bf16_only(lib):
    d = B.dims(256, 64, 4, 2, 16, 128, 1e-6, B.AFF_FP32)
    n = ctypes.c_size_t(0)
    assert lib.affinity_workspace_size(ctypes.byref(d), B.AFF_MODE_LOO, 0, ctypes.byref(n)) == \
        B.AFF_ERR_UNSUPPORTED_DTYPE
    db = B.dims(256, 64, 4, 2, 16, 128, 1e-6, B.AFF_BF16, B.AFF_FLAG_ADD_DIRECT)
    assert B.workspace_size(db, B.AFF_MODE_LOO) > B.workspace_size(db, B.AFF_MODE_ADD)


def test_selftest_timeout_argument_checks(lib):
    fake = ctypes.c_void_p(1 << 20)
    assert lib.affinity_selftest_timeout(fake, 128, 5_000_000, None) == B.AFF_ERR_WORKSPACE
    assert lib.affinity_selftest_timeout(ctypes.c_void_p((1 << 20) + 16), 256, 5_000_000, None) == B.AFF_ERR_WORKSPACE
    assert lib.affinity_selftest_timeout(fake, 256, 10, None) == B.AFF_ERR_INVALID_ARG
    assert lib.affinity_selftest_timeout(fake, 256, 5_000_000, None) == B.AFF_ERR_ARCH
