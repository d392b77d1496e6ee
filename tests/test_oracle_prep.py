"""Pins for the oracle's preparation steps: block quantiser, k-means, stable argsort, demeaning.

"VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention", Sec. 3.2 (value-guided
permutation, Eq. 3; block demeaning, Eq. 4; energy identity, Eq. 5; unbalanced clusters);
"Open-VC Attention" (MachGen blog), "Scheduling around ExpCast" (per-128-token Q/K scales,
per-head V scale). Independent references: torch's float8 cast, numpy's stable argsort,
scikit-learn's Lloyd k-means, brute force over all labelings.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle


def bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def f32(u16) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("S,D", [(128, 128), (300, 64), (1, 128), (257, 128)])
def test_quant_blocks_matches_torch(S, D):
    rng = np.random.default_rng(S + D)
    x = rng.normal(0, 2, (S, D)).astype(np.float32)
    x[rng.integers(0, S), rng.integers(0, D)] = 90.0
    xb = bf16(x)
    codes, scales = oracle.quant_blocks(xb)
    nkb = (S + 127) // 128
    assert codes.shape == (nkb * 128, D) and scales.shape == (nkb,)
    xf = f32(xb)
    for j in range(nkb):
        blk = xf[j * 128:(j + 1) * 128]
        amax = np.float32(np.abs(blk).max())
        inv = np.float32(448.0) / amax
        want = torch.from_numpy((blk * inv).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes[j * 128:j * 128 + blk.shape[0]], want)
        assert scales[j] == np.float32(amax / np.float32(448.0))
    assert not codes[S:].any()  # padding rows are zero


def test_quant_blocks_zero_block():
    codes, scales = oracle.quant_blocks(np.zeros((130, 64), dtype=np.uint16))
    assert scales.tolist() == [1.0, 1.0] and not codes.any()


def make_v(S, D, seed=0, k_true=5):
    rng = np.random.default_rng(seed)
    cent = rng.normal(0, 4, (k_true, D))
    lab = rng.integers(0, k_true, S)
    return bf16(cent[lab] + rng.normal(0, 1, (S, D)))


def test_kmeans_matches_sklearn_lloyd():
    skc = pytest.importorskip("sklearn.cluster")
    v = make_v(600, 32, seed=1, k_true=6)
    k, iters = 8, 4
    labels, cent, J = oracle.kmeans(v, k, iters)
    x = f32(v).astype(np.float64)
    init = x[(np.arange(k) * 600 / k).astype(np.int64)]
    # sklearn re-assigns after its last centre update, so its max_iter = iters - 1 gives our labels
    km = skc.KMeans(n_clusters=k, init=init, n_init=1, max_iter=iters - 1, tol=0.0, algorithm="lloyd").fit(x)
    assert np.array_equal(labels, km.labels_.astype(np.int32))


def test_kmeans_objective_non_increasing_and_valid():
    v = make_v(2000, 64, seed=2, k_true=12)
    labels, cent, J = oracle.kmeans(v, 16, 6)
    assert labels.min() >= 0 and labels.max() < 16
    assert np.all(np.diff(J) <= 1e-9 * J[0])
    assert abs(oracle.kmeans_objective(v, 16, labels) - J[-1]) <= 1e-9 * J[-1]


def test_kmeans_degenerate_k():
    v = make_v(300, 16, seed=3)
    labels, _, _ = oracle.kmeans(v, 1, 3)
    assert not labels.any()
    labels, _, J = oracle.kmeans(v, 300, 2)  # every token its own centroid from the initialisation
    assert np.array_equal(labels, np.arange(300)) and J[-1] == 0.0


def test_kmeans_brute_force_tiny():
    rng = np.random.default_rng(4)
    for trial in range(6):
        S = int(rng.integers(4, 11))
        v = bf16(rng.normal(0, 1, (S, 3)) + (np.arange(S)[:, None] % 2) * 6.0 * (trial % 2))
        best = min(oracle.kmeans_objective(v, 2, np.array(lab, dtype=np.int32))
                   for lab in itertools.product([0, 1], repeat=S) if 0 < sum(lab) < S)
        labels, _, J = oracle.kmeans(v, 2, 5)
        assert J[-1] >= best - 1e-9
        if trial % 2 == 1:  # two well-separated groups: Lloyd reaches the optimum
            assert abs(J[-1] - best) <= 1e-9 * max(best, 1.0)


def test_stable_argsort_matches_numpy():
    rng = np.random.default_rng(5)
    for k, S in [(1, 10), (7, 1000), (591, 75600), (64, 8192)]:
        z = rng.integers(0, k, S).astype(np.int32)
        assert np.array_equal(oracle.stable_argsort(z, k), np.argsort(z, kind="stable").astype(np.int32))


def test_gather_rows():
    rng = np.random.default_rng(6)
    x = rng.integers(0, 65535, (50, 16)).astype(np.uint16)
    p = rng.permutation(50).astype(np.int32)
    assert np.array_equal(oracle.gather_rows(x, p), x[p])


@pytest.mark.parametrize("S", [128, 300, 1000])
def test_demean_energy_identity_and_residual(S):
    D = 64
    rng = np.random.default_rng(S)
    v = bf16(rng.normal(2, 3, (S, D)))
    perm = rng.permutation(S).astype(np.int32)
    out = oracle.demean(v, perm)
    vp = f32(v)[perm].astype(np.float64)
    nkb = (S + 127) // 128
    for j in range(nkb):
        blk = vp[j * 128:(j + 1) * 128]
        mu = out["mu"][j]
        assert np.allclose(mu, blk.mean(axis=0), rtol=0, atol=1e-12)  # mean over the valid rows only
        c = rng.normal(0, 1, D)
        lhs = ((blk - c) ** 2).sum()
        rhs = ((blk - mu) ** 2).sum() + blk.shape[0] * ((c - mu) ** 2).sum()
        assert abs(lhs - rhs) <= 1e-9 * lhs  # Eq. 5
        assert np.array_equal(out["mub"][j], oracle.f64_to_bf16(mu))
        resid = out["resid"][j * 128:j * 128 + blk.shape[0]]
        assert np.array_equal(resid, (blk.astype(np.float32) - f32(out["mub"][j])).astype(np.float32))
    amax = np.abs(out["resid"]).max()
    assert out["amax"] == amax and out["sv"] == np.float32(amax / np.float32(448))
    inv = np.float32(448) / np.float32(amax)
    want = torch.from_numpy(out["resid"] * inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(out["rc"], want)


def test_demean_off_is_plain_quantisation():
    rng = np.random.default_rng(9)
    v = bf16(rng.normal(0, 1, (200, 32)))
    out = oracle.demean(v, None, subtract_mean=False)
    assert not out["mu"].any() and not out["mub"].any()
    assert np.array_equal(out["resid"][:200], f32(v))


def test_visit_order():
    for nkb in [1, 2, 5, 64, 591]:
        for qt in sorted({0, 1, nkb // 2, max(nkb - 3, 0), nkb - 1}):
            o = oracle.visit_order(nkb, qt, True)
            assert sorted(o.tolist()) == list(range(nkb))
            start = min(nkb - 1, 2 * (qt // 2) + 2)  # shared by the query tiles 2m and 2m+1
            assert o[0] == start
            assert o[:start + 1].tolist() == list(range(start, -1, -1))
            assert o[start + 1:].tolist() == list(range(start + 1, nkb))
        assert oracle.visit_order(nkb, 0, False).tolist() == list(range(nkb))
