"""Pins for the oracle's attention: the exact fp64 forward (ii) and the quantised forward (i).

"VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention": Sec. 3.1 Eq. 1 (online
softmax), Sec. 3.2 Eq. 3 (P'V' = PV), Eq. 6 (online mean restoration), Sec. 3.3 Eq. 7 and Prop. 3.1
(row guarantee); "Open-VC Attention" (MachGen blog), "Scheduling around ExpCast" (true-score max,
consistent denominator, mid-window order). Independent references: torch.softmax in fp64, a
closed-form restatement of the tiled recurrence written here with per-tile weights instead of a
running rescale, and the Prop. 3.1 bound.
"""
import math

import numpy as np
import pytest
import torch

import oracle

LOG2E = 1.4426950408889634


def bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def f64(u16) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dec(codes) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def test_exact_matches_torch_softmax():
    rng = np.random.default_rng(0)
    S, D = 300, 64
    q, k, v = (bf16(rng.normal(0, 1.5, (S, D))) for _ in range(3))
    rows = np.arange(S)
    ours = oracle.attention_exact(q, k, v, rows)
    Q, K, V = (torch.from_numpy(f64(x)) for x in (q, k, v))
    ref = torch.softmax(Q @ K.T / math.sqrt(D), dim=-1) @ V
    assert np.abs(ours - ref.numpy()).max() < 1e-12


def test_permutation_invariance():
    rng = np.random.default_rng(1)
    S, D = 500, 32
    q, k, v = (bf16(rng.normal(0, 2, (S, D))) for _ in range(3))
    perm = rng.permutation(S)
    rows = rng.choice(S, 40, replace=False)
    a = oracle.attention_exact(q, k, v, rows)
    b = oracle.attention_exact(q, k[perm], v[perm], rows)
    assert np.abs(a - b).max() < 1e-12


@pytest.mark.parametrize("S,midwindow", [(300, True), (300, False), (1000, True), (128, True)])
def test_mean_restoration_identity(S, midwindow):
    """Tiled recurrence on demeaned fp64 values with exact exp reproduces exact attention."""
    rng = np.random.default_rng(S)
    D = 32
    q, k, v = (bf16(rng.normal(0, 2, (S, D))) for _ in range(3))
    v = bf16(f64(v) + 10.0 * rng.normal(0, 1, (1, D)))  # a large common component worth removing
    perm = rng.permutation(S)
    rows = rng.choice(S, 60, replace=False)
    ref = oracle.attention_exact(q, k, v, rows)
    ours = oracle.attention_demeaned_exact(f64(q), f64(k)[perm], f64(v)[perm], rows, midwindow)
    assert np.abs(ours - ref).max() < 1e-10 * np.abs(ref).max()


def fma32(a, b, c):
    """Single-rounded fp32 a*b+c: the product is exact in long double and so is the sum here."""
    r = np.longdouble(np.float32(a)) * np.longdouble(np.float32(b)) + np.longdouble(np.float32(c))
    return np.float32(r)


def closed_form(prep, r, expcast=True, midwindow=True, with_mean=True):
    """Quantised forward of one row restated with per-tile weights 2^((M_j - M_final)/8)."""
    S, D = prep["S"], prep["D"]
    nkb = (S + 127) // 128
    qt = r // 128
    order = list(range(nkb))
    if midwindow:
        st = min(nkb - 1, 2 * (qt // 2) + 2)  # the pair of query tiles (2m, 2m+1) starts at 2m+2
        order = list(range(st, -1, -1)) + list(range(st + 1, nkb))
    C = np.float32(8.0 * LOG2E / math.sqrt(D))
    aq = np.float32(C * prep["sq"][qt])
    qd = dec(prep["qc"][r])
    M = -np.inf
    tiles = []
    for j in order:
        n = min(128, S - 128 * j)
        kd = dec(prep["kc"][128 * j:128 * j + n])
        s32 = (kd @ qd).astype(np.float32)  # exact in fp64 then one rounding
        aj = np.float32(aq * prep["sk"][j])
        t = np.max((s32 * aj).astype(np.float32))
        M = max(M, t)
        b = np.float32(np.float32(119.65) - np.float32(M))
        y = np.array([fma32(x, aj, b) for x in s32], dtype=np.float32)
        if expcast:
            code = np.clip(np.rint(y), 0, 120).astype(np.uint8)
        else:
            ze = ((y - np.float32(119.65)) * np.float32(0.125) + np.float32(8.0)).astype(np.float32)
            p = np.exp2(ze.astype(np.float64)).astype(np.float32)
            code = torch.from_numpy(p).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        ph = dec(code)
        vals = dec(prep["rc"][128 * j:128 * j + n]) * prep["sv"]
        if with_mean:
            vals = vals + f64(prep["mub"][j])[None, :]
        tiles.append((np.float32(M), ph, vals))
    Mf = tiles[-1][0]
    num = sum(2.0 ** ((float(Mj) - float(Mf)) / 8) * (ph @ vals) for Mj, ph, vals in tiles)
    den = sum(2.0 ** ((float(Mj) - float(Mf)) / 8) * ph.sum() for Mj, ph, vals in tiles)
    return num / den


@pytest.mark.parametrize("S,vsmooth,expcast,midwindow", [
    (100, True, True, True),      # one ragged key tile
    (128, False, True, True),
    (300, True, True, True),      # three tiles, ragged tail
    (300, True, True, False),
    (300, True, False, True),     # exponentiate-then-cast path
    (520, False, True, True),
])
def test_quantised_forward_matches_closed_form(S, vsmooth, expcast, midwindow):
    rng = np.random.default_rng(S * 7 + vsmooth)
    D = 64
    q = bf16(rng.normal(0, 1.2, (S, D)))
    k = bf16(rng.normal(0, 1.2, (S, D)))
    v = bf16(rng.normal(1.0, 2.0, (S, D)))
    prep = oracle.prepare_head(q, k, v, k_clusters=max(1, S // 128), iters=2, vsmooth=vsmooth)
    rows = np.unique(np.concatenate([[0, S - 1], rng.choice(S, 10, replace=False)]))
    out, l, m = oracle.forward_head(prep, rows, expcast=expcast, midwindow=midwindow)
    for i, r in enumerate(rows):
        want = closed_form(prep, int(r), expcast, midwindow, with_mean=vsmooth)
        assert np.abs(out[i] - want).max() <= 1e-9 * max(1.0, np.abs(want).max())


def exact_grid_inputs(S, D, rng, qk_pow=-4, v_pow=-6):
    """Q, K, V whose per-block (Q, K) and per-head (V) quantisation is exact: every value is an
    E4M3 value times 2^pow and every block holds an entry of magnitude 448*2^pow (score std ~1)."""
    grid = dec(np.arange(256, dtype=np.uint8))
    ok = np.isfinite(grid) & (np.abs(grid) <= 448)
    vals = grid[ok]
    small = vals[np.abs(vals) <= 64]

    def make(p):
        x = rng.choice(small, size=(S, D)) * 2.0 ** p
        for j in range(0, S, 128):
            x[j, rng.integers(0, D)] = 448 * 2.0 ** p * rng.choice([-1, 1])
        return x
    return bf16(make(qk_pow)), bf16(make(qk_pow)), bf16(make(v_pow))


@pytest.mark.parametrize("midwindow", [True, False])
def test_prop31_on_full_path(midwindow):
    """With exact Q/K/V quantisation the only error left is the probability path: Prop. 3.1."""
    rng = np.random.default_rng(11)
    S, D = 700, 64
    q, k, v = exact_grid_inputs(S, D, rng)
    prep = oracle.prepare_head(q, k, v, 1, 1, vsmooth=False)
    assert np.array_equal(dec(prep["rc"][:S]) * prep["sv"], f64(v))  # V exact
    rows = np.arange(0, S, 7)
    out, _, _ = oracle.forward_head(prep, rows, expcast=True, midwindow=midwindow)
    ref = oracle.attention_exact(q, k, v, rows)
    V = f64(v)
    diam = max(np.linalg.norm(V[i] - V, axis=1).max() for i in range(S))
    Q, K = f64(q), f64(k)
    for i, r in enumerate(rows):
        s = K @ Q[r] / math.sqrt(D)
        u = (s - s.max()) * LOG2E
        p = np.exp(s - s.max())
        p /= p.sum()
        # p_hat(T): each tail weight is below 2^-6 * 1.0746 and the row max codes to 256
        tau = max(p[u < -14].sum(), (u < -14).sum() * 2.0**-6 * 1.0746 / 256)
        err = np.linalg.norm(out[i] - ref[i])
        assert err <= (0.0364 + tau) * diam + 1e-9


def test_exp_then_cast_bound_on_full_path():
    """Exponentiate-then-cast: each weight within half an E4M3 step (ratio in [15/16, 17/16])."""
    rng = np.random.default_rng(12)
    S, D = 400, 64
    q, k, v = exact_grid_inputs(S, D, rng)
    prep = oracle.prepare_head(q, k, v, 1, 1, vsmooth=False)
    rows = np.arange(0, S, 5)
    out, _, _ = oracle.forward_head(prep, rows, expcast=False, midwindow=True)
    ref = oracle.attention_exact(q, k, v, rows)
    a, b = 15 / 16, 17 / 16
    bound = (math.sqrt(b) - math.sqrt(a)) / (math.sqrt(b) + math.sqrt(a))
    V = f64(v)
    diam = max(np.linalg.norm(V[i] - V, axis=1).max() for i in range(S))
    Q, K = f64(q), f64(k)
    for i, r in enumerate(rows):
        s = K @ Q[r] / math.sqrt(D)
        u = (s - s.max()) * LOG2E
        p = np.exp(s - s.max())
        p /= p.sum()
        tau = max(p[u < -14].sum(), (u < -14).sum() * 2.0**-6 * b / 256)
        assert np.linalg.norm(out[i] - ref[i]) <= (bound + tau) * diam + 1e-9


def test_mean_restoration_on_quantised_path():
    """Blocks = bf16 mean + exactly quantisable residual: restoring the mean gives the weighted
    average of V' itself, so (i) with the mean term equals the closed form on V' = R + mu."""
    rng = np.random.default_rng(13)
    S, D = 384, 32
    q = bf16(rng.normal(0, 1, (S, D)))
    k = bf16(rng.normal(0, 1, (S, D)))
    levels = np.array([0.5, 1.0, 2.0, 4.0, 7.0])
    R = np.zeros((S, D))
    for j in range(0, S, 128):
        half = rng.choice(levels, size=(64, D)) * rng.choice([-1, 1], size=(64, D))
        R[j:j + 128] = np.concatenate([half, -half])  # zero block mean
    R[0, 0], R[64, 0] = 7.0, -7.0
    mu = np.round(rng.normal(0, 4, (S // 128, D)) * 2) / 2
    v = bf16(R + np.repeat(mu, 128, axis=0))
    prep = oracle.prepare_head(q, k, v, 1, 1, vsmooth=True, perm=np.arange(S))
    assert np.array_equal(f64(prep["mub"]), mu)
    assert np.array_equal(dec(prep["rc"][:S]) * prep["sv"], R)
    rows = rng.choice(S, 16, replace=False)
    out, _, _ = oracle.forward_head(prep, rows)
    for i, r in enumerate(rows):
        want = closed_form(prep, int(r), with_mean=True)
        assert np.abs(out[i] - want).max() <= 1e-10 * np.abs(want).max()
    # and dropping the mean term is visibly wrong (the pin is not vacuous)
    prep_nomean = dict(prep, vsmooth=False)
    bad, _, _ = oracle.forward_head(prep_nomean, rows)
    assert np.abs(bad - out).max() > 0.1


@pytest.mark.parametrize("nkb", [1, 2, 3, 7, 64])
def test_visit_order_reading(nkb):
    """Mid-window key traversal ("Open-VC Attention", "Scheduling around ExpCast"): every key tile once,
    starting a few tiles past the query tile's diagonal, down to tile 0, then the tail in order. Reading:
    the pair of query tiles (2m, 2m+1) starts at min(nkb-1, 2m+2), so both tiles of a pair share one order."""
    for qt in range(nkb):
        o = oracle.visit_order(nkb, qt)
        start = min(nkb - 1, 2 * (qt // 2) + 2)
        assert sorted(o.tolist()) == list(range(nkb))
        assert o[0] == start and start >= min(nkb - 1, qt + 1)
        assert o.tolist() == list(range(start, -1, -1)) + list(range(start + 1, nkb))
        assert np.array_equal(o, oracle.visit_order(nkb, qt ^ 1)) or (qt ^ 1) >= nkb
        assert np.array_equal(oracle.visit_order(nkb, qt, midwindow=False), np.arange(nkb))
