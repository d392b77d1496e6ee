"""Oracle pins of the V residual repair ("Open-VC Attention", "Why V residual repair": the tokens of
largest residual energy become extra FP8 value rows, each paired with a copy of its key, visited last,
adding to the numerator only).

Independent references: residual energies recomputed here in fp64 with torch's E4M3 cast, the E4M3
rounding bound, the denominator and running max left unchanged, exactly representable values
(nothing to repair), a closed form of the forward with per-tile weights, and exact fp64 attention.
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


def heavy_v(S, D, rng):
    """Values with a heavy tail: a few tokens carry large magnitudes, and so large rounding residuals."""
    v = rng.normal(0, 1, (S, D))
    v[rng.choice(S, max(1, S // 50), replace=False)] *= 12.0
    return bf16(v)


def residual_energy64(v, amax):
    """sum_c (s_c (x - dec(E4M3(x))))^2 in fp64, x = fl32(v * fl32(448 / amax))."""
    a = np.asarray(amax, dtype=np.float32)
    inv = np.where(a > 0, np.float32(448) / np.where(a > 0, a, 1), np.float32(1)).astype(np.float32)
    s = np.where(a > 0, a / np.float32(448), np.float32(1)).astype(np.float32)
    x = (f64(v).astype(np.float32) * inv[None, :]).astype(np.float32)
    xd = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    r = (x.astype(np.float64) - xd) * s[None, :].astype(np.float64)
    return (r * r).sum(axis=1), x.astype(np.float64) - xd


@pytest.mark.parametrize("S,D,n", [(300, 64, 7), (1000, 128, 128), (257, 64, 200), (129, 32, 129)])
def test_selection_is_the_top_energy_tokens(S, D, n):
    rng = np.random.default_rng(S + n)
    v = heavy_v(S, D, rng)
    amax = np.full(D, np.abs(f64(v)).max(), dtype=np.float32)
    idx, energy, _ = oracle.repair_select(v, amax, n)
    assert idx.shape == (n,) and np.all(np.diff(idx) > 0) and idx.min() >= 0 and idx.max() < S
    e64, _ = residual_energy64(v, amax)
    assert np.allclose(energy, e64, rtol=1e-5, atol=0)
    sel = np.zeros(S, dtype=bool)
    sel[idx] = True
    if n < S:
        assert e64[sel].min() >= e64[~sel].max() * (1 - 1e-5)


def test_selection_ties_go_to_the_lower_index():
    """Identical rows have identical energies: the earliest ones are kept."""
    rng = np.random.default_rng(1)
    row = rng.normal(0, 3, 32)
    v = bf16(np.tile(row, (50, 1)))
    idx, _, _ = oracle.repair_select(v, np.full(32, np.abs(f64(v)).max(), dtype=np.float32), 9)
    assert idx.tolist() == list(range(9))


def test_repair_codes_are_the_rounding_residuals():
    rng = np.random.default_rng(2)
    S, D, n = 400, 64, 150
    v = heavy_v(S, D, rng)
    amax = np.full(D, np.abs(f64(v)).max(), dtype=np.float32)
    idx, _, rep = oracle.repair_select(v, amax, n)
    _, rr = residual_energy64(v, amax)
    want = rr[idx]
    got = dec(rep[:n])
    assert (np.abs(got - want) <= np.maximum(2.0 ** -4 * np.abs(want), 2.0 ** -10) + 1e-12).all()
    assert not rep[n:].any()
    assert rep.shape == (256, D)


def test_repair_keys_are_copies_of_the_selected_keys():
    rng = np.random.default_rng(3)
    S, D, n = 500, 64, 140
    k = bf16(rng.normal(0, 1.5, (S, D)))
    v = heavy_v(S, D, rng)
    amax = np.full(D, np.abs(f64(v)).max(), dtype=np.float32)
    rp = oracle.repair_rows(k, v, amax, n)
    K = f64(k)[rp["idx"]]
    assert rp["kc"].shape == (256, D) and rp["sk"].shape == (2,)
    kd = dec(rp["kc"][:n]) * np.repeat(rp["sk"], 128)[:n, None]
    blk_max = np.repeat([np.abs(K[:128]).max(), np.abs(K[128:]).max()], 128)[:n, None]
    assert (np.abs(kd - K) <= np.maximum(2.0 ** -4 * np.abs(K), 2.0 ** -10 * blk_max / 448) + 1e-12).all()
    assert not rp["kc"][n:].any()


def test_denominator_and_running_max_are_left_unchanged():
    rng = np.random.default_rng(4)
    S, D = 600, 64
    q, k = bf16(rng.normal(0, 1, (S, D))), bf16(rng.normal(0, 1, (S, D)))
    v = heavy_v(S, D, rng)
    rows = rng.choice(S, 20, replace=False)
    p0 = oracle.prepare_head(q, k, v, 1, 1, vsmooth=False)
    pz = oracle.prepare_head(q, k, v, 1, 1, vsmooth=False, n_repair=0)
    p1 = oracle.prepare_head(q, k, v, 1, 1, vsmooth=False, n_repair=40)
    o0, l0, m0 = oracle.forward_head(p0, rows)
    oz, _, _ = oracle.forward_head(pz, rows)
    o1, l1, m1 = oracle.forward_head(p1, rows)
    assert np.array_equal(o0, oz)
    assert np.array_equal(l0, l1) and np.array_equal(m0, m1)
    assert not np.array_equal(o0, o1)


def test_exactly_representable_values_need_no_repair():
    rng = np.random.default_rng(5)
    S, D = 300, 32
    grid = dec(np.arange(256, dtype=np.uint8))
    vals = grid[np.isfinite(grid) & (np.abs(grid) <= 64)]
    V = rng.choice(vals, size=(S, D)) * 2.0 ** -5
    V[0, 0] = 448 * 2.0 ** -5
    v = bf16(V)
    q, k = bf16(rng.normal(0, 1, (S, D))), bf16(rng.normal(0, 1, (S, D)))
    p0 = oracle.prepare_head(q, k, v, 1, 1, vsmooth=False)
    p1 = oracle.prepare_head(q, k, v, 1, 1, vsmooth=False, n_repair=50)
    assert not p1["repair"]["rc"].any()
    assert not p1["repair"]["energy"].any()
    rows = np.arange(0, S, 11)
    assert np.array_equal(oracle.forward_head(p0, rows)[0], oracle.forward_head(p1, rows)[0])


def fma32(a, b, c):
    return np.float32(np.float64(np.float32(a)) * np.float64(np.float32(b)) + np.float64(np.float32(c)))


def codes_of(s32, aj, M, expcast):
    b = np.float32(np.float32(119.65) - np.float32(M))
    y = np.array([fma32(x, aj, b) for x in s32], dtype=np.float32)
    if expcast:
        return dec(np.clip(np.rint(y), 0, 120).astype(np.uint8))
    ze = ((y - np.float32(119.65)) * np.float32(0.125) + np.float32(8.0)).astype(np.float32)
    p = np.exp2(ze.astype(np.float64)).astype(np.float32)
    return dec(torch.from_numpy(p).to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def closed_form(prep, r, expcast=True, midwindow=True, values=None):
    """Regular tiles with per-tile weights 2^((M_j - M)/8); the repair tiles at the final M, their
    probabilities times the repair codes added to the numerator only.  values: [S, D] fp64 to weight
    instead of the codes (the same probabilities on unquantised values; no repair term)."""
    S, D = prep["S"], prep["D"]
    nkb = (S + 127) // 128
    qt = r // 128
    order = list(range(nkb))
    if midwindow:
        st = min(nkb - 1, 2 * (qt // 2) + 2)
        order = list(range(st, -1, -1)) + list(range(st + 1, nkb))
    aq = np.float32(np.float32(8.0 * LOG2E / math.sqrt(D)) * prep["sq"][qt])
    qd = dec(prep["qc"][r])
    M = -np.inf
    tiles = []
    for j in order:
        n = min(128, S - 128 * j)
        s32 = (dec(prep["kc"][128 * j:128 * j + n]) @ qd).astype(np.float32)
        aj = np.float32(aq * prep["sk"][j])
        M = max(M, np.max((s32 * aj).astype(np.float32)))
        vals = values[128 * j:128 * j + n] if values is not None else dec(prep["rc"][128 * j:128 * j + n])
        tiles.append((np.float32(M), codes_of(s32, aj, M, expcast), vals))
    Mf = tiles[-1][0]
    num = sum(2.0 ** ((float(Mj) - float(Mf)) / 8) * (ph @ vals) for Mj, ph, vals in tiles)
    den = sum(2.0 ** ((float(Mj) - float(Mf)) / 8) * ph.sum() for Mj, ph, vals in tiles)
    if values is not None:
        return num / den
    rp = prep["repair"]
    if rp is not None:
        for jr in range((rp["n"] + 127) // 128):
            n = min(128, rp["n"] - 128 * jr)
            s32 = (dec(rp["kc"][128 * jr:128 * jr + n]) @ qd).astype(np.float32)
            aj = np.float32(aq * rp["sk"][jr])
            num = num + codes_of(s32, aj, Mf, expcast) @ dec(rp["rc"][128 * jr:128 * jr + n])
    return np.asarray(prep["sv"], dtype=np.float64) * num / den


@pytest.mark.parametrize("S,n,expcast,midwindow,channel", [
    (300, 7, True, True, False),
    (300, 200, True, False, False),   # two repair tiles, the second ragged
    (520, 128, False, True, False),   # exponentiate-then-cast path
    (257, 60, True, True, True),      # per-channel scales
])
def test_forward_with_repair_matches_closed_form(S, n, expcast, midwindow, channel):
    rng = np.random.default_rng(S + n)
    D = 32
    q, k = bf16(rng.normal(0, 1.2, (S, D))), bf16(rng.normal(0, 1.2, (S, D)))
    v = heavy_v(S, D, rng)
    prep = oracle.prepare_head(q, k, v, 1, 1, vsmooth=False, n_repair=n, vscale_channel=channel)
    rows = np.unique(np.concatenate([[0, S - 1], rng.choice(S, 10, replace=False)]))
    out, _, _ = oracle.forward_head(prep, rows, expcast=expcast, midwindow=midwindow)
    for i, r in enumerate(rows):
        want = closed_form(prep, int(r), expcast, midwindow)
        assert np.abs(out[i] - want).max() <= 1e-9 * max(1.0, np.abs(want).max())


def test_repair_removes_value_error():
    """The V part of the error, measured against the same probabilities on the unquantised values:
    repairing every token leaves only the mismatch of the copied keys' probabilities and the repair
    codes' own rounding; a small budget removes part of it, a larger one more."""
    rng = np.random.default_rng(6)
    S, D = 768, 64
    q, k = bf16(rng.normal(0, 0.7, (S, D))), bf16(rng.normal(0, 0.7, (S, D)))
    v = heavy_v(S, D, rng)
    V = f64(v)
    rows = rng.choice(S, 24, replace=False)
    ref = oracle.attention_exact(q, k, v, rows)
    err = {}
    for n in (0, math.ceil(0.005 * S), S // 10, S):
        prep = oracle.prepare_head(q, k, v, 1, 1, vsmooth=False, n_repair=n)
        out, _, _ = oracle.forward_head(prep, rows)
        same_p = np.stack([closed_form(prep, int(r), values=V) for r in rows])
        err[n] = np.linalg.norm(out - same_p) / np.linalg.norm(same_p)
        assert np.linalg.norm(out - ref) <= 0.06 * np.linalg.norm(ref)
    assert err[math.ceil(0.005 * S)] < err[0]
    assert err[S // 10] < 0.6 * err[0]
    assert err[S] < 0.1 * err[0]
