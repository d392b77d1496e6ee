"""Oracle pins of the per-channel V residual scale ("VC-Attention", Sec. 3.2 "Block demeaning": the
residual is quantised per channel to E4M3; App. B: the stored means are divided by the channel
scale, so one epilogue multiply per channel serves both terms of Eq. 6).

Independent references: the E4M3 rounding bound, exact power-of-two scaling of one channel, the
per-head mode as the special case of equal channel ranges, a closed form of the forward with
per-tile weights, and exact fp64 attention.
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


def skewed_v(S, D, rng):
    """Channels with offsets and a spread over three octaves, a few of them outliers 2^14 wider: with
    one scale per head the other channels then fall into E4M3's subnormal range."""
    scale = 2.0 ** rng.uniform(-2, 1, D)
    scale[rng.choice(D, 3, replace=False)] *= 2.0 ** 14
    off = rng.normal(0, 1, D) * scale * 3
    return bf16(rng.normal(0, 1, (S, D)) * scale + off)


@pytest.mark.parametrize("S,vsmooth", [(300, True), (257, False), (128, True)])
def test_each_channel_spans_the_full_code_range(S, vsmooth):
    rng = np.random.default_rng(S)
    D = 32
    v = skewed_v(S, D, rng)
    perm = rng.permutation(S).astype(np.int32)
    dm = oracle.demean(v, perm, subtract_mean=vsmooth, per_channel=True)
    R = dm["resid"][:S].astype(np.float64)
    amax = np.abs(R).max(axis=0)
    assert np.array_equal(dm["amax"].astype(np.float64), amax)
    assert np.array_equal(dm["sv"], (dm["amax"] / np.float32(448)).astype(np.float32))
    codes = dec(dm["rc"][:S])
    assert np.array_equal(np.abs(codes).max(axis=0), np.full(D, 448.0))  # the max row of every channel
    assert not dm["rc"][S:].any()  # pad rows stay zero


def test_per_channel_dequantisation_bound():
    """Each residual within half an E4M3 step of its code times the channel scale."""
    rng = np.random.default_rng(5)
    S, D = 400, 64
    v = skewed_v(S, D, rng)
    dm = oracle.demean(v, None, subtract_mean=True, per_channel=True)
    R = dm["resid"][:S].astype(np.float64)
    x = R / dm["sv"][None, :].astype(np.float64)
    err = np.abs(dec(dm["rc"][:S]) - x)
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10) * (1 + 1e-6) + 1e-9
    assert (err <= bound).all()
    # per channel the relative L2 error of the reconstruction stays at E4M3's normal-range level;
    # one scale per head pushes the narrow channels into the subnormals
    dh = oracle.demean(v, None, subtract_mean=True, per_channel=False)
    rel = lambda a: np.linalg.norm(a - R, axis=0) / np.linalg.norm(R, axis=0)
    e_ch = rel(dec(dm["rc"][:S]) * dm["sv"][None, :])
    e_hd = rel(dec(dh["rc"][:S]) * dh["sv"])
    assert e_ch.max() <= 2.0 ** -4
    assert e_hd.max() > 4 * e_ch.max()


def test_equal_channel_ranges_reduce_to_one_scale_per_head():
    rng = np.random.default_rng(6)
    S, D = 256, 16
    levels = np.array([0.5, 1.0, 2.0, 3.0, 6.0])
    R = np.zeros((S, D))
    for j in range(0, S, 128):
        half = rng.choice(levels, size=(64, D)) * rng.choice([-1, 1], size=(64, D))
        half[0] = 7.0  # every channel reaches 7 in every block
        R[j:j + 128] = np.concatenate([half, -half])
    mu = np.round(rng.normal(0, 3, (S // 128, D)) * 4) / 4
    v = bf16(R + np.repeat(mu, 128, axis=0))
    a = oracle.demean(v, None, per_channel=True)
    b = oracle.demean(v, None, per_channel=False)
    assert np.array_equal(a["rc"], b["rc"])
    assert np.array_equal(a["sv"], np.full(D, b["sv"], dtype=np.float32))
    assert np.array_equal(f64(a["mub"]), mu)
    assert np.array_equal(f64(a["mut"]) * a["sv"][None, :].astype(np.float64) * 64, mu * 64)  # 7/448 = 2^-6


def test_stored_means_are_the_means_over_the_channel_scale():
    rng = np.random.default_rng(7)
    S, D = 520, 48
    v = skewed_v(S, D, rng)
    dm = oracle.demean(v, rng.permutation(S).astype(np.int32), per_channel=True)
    want = f64(dm["mub"]) / dm["sv"][None, :].astype(np.float64)
    got = f64(dm["mut"])
    assert (np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-30).all()  # one bf16 rounding


def channel_scaled(v, d_scale):
    x = f64(v).copy()
    for d, e in d_scale.items():
        x[:, d] *= 2.0 ** e
    return bf16(x)


def test_power_of_two_scaling_of_one_channel_scales_only_that_channel():
    """Codes and stored means do not move; the channel's scale and output carry the exact factor."""
    rng = np.random.default_rng(8)
    S, D = 300, 32
    q = bf16(rng.normal(0, 1, (S, D)))
    k = bf16(rng.normal(0, 1, (S, D)))
    v = skewed_v(S, D, rng)
    perm = rng.permutation(S).astype(np.int32)
    widest = int(np.argmax(oracle.demean(v, perm, per_channel=True)["amax"]))
    ds = {3: 5, 7: -3, 30: 2}
    ds[widest] = 2  # the channel that sets the per-head scale
    v2 = channel_scaled(v, ds)
    p1 = oracle.prepare_head(q, k, v, 1, 1, perm=perm, vscale_channel=True)
    p2 = oracle.prepare_head(q, k, v2, 1, 1, perm=perm, vscale_channel=True)
    assert np.array_equal(p1["rc"], p2["rc"])
    assert np.array_equal(p1["mut"], p2["mut"])
    f = np.ones(D)
    for d, e in ds.items():
        f[d] = 2.0 ** e
    assert np.array_equal(p2["sv"].astype(np.float64), p1["sv"] * f)
    rows = rng.choice(S, 12, replace=False)
    o1, l1, _ = oracle.forward_head(p1, rows)
    o2, l2, _ = oracle.forward_head(p2, rows)
    assert np.array_equal(l1, l2)
    assert np.array_equal(o2, o1 * f[None, :])
    # with one scale per head every other channel's codes move (the pin is not vacuous)
    h1 = oracle.prepare_head(q, k, v, 1, 1, perm=perm)
    h2 = oracle.prepare_head(q, k, v2, 1, 1, perm=perm)
    other = next(d for d in range(D) if d not in ds)
    assert not np.array_equal(h1["rc"][:, other], h2["rc"][:, other])


def fma32(a, b, c):
    return np.float32(np.float64(np.float32(a)) * np.float64(np.float32(b)) + np.float64(np.float32(c)))


def closed_form_channel(prep, r, midwindow=True, values=None):
    """Per-tile weights 2^((M_j - M_final)/8); values (R/s + mu/s) * s per channel, or the given
    [S, D] fp64 values in key order (the same probabilities on unquantised values)."""
    S, D = prep["S"], prep["D"]
    nkb = (S + 127) // 128
    qt = r // 128
    order = list(range(nkb))
    if midwindow:
        st = min(nkb - 1, 2 * (qt // 2) + 2)
        order = list(range(st, -1, -1)) + list(range(st + 1, nkb))
    C = np.float32(8.0 * LOG2E / math.sqrt(D))
    aq = np.float32(C * prep["sq"][qt])
    qd = dec(prep["qc"][r])
    sv = np.asarray(prep["sv"], dtype=np.float64)
    M = -np.inf
    tiles = []
    for j in order:
        n = min(128, S - 128 * j)
        s32 = (dec(prep["kc"][128 * j:128 * j + n]) @ qd).astype(np.float32)
        aj = np.float32(aq * prep["sk"][j])
        M = max(M, np.max((s32 * aj).astype(np.float32)))
        b = np.float32(np.float32(119.65) - np.float32(M))
        y = np.array([fma32(x, aj, b) for x in s32], dtype=np.float32)
        ph = dec(np.clip(np.rint(y), 0, 120).astype(np.uint8))
        if values is not None:
            tiles.append((np.float32(M), ph, values[128 * j:128 * j + n]))
            continue
        vals = dec(prep["rc"][128 * j:128 * j + n])
        if prep["vsmooth"]:
            vals = vals + f64(prep["mut"][j])[None, :]
        tiles.append((np.float32(M), ph, vals * sv[None, :]))
    Mf = tiles[-1][0]
    num = sum(2.0 ** ((float(Mj) - float(Mf)) / 8) * (ph @ vals) for Mj, ph, vals in tiles)
    den = sum(2.0 ** ((float(Mj) - float(Mf)) / 8) * ph.sum() for Mj, ph, vals in tiles)
    return num / den


@pytest.mark.parametrize("S,vsmooth,midwindow", [(300, True, True), (300, True, False), (257, False, True)])
def test_per_channel_forward_matches_closed_form(S, vsmooth, midwindow):
    rng = np.random.default_rng(S + 10 * vsmooth + midwindow)
    D = 32
    q = bf16(rng.normal(0, 1.2, (S, D)))
    k = bf16(rng.normal(0, 1.2, (S, D)))
    v = skewed_v(S, D, rng)
    prep = oracle.prepare_head(q, k, v, 2, 2, vsmooth=vsmooth, vscale_channel=True)
    rows = np.unique(np.concatenate([[0, S - 1], rng.choice(S, 10, replace=False)]))
    out, _, _ = oracle.forward_head(prep, rows, midwindow=midwindow)
    for i, r in enumerate(rows):
        want = closed_form_channel(prep, int(r), midwindow)
        assert np.abs(out[i] - want).max() <= 1e-9 * max(1e-3, np.abs(want).max())
    # the mean term is there: dropping it is visibly wrong
    if vsmooth:
        bad, _, _ = oracle.forward_head(dict(prep, vsmooth=False), rows, midwindow=midwindow)
        assert np.abs(bad - out).max() > 0.1 * np.abs(out).max()


def test_per_channel_scale_is_more_accurate_on_skewed_channels():
    """The V part of the error: both modes share the probabilities, so each is compared with the same
    closed form on the unquantised values; per channel the narrow channels keep their accuracy."""
    rng = np.random.default_rng(9)
    S, D = 640, 64
    q = bf16(rng.normal(0, 1, (S, D)))
    k = bf16(rng.normal(0, 1, (S, D)))
    v = skewed_v(S, D, rng)
    V = f64(v)
    span = np.abs(V - V.mean(axis=0)).max(axis=0)
    rows = rng.choice(S, 16, replace=False)
    ref = oracle.attention_exact(q, k, v, rows)
    perm = rng.permutation(S).astype(np.int32)
    errs = {}
    for ch in (False, True):
        prep = oracle.prepare_head(q, k, v, 1, 1, perm=perm, vscale_channel=ch)
        out, _, _ = oracle.forward_head(prep, rows)
        assert np.linalg.norm(out - ref) <= 1e-2 * np.linalg.norm(ref)
        same_p = np.stack([closed_form_channel(prep, int(r), values=V[perm]) for r in rows])
        errs[ch] = np.abs(out - same_p).max(axis=0) / span
    assert errs[True].max() <= 2.0 ** -6
    assert errs[True].max() < 0.5 * errs[False].max()
