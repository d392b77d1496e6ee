"""Pins for the oracle's ExpCast-FP8 map against the numbers the pages print.

"VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention", Sec. 3.3 Eq. 7,
Fig. 5, Prop. 3.1, Appendix C/D; "Open-VC Attention" (MachGen blog), "Scheduling around ExpCast".
"""
import json
import math
import os

import numpy as np
import torch

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "paper_values.json")))
LOG2E = 1.4426950408889634


def dec(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_worked_example():
    g = GOLD["expcast_worked_example"]
    u = g["u"]
    assert abs(8 * (u + 8) + 56 - 0.35 - g["pre_round"]) < 1e-9
    assert oracle.expcast_of_u(u) == g["code"]
    assert dec([g["code"]])[0] == g["value"]
    assert abs(2 ** (u + 8) - g["exp_value"]) < 0.05
    assert oracle.exp_then_cast(u) == g["exp_cast_code"]


def test_row_max_lands_at_256():
    g = GOLD["expcast_row_max"]
    assert oracle.expcast_of_u(g["u"]) == g["code"]
    assert dec([g["code"]])[0] == g["value"]


def test_beta_shift_and_sign():
    g = GOLD["beta"]
    f = np.linspace(0.0, 1.0, 2_000_001)
    e = 8 * (f - (2.0**f - 1))
    assert abs(e.max() - g["e_max"]) < 5e-5 and e.min() >= -1e-12
    assert abs(-e.max() / 2 - g["minimax_shift"]) < 5e-5
    # the pages round the minimax shift outward to beta = -0.35
    assert abs(g["beta"] - (-e.max() / 2)) < 0.01 and g["beta"] <= -e.max() / 2
    # the oracle's map uses beta = -0.35: 8(u+8)+56 = 100.8 -> 100.45 -> 100 (beta = 0 would give 101)
    u = (100.8 - 56) / 8 - 8
    assert oracle.expcast_of_u(u) == 100


def test_agreement_with_exp_then_cast_over_a_doubling():
    g = GOLD["expcast_agreement"]
    us = np.linspace(-3.0, -2.0, 200_001)[:-1]
    direct = np.array([oracle.expcast_of_u(u) for u in us])
    conv = np.array([oracle.exp_then_cast(u) for u in us])
    diff = np.abs(direct - conv)
    assert diff.max() == g["max_code_difference"]
    assert abs((diff == 0).mean() - g["same_fraction"]) < 0.002


def test_at_most_one_code_and_relative_error_over_normal_range():
    us = np.linspace(-14.0, 0.0, 400_001)
    direct = np.array([oracle.expcast_of_u(u) for u in us])
    conv = np.array([oracle.exp_then_cast(u) for u in us])
    assert np.abs(direct - conv).max() <= 1
    rel = np.abs(dec(direct) - 2.0 ** (us + 8)) / 2.0 ** (us + 8)
    assert rel.max() <= GOLD["relative_error_per_element"]["max_rel"] + 1e-3


def test_ratio_bounds():
    g = GOLD["ratio_bounds"]
    us = np.linspace(-5.0, -4.0, 400_001)[:-1]
    r = dec([oracle.expcast_of_u(u) for u in us]) / 2.0 ** (us + 8)
    assert abs(r.min() - g["r_min"]) < 2e-4 and abs(r.max() - g["r_max"]) < 2e-4
    a, b = g["r_min"], g["r_max"]
    tv = (math.sqrt(b) - math.sqrt(a)) / (math.sqrt(b) + math.sqrt(a))
    assert tv < GOLD["tv_bound"]["tv"] and abs(tv - 0.03638) < 5e-5


def test_normal_range_boundary():
    assert oracle.expcast_of_u(GOLD["normal_range"]["u_min_normal"]) == 8  # smallest normal code
    assert oracle.expcast_of_u(-14.1) == 7  # 6.85 -> 7: a subnormal code, kept by the literal clip
    assert oracle.expcast_of_u(-15.0) == 0


def test_fp32_contract_matches_eq7():
    """The fp32 one-FMA form equals Eq. 7 wherever fp32 rounding does not move a .5 boundary."""
    rng = np.random.default_rng(0)
    u = rng.uniform(-16, 0, 200_000)
    s = (8 * u).astype(np.float32)
    codes = oracle.expcast_codes(s, np.float32(1.0), np.float32(119.65))
    ref = np.array([oracle.expcast_of_u(float(x) / 8) for x in s])
    assert (codes == ref).mean() > 0.9999
    assert np.abs(codes.astype(int) - ref).max() <= 1


def test_clip_onset_above_stale_max():
    """A score above the running max codes past 120 once 8 du >= 0.85, i.e. du >= 0.10625 log2 units."""
    M = 500.0
    b = np.float32(119.65) - np.float32(M)
    deltas = np.arange(0, 20000) * 1e-5
    first = None
    for d in deltas:
        s = np.float32(M + 8 * d)
        if oracle.expcast_unclipped(float(s), 1.0, float(b)) > 120:
            first = d
            break
    assert first is not None and abs(first - 0.10625) < 2e-4
    assert round(first / LOG2E, 3) == GOLD["clip_onset"]["nats"]
    assert oracle.expcast_code(float(np.float32(M + 8)), 1.0, float(b)) == 120  # clipped


def test_prop31_rows():
    """TV(p, p_hat) < 0.0364 + tau and ||o_hat - o|| <= (0.0364 + tau) diam(V) on random rows."""
    rng = np.random.default_rng(5)
    bound = GOLD["tv_bound"]["tv"]
    for trial in range(40):
        n = int(rng.integers(16, 2000))
        s = rng.normal(0, float(rng.choice([0.3, 1.0, 3.0, 8.0])), n)
        y = (8 * LOG2E * s).astype(np.float32)
        M = y.max()
        codes = oracle.expcast_codes(y, np.float32(1.0), np.float32(119.65) - M)
        ph = dec(codes)
        ph = ph / ph.sum()
        p = np.exp(s - s.max())
        p = p / p.sum()
        u = (s - s.max()) * LOG2E
        tail = u < -14
        tau = max(p[tail].sum(), ph[tail].sum())
        tv = 0.5 * np.abs(p - ph).sum()
        assert tv < bound + tau
        V = rng.normal(0, 1, (n, 8))
        diam = max(np.linalg.norm(V[i] - V, axis=1).max() for i in range(n))
        assert np.linalg.norm(ph @ V - p @ V) <= (bound + tau) * diam + 1e-12
