"""Pins for the oracle's E4M3 and bf16 codecs, against independent implementations.

E4M3: "VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention", Sec. 3.3
(v = 2^(e-7)(1+m/8)); OCP subnormals/NaN/saturation by reading. The independent references are
torch's float8_e4m3fn codec and a brute-force nearest-value search written here.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "paper_values.json")))


def torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_torch_all_codes():
    ours = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = torch_decode_all()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_printed_values():
    for code, val in GOLD["e4m3_decode"]["codes"].items():
        assert oracle.e4m3_decode([int(code)])[0] == val
    # 107 = 8*13 + 3: exponent field 13, mantissa 3 -> 2^6 * 1.375 = 88
    assert 107 == 8 * 13 + 3


def finite_table():
    ref = torch_decode_all()
    codes = np.array([c for c in range(256) if not np.isnan(ref[c])], dtype=np.int64)
    return codes, ref[codes]


def brute_encode(x: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value, ties to the code with an even mantissa, saturating at +-448."""
    codes, vals = finite_table()
    out = np.empty(x.shape, dtype=np.uint8)
    for i, xi in enumerate(x.astype(np.float64)):
        if xi > 448:
            out[i] = 0x7E
            continue
        if xi < -448:
            out[i] = 0xFE
            continue
        d = np.abs(vals - xi)
        best = np.flatnonzero(d == d.min())
        # the two codes of a tie are neighbours; prefer the even one; among +0/-0 keep the sign
        cand = [c for c in codes[best]]
        if len(cand) > 1:
            even = [c for c in cand if c % 2 == 0]
            cand = even if even else cand
            if len(cand) > 1:  # zero: +0 (0x00) vs -0 (0x80)
                cand = [0x80 if np.signbit(xi) else 0x00]
        out[i] = cand[0]
    return out


def test_encode_roundtrip_all_finite_codes():
    codes, vals = finite_table()
    enc = oracle.e4m3_encode(vals.astype(np.float32))
    assert np.array_equal(enc.astype(np.int64), codes)


def test_encode_midpoints_round_to_even():
    codes, vals = finite_table()
    pos = codes[(vals > 0)]
    pv = vals[(vals > 0)]
    order = np.argsort(pv)
    pos, pv = pos[order], pv[order]
    mids = ((pv[:-1] + pv[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (pv[:-1] + pv[1:]) / 2)  # midpoints exact in fp32
    enc = oracle.e4m3_encode(mids)
    want = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:])
    assert np.array_equal(enc, want.astype(np.uint8))


def test_encode_matches_brute_force_random():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 50, 3000), rng.normal(0, 0.01, 1000), rng.uniform(-600, 600, 500),
                        [0.0, -0.0, 448.0, -448.0, 449.0, 464.0, 1e9, -1e9, 2.0**-10, -(2.0**-10), 2.0**-9 * 1.5]])
    x = x.astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), brute_encode(x))


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 5000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def brute_bf16(x: float) -> int:
    """Nearest bf16 to a double, ties to even, by scanning the two bf16 neighbours of fp32(x)."""
    f = np.float32(x)
    u = int(np.array([f]).view(np.uint32)[0]) >> 16
    best = None
    for cand in (u - 1, u, u + 1, u + 2):
        if cand < 0 or cand > 0xFFFF:
            continue
        v = float(np.array([cand << 16], dtype=np.uint32).view(np.float32)[0])
        if not np.isfinite(v):
            continue
        key = (abs(v - x), cand % 2)
        if best is None or key < best[0]:
            best = (key, cand)
    return best[1]


def test_bf16_rounding_from_f64():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, 3, 3000), rng.normal(0, 1e-3, 500)])
    ours = oracle.f64_to_bf16(x)
    ref = np.array([brute_bf16(abs(v)) | (0x8000 if v < 0 else 0) for v in x], dtype=np.uint16)
    assert np.array_equal(ours, ref)
    # values exactly representable in fp32 agree with torch's fp32 -> bf16 rounding
    x32 = rng.normal(0, 10, 5000).astype(np.float32)
    t = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16(x32.astype(np.float64)), t)
    # a double between two fp32 values whose fp32 rounding would tie: single rounding decides
    assert oracle.f64_to_bf16(np.array([1.0 + 2.0**-8 + 2.0**-40]))[0] == 0x3F81
