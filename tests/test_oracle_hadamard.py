"""Oracle pins of the QK Hadamard rotation ("VC-Attention", Sec. 3.4 "Fused preprocessing", App. B: the
Q and K quantisation passes fuse a Hadamard rotation; Fig. 3: it shrinks the probability term).

Independent references: the Sylvester closed form H[i][j] = (-1)^popcount(i & j), H H = D I, the
inner-product identity <Hx, Hy> = D <x, y>, exactly representable rotated rows, and exact fp64
attention (the rotation leaves Q K^T unchanged, so only the quantisation error moves).
"""

import numpy as np
import pytest
import torch

import oracle


def bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def f64(u16) -> np.ndarray:
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dec(codes) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def sylvester(D):
    i = np.arange(D)
    bits = np.bitwise_and(i[:, None], i[None, :])
    pop = np.array([bin(b).count("1") for b in bits.ravel()]).reshape(D, D)
    return np.where(pop % 2 == 0, 1.0, -1.0)


@pytest.mark.parametrize("D", [64, 128])
def test_transform_of_the_unit_vectors_is_the_sylvester_matrix(D):
    got = oracle.fwht(np.eye(D, dtype=np.float32))
    assert np.array_equal(got.astype(np.float64), sylvester(D))  # H is symmetric: row i = H e_i


@pytest.mark.parametrize("D", [64, 128])
def test_transform_twice_is_d_times_identity(D):
    rng = np.random.default_rng(D)
    x = rng.integers(-50, 50, size=(5, D)).astype(np.float32)
    assert np.array_equal(oracle.fwht(oracle.fwht(x)), D * x)  # small integers: every step exact


def test_inner_products_scale_by_d_and_the_score_constant_takes_it():
    rng = np.random.default_rng(1)
    D = 128
    x, y = rng.normal(0, 1, (2, D)).astype(np.float32)
    hx, hy = oracle.fwht(x).astype(np.float64), oracle.fwht(y).astype(np.float64)
    assert abs(hx @ hy - D * float(x.astype(np.float64) @ y)) <= 1e-4 * D * np.linalg.norm(x) * np.linalg.norm(y)
    c, cr = oracle.code_scale(D), float(oracle.lib().orc_code_scale_rot(D))
    assert abs(cr * D - c) <= 2.0 ** -22 * c


def test_rotated_quantiser_is_exact_on_rows_that_rotate_to_a_grid():
    """A multiple of a unit vector rotates to +-c in every channel: one code magnitude, no rounding."""
    rng = np.random.default_rng(2)
    S, D = 200, 64
    x = np.zeros((S, D))
    mag = rng.choice([-4.0, -1.0, 0.5, 2.0, 4.0], S)
    mag[[0, 128]] = 4.0  # every block's largest |value| is 4, so its codes are value * 448/4
    x[np.arange(S), rng.integers(0, D, S)] = mag
    codes, scales = oracle.quant_blocks(bf16(x), rotate=True)
    want = sylvester(D)[np.argmax(np.abs(x), axis=1)] * mag[:, None] * (448.0 / 4.0)
    assert np.array_equal(dec(codes[:S]), want)
    assert np.array_equal(scales, np.full(2, np.float32(4.0) / np.float32(448.0)))


def test_rotation_leaves_the_softmax_target_and_shrinks_outlier_error():
    """Keys and queries with a few outlier channels: exact attention is unchanged by construction, and the
    quantised forward with the rotation lands closer to it."""
    rng = np.random.default_rng(3)
    S, D = 512, 64
    gain = np.ones(D)
    gain[rng.choice(D, 3, replace=False)] = 25.0
    q = bf16(rng.normal(0, 0.3, (S, D)) * gain)
    k = bf16(rng.normal(0, 0.3, (S, D)) * gain)
    v = bf16(rng.normal(0, 1, (S, D)))
    rows = rng.choice(S, 32, replace=False)
    ref = oracle.attention_exact(q, k, v, rows)
    err = {}
    for rot in (False, True):
        prep = oracle.prepare_head(q, k, v, 1, 1, vsmooth=False, hadamard=rot)
        out, _, _ = oracle.forward_head(prep, rows)
        err[rot] = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    assert err[True] < err[False]
    assert err[True] <= 0.05


def test_rotated_forward_matches_the_plain_one_on_exact_scores():
    """With Q and K on a coarse grid both paths quantise exactly, so the two forwards coincide up to the
    fp32 rounding of the score constant."""
    rng = np.random.default_rng(4)
    S, D = 256, 64
    q = np.zeros((S, D))
    k = np.zeros((S, D))
    q[np.arange(S), rng.integers(0, D, S)] = rng.choice([-1.0, 1.0], S)
    k[np.arange(S), rng.integers(0, D, S)] = rng.choice([-1.0, 1.0], S)
    q, k = bf16(q), bf16(k)
    v = bf16(rng.normal(0, 1, (S, D)))
    rows = np.arange(0, S, 9)
    a, _, _ = oracle.forward_head(oracle.prepare_head(q, k, v, 1, 1, vsmooth=False), rows)
    b, _, _ = oracle.forward_head(oracle.prepare_head(q, k, v, 1, 1, vsmooth=False, hadamard=True), rows)
    assert np.abs(a - b).max() <= 0.02 * np.abs(a).max()
