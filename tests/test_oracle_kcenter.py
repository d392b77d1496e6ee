"""Oracle pins of the K channel centering ("VC-Attention", Sec. 3.4 "Fused preprocessing", App. B:
the keys' quantisation pass subtracts the channel mean it has gathered statistics for)."""
import numpy as np
import pytest
import torch

import oracle


def bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f64(u16) -> np.ndarray:
    return torch.from_numpy(np.asarray(u16, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_channel_mean_of_symmetric_columns():
    """Columns a_d +- e_d in equal numbers have the exact mean a_d, whatever the order."""
    rng = np.random.default_rng(3)
    S, D = 1000, 16
    a = np.array([1.5, -3.0, 0.0, 40.0, 0.25, -0.75, 2.0, 5.0, -7.5, 0.5, 1.0, 24.0, -0.125, 3.5, 12.0, -1.0])
    e = np.array([0.25, 0.5, 1.0, 4.0, 0.0625, 0.125, 0.5, 1.0, 0.5, 0.125, 0.25, 8.0, 0.03125, 0.5, 2.0, 0.25])
    x = np.empty((S, D))
    x[0::2] = a - e
    x[1::2] = a + e
    x = x[rng.permutation(S)]
    assert np.array_equal(f64(bf16(x)), x)  # every entry is a bf16 value
    mu = oracle.channel_mean_bf16(bf16(x))
    assert np.array_equal(f64(mu), a)


def test_zero_center_is_the_plain_quantiser():
    rng = np.random.default_rng(4)
    x = bf16(rng.normal(0, 2, (300, 64)))
    c0, s0 = oracle.quant_blocks(x)
    c1, s1 = oracle.quant_blocks(x, center=np.zeros(64, dtype=np.uint16))
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)


def test_centered_quantiser_equals_quantiser_of_the_difference():
    """When K - mu is itself a bf16 matrix, quantising K with the centre equals quantising K - mu."""
    rng = np.random.default_rng(5)
    S, D = 260, 32
    mu = 2.0 ** rng.integers(-2, 3, D) * rng.choice([-1, 1], D)
    diff = rng.integers(-64, 65, (S, D)) * 2.0 ** -5  # small dyadic offsets: K and K - mu both exact in bf16
    k = mu[None, :] + diff
    assert np.array_equal(f64(bf16(k)), k) and np.array_equal(f64(bf16(diff)), diff)
    c_center, s_center = oracle.quant_blocks(bf16(k), center=bf16(mu))
    c_diff, s_diff = oracle.quant_blocks(bf16(diff))
    assert np.array_equal(c_center, c_diff) and np.array_equal(s_center, s_diff)


def test_centering_leaves_exact_attention_unchanged():
    """Subtracting one vector from every key shifts each query's scores by a constant."""
    rng = np.random.default_rng(6)
    S, D = 300, 64
    q = rng.normal(0, 1, (S, D))
    k = rng.normal(0, 1, (S, D)) + rng.normal(0, 5, D)
    v = rng.normal(0, 1, (S, D))
    mu = k.mean(axis=0)
    rows = np.arange(0, S, 7)
    a = oracle.attention_demeaned_exact(q, k, v, rows)
    b = oracle.attention_demeaned_exact(q, k - mu, v, rows)
    assert np.abs(a - b).max() <= 1e-12 * np.abs(a).max()


@pytest.mark.parametrize("offset", [8.0, 30.0])
def test_centering_reduces_error_of_offset_keys(offset):
    """Keys sharing a large channel offset: the offset dominates each block's range, so uncentred codes
    resolve the informative part poorly. Centred, the quantised forward is as close to exact attention
    as it is for the same keys without the offset, and several times closer than uncentred."""
    def rel_error(off, kcenter):
        rng = np.random.default_rng(7)
        S, D = 512, 64
        q = bf16(rng.normal(0, 1.0, (S, D)))
        k = bf16(rng.normal(0, 1.0, (S, D)) + off * rng.choice([-1.0, 1.0], D))
        v = bf16(rng.normal(0, 1.0, (S, D)))
        rows = np.arange(0, S, 5)
        exact = oracle.attention_exact(q, k, v, rows)
        prep = oracle.prepare_head(q, k, v, k_clusters=4, iters=2, vsmooth=False, kcenter=kcenter)
        out, _, _ = oracle.forward_head(prep, rows)
        return np.linalg.norm(out - exact) / np.linalg.norm(exact)

    base = rel_error(0.0, False)
    plain, centred = rel_error(offset, False), rel_error(offset, True)
    assert centred <= 1.2 * base, (centred, base)
    assert centred < plain / 3, (centred, plain)
