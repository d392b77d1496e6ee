"""Grouping schedule and warm-started k-means ("VC-Attention", Sec. 3.2 "Unbalanced clusters cost little",
Sec. 3.4 "Amortized grouping schedule", App. A "Grouping schedule"). CPU only: the oracle against the
pages' printed schedules, the library's schedule against the oracle, and warm-start properties."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "paper_values.json")))["grouping_schedule"]


def regroup_steps(action, n):
    return [s for s in range(n) if action(s, n, 4) in (oracle.GROUP, oracle.GROUP_WARM)]


def test_schedule_matches_the_pages():
    assert regroup_steps(oracle.schedule_action, 40) == GOLDEN["steps40"]
    assert regroup_steps(oracle.schedule_action, 50) == GOLDEN["steps50"]
    assert sum(oracle.schedule_action(s, 8, 4) != oracle.PLAIN for s in range(8)) == GOLDEN["window8"]
    # only the first step groups from scratch; the window's other steps reuse pi; then the plain kernel
    acts = [oracle.schedule_action(s, 40, 4) for s in range(40)]
    assert acts[0] == oracle.GROUP and acts[4] == acts[8] == oracle.GROUP_WARM
    assert all(a == oracle.REUSE for i, a in enumerate(acts[:10]) if i % 4)
    assert all(a == oracle.PLAIN for a in acts[10:])


@pytest.fixture(scope="module")
def vc():
    from bit_fp8_attention_gb300 import build

    build.build()
    import bit_fp8_attention_gb300 as mod

    return mod


def test_library_schedule_matches_oracle(vc):
    for n in range(1, 61):
        for reuse in range(1, 6):
            for s in range(n):
                assert vc.vc_schedule_action(s, n, reuse) == oracle.schedule_action(s, n, reuse), (s, n, reuse)
    for bad in ((-1, 10, 4), (10, 10, 4), (0, 0, 4), (0, 10, 0)):
        with pytest.raises(vc.VCError):
            vc.vc_schedule_action(*bad)


def bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def clustered(rng, S, D, k, spread=0.3):
    centres = rng.normal(0, 3, (k, D))
    return centres[rng.integers(0, k, S)] + rng.normal(0, spread, (S, D))


def test_warm_start_from_rows_equals_cold_start():
    rng = np.random.default_rng(1)
    S, D, k = 900, 16, 12
    v = bf16(clustered(rng, S, D, k))
    rows = (np.arange(k) * S) // k
    init = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).double().numpy()[rows]
    a = oracle.kmeans(v, k, 3)
    b = oracle.kmeans(v, k, 3, init=init)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


def test_converged_centroids_are_a_fixed_point():
    rng = np.random.default_rng(2)
    S, D, k = 700, 8, 6
    v = bf16(clustered(rng, S, D, k, spread=0.2))
    labels, cent, J = oracle.kmeans(v, k, 30)
    l2, c2, J2 = oracle.kmeans(v, k, 1, init=cent)
    assert np.array_equal(labels, l2) and J2[0] == pytest.approx(J[-1], rel=1e-12)


def test_warm_start_on_the_next_step_needs_half_the_rounds():
    """Activations change little between adjacent steps: from the previous step's centroids, 2 rounds on
    the next step reach (within 1%) the objective of 4 rounds from scratch."""
    rng = np.random.default_rng(3)
    S, D, k = 4000, 32, 40
    x = clustered(rng, S, D, k, spread=0.6)
    v0 = bf16(x)
    v1 = bf16(x + rng.normal(0, 0.05, x.shape))  # the next denoising step
    _, cent0, _ = oracle.kmeans(v0, k, 4)
    _, _, J_cold = oracle.kmeans(v1, k, 4)
    _, _, J_warm = oracle.kmeans(v1, k, 2, init=cent0)
    assert J_warm[-1] <= 1.01 * J_cold[-1], (J_warm, J_cold)
