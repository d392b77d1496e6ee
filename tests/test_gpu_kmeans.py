"""The grouping kernels against brute force in fp64 ("VC-Attention", Sec. 3.2).

* assignment: after one round the labels are those of the nearest initial centroid (rows
  floor(i*S/k)); where the GPU's fp32 distance picks another centroid, the two fp64 distances
  differ by less than the rounding of an fp32 evaluation of ||c||^2 - 2 x.c;
* argsort: bit-exact against the oracle's stable argsort of the GPU labels;
* update: every centroid equals the fp64 mean of its members to within 2 fp32 ulps; an empty
  cluster keeps its previous centroid.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import f64, plan_host, vc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return vc()


def sq_dists(x: np.ndarray, c: np.ndarray) -> np.ndarray:
    """||x_t - c_i||^2 in fp64 for all pairs (inputs are bf16 values, so x.c is exact to ~1e-16)."""
    return (x * x).sum(1)[:, None] + (c * c).sum(1)[None, :] - 2.0 * (x @ c.T)


@pytest.mark.parametrize("D,S,k", [(128, 3000, 37), (64, 5000, 300), (128, 20000, 591), (64, 777, 777)])
def test_first_round_assigns_nearest_initial_centroid(m, D, S, k):
    cfg = synth.custom(S=S, D=D, H=2, k=k, iters=1)
    Q, K, V = synth.make_inputs(cfg, seed=5, device="cuda")
    plan = m.vc_attn_prepare(Q, K, V, k, 1)
    assert m.vc_plan_status(plan) == (0, 0)
    labels = plan_host(m, plan, m.VC_PLAN_LABELS)
    perm = plan_host(m, plan, m.VC_PLAN_PERM)
    for h in range(2):
        x = f64(V[0, h])
        c0 = x[(np.arange(k) * S) // k]
        d = sq_dists(x, c0)
        lab = labels[0, h]
        assert lab.min() >= 0 and lab.max() < k
        best = d.min(1)
        chosen = d[np.arange(S), lab]
        # fp32 evaluation: |err| <~ 2^-16 |x||c| (hi + lo split) + D 2^-24 (|x||c| + ||c||^2)
        xn = np.sqrt((x * x).sum(1))
        cmax = np.sqrt((c0 * c0).sum(1)).max()
        tol = 4.0 * (2.0**-16 * xn * cmax + D * 2.0**-24 * (xn * cmax + cmax * cmax))
        gap = chosen - best
        assert (gap <= tol).all(), f"head {h}: worst gap {gap.max():.3e}"
        exact = lab == d.argmin(1)
        assert exact.mean() >= 0.995, f"head {h}: only {exact.mean():.4f} of the labels match fp64"
        assert np.array_equal(perm[0, h], oracle.stable_argsort(lab, k)), f"head {h}: permutation"
    plan.destroy()


@pytest.mark.parametrize("D,S,k,iters", [(128, 4096, 64, 3), (64, 9000, 500, 2)])
def test_update_is_member_mean(m, D, S, k, iters):
    cfg = synth.custom(S=S, D=D, H=2, k=k, iters=iters)
    Q, K, V = synth.make_inputs(cfg, seed=6, device="cuda")
    plan = m.vc_attn_prepare(Q, K, V, k, iters)
    assert m.vc_plan_status(plan) == (0, 0)
    labels = plan_host(m, plan, m.VC_PLAN_LABELS)
    cent = plan_host(m, plan, m.VC_PLAN_CENTROIDS)
    plan1 = m.vc_attn_prepare(Q, K, V, k, iters - 1)  # centroids the last assignment used
    prev = plan_host(m, plan1, m.VC_PLAN_CENTROIDS)
    for h in range(2):
        x = f64(V[0, h])
        lab = labels[0, h]
        cnt = np.bincount(lab, minlength=k)
        sums = np.zeros((k, D))
        np.add.at(sums, lab, x)
        ref = np.where(cnt[:, None] > 0, sums / np.maximum(cnt, 1)[:, None], prev[0, h].astype(np.float64))
        got = cent[0, h].astype(np.float64)
        ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
        err = np.abs(got - ref)
        assert (err <= 2 * ulp + 1e-30).all(), f"head {h}: worst {np.max(err / ulp):.2f} ulp"
        empty = cnt == 0
        assert np.array_equal(got[empty], prev[0, h][empty].astype(np.float64))
    plan.destroy()
    plan1.destroy()
