"""Warm-started grouping and the grouping schedule on the GPU ("VC-Attention", Sec. 3.2 "Unbalanced clusters
cost little", Sec. 3.4 "Amortized grouping schedule", App. A "Grouping schedule")."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_within, compare_prep, errors, f64, gpu_plan_all, head_of, oracle_forward_from_plan, u16, vc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return vc()


def next_step(V, s, scale=0.03):
    """The values of denoising step s: a small seeded drift of V."""
    gen = torch.Generator().manual_seed(100 + s)
    noise = torch.randn(V.shape, generator=gen).to(V.device)
    return (V.float() + scale * V.float().std() * noise).to(torch.bfloat16).contiguous()


def test_warm_start_from_the_previous_centroids(m):
    cfg = synth.custom(S=6000, D=128, H=2, k=48, iters=4, locality=True)
    Q, K, V0 = synth.make_inputs(cfg, seed=31, device="cuda")
    plan = m.vc_attn_prepare(Q, K, V0, cfg["k"], 4)
    cent0 = m.vc_plan_get(plan, m.VC_PLAN_CENTROIDS).cpu().numpy().astype(np.float64)
    V1 = next_step(V0, 1)
    m.vc_attn_prepare_ex(Q, K, V1, cfg["k"], 2, flags=m.VC_VSMOOTH | m.VC_WARM_START, plan=plan)
    O = m.vc_attn_forward(plan)
    assert m.vc_plan_status(plan) == (0, 0)
    allp = gpu_plan_all(m, plan)
    for h in range(2):
        g = head_of(allp, 0, h)
        v1 = u16(V1[0, h])
        assert np.array_equal(g["perm"], oracle.stable_argsort(g["labels"], cfg["k"]))
        _, _, J = oracle.kmeans(v1, cfg["k"], 2, init=cent0[0, h])
        Jg = oracle.kmeans_objective(v1, cfg["k"], g["labels"])
        assert abs(Jg - J[-1]) <= 0.01 * J[-1], f"head {h}: J_gpu {Jg} vs warm-started oracle {J[-1]}"
        o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), v1, cfg["k"], 2, perm=g["perm"])
        compare_prep(g, o, cfg["S"])
        rows = np.arange(0, cfg["S"], 7)
        assert_within(f64(O[0, h])[rows], oracle.forward_head(o, rows)[0], float(np.abs(f64(V1[0, h])).max()))
    plan.destroy()


def test_schedule_run_exercises_every_action(m):
    """A 10-step run with reuse 2: window ceil(10/4) = 3 steps -> group, reuse, warm group, then plain."""
    n_steps, reuse = 10, 2
    cfg = synth.custom(S=3000, D=64, H=2, k=24, iters=4, locality=True)
    Q, K, V = synth.make_inputs(cfg, seed=32, device="cuda")
    plan, prev_perm = None, None
    seen = []
    for s in range(5):
        act = m.vc_schedule_action(s, n_steps, reuse)
        seen.append(act)
        Vs = next_step(V, s)
        iters = 2 if act == m.VC_STEP_GROUP_WARM else 4
        plan = m.vc_attn_prepare_ex(Q, K, Vs, cfg["k"], iters, flags=m.STEP_PREPARE_FLAGS[act], plan=plan)
        O = m.vc_attn_forward(plan)
        assert m.vc_plan_status(plan) == (0, 0)
        allp = gpu_plan_all(m, plan)
        perm = allp["perm"].copy()
        if act in (m.VC_STEP_REUSE, m.VC_STEP_PLAIN):
            assert np.array_equal(perm, prev_perm), f"step {s}: pi must be kept"
        prev_perm = perm
        vsmooth = act != m.VC_STEP_PLAIN
        rows = np.arange(0, cfg["S"], 11)
        for h in range(2):
            g = head_of(allp, 0, h)
            o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(Vs[0, h]), cfg["k"], iters, perm=g["perm"],
                                    vsmooth=vsmooth)
            if not vsmooth:  # the plain kernel keeps pi but uses no means
                o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(Vs[0, h]), cfg["k"], iters, perm=g["perm"],
                                        vsmooth=True)
                o["mub"] = np.zeros_like(o["mub"])
                o["vsmooth"] = False
                dm = oracle.demean(u16(Vs[0, h]), g["perm"], subtract_mean=False)
                o.update(rc=dm["rc"], sv=dm["sv"], amax=dm["amax"], resid=dm["resid"])
            compare_prep(g, o, cfg["S"])
            got = f64(O[0, h])[rows]
            assert_within(got, oracle.forward_head(o, rows)[0], float(np.abs(f64(Vs[0, h])).max()), f"step {s} head {h}")
            rel_f, _ = errors(got, oracle_forward_from_plan(g, cfg["S"], rows, with_mean=vsmooth))
            assert rel_f <= 4e-3, f"step {s} head {h}: forward-only {rel_f:.3e}"
    assert seen == [m.VC_STEP_GROUP, m.VC_STEP_REUSE, m.VC_STEP_GROUP_WARM, m.VC_STEP_PLAIN, m.VC_STEP_PLAIN]
    plan.destroy()
