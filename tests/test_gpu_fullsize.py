"""Parity at the benchmark sizes on sampled outputs the oracle computes one row at a time.

Same launch configuration as bench.py (vc_attn_prepare + vc_attn_forward with the default flags).
For every head: the GPU's permutation is bit-exact against the oracle's argsort of the GPU labels,
and the forward on sampled rows (one whole query tile of the first head plus random rows of all
heads) meets the acceptance bound against the oracle fed the GPU's plan. On two heads the oracle
also recomputes the prepare outputs from the bf16 inputs (bit-exact) and runs its own k-means
(objective within 1%, "VC-Attention", Sec. 3.2).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import (assert_within, compare_prep, f64, gpu_plan_all, gpu_plan_one_head, head_of,
                         oracle_forward_from_plan, u16, vc)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return vc()


def check_fullsize(m, cfg, rows_per_head=6, tile_heads=(0,), prep_heads=(0,), kmeans_heads=(), seed=0):
    Q, K, V = synth.make_inputs(cfg, seed=seed, device="cuda")
    plan = m.vc_attn_prepare(Q, K, V, cfg["k"], cfg["iters"])
    O = m.vc_attn_forward(plan)
    torch.cuda.synchronize()
    assert m.vc_plan_status(plan)[0] == 0
    S = cfg["S"]
    rng = np.random.default_rng(seed + 7)
    allp = gpu_plan_all(m, plan)
    worst = 0.0
    for h in range(cfg["H"]):
        g = head_of(allp, 0, h)
        assert np.array_equal(g["perm"], oracle.stable_argsort(g["labels"], cfg["k"])), f"head {h}"
        if h in prep_heads:
            o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(V[0, h]), cfg["k"], cfg["iters"], perm=g["perm"])
            compare_prep(g, o, S)
        if h in kmeans_heads:
            vh = u16(V[0, h])
            _, _, J = oracle.kmeans(vh, cfg["k"], cfg["iters"])
            Jg = oracle.kmeans_objective(vh, cfg["k"], g["labels"])
            assert abs(Jg - J[-1]) <= 0.01 * J[-1], f"head {h}: J_gpu {Jg} vs J_oracle {J[-1]}"
        rows = rng.choice(S, rows_per_head, replace=False)
        if h in tile_heads:
            t = int(rng.integers(0, (S + 127) // 128))
            rows = np.concatenate([rows, np.arange(t * 128, min(S, t * 128 + 128)), [S - 1]])
        rows = np.unique(rows)
        ref = oracle_forward_from_plan(g, S, rows)
        got = f64(O[0, h])[rows]
        rel, _ = assert_within(got, ref, float(np.abs(f64(V[0, h])).max()), f"{cfg['name']} head {h}")
        worst = max(worst, rel)
    plan.destroy()
    return worst


def test_wan_fullsize(m):
    check_fullsize(m, synth.config("wan"), kmeans_heads=(3,), prep_heads=(0, 3))


def test_l1344_fullsize(m):
    # 10% of heads have near-uniform scores: every head is checked; the oracle's own k-means on head 1
    check_fullsize(m, synth.config("l1344"), prep_heads=(0,), kmeans_heads=(1,))


# The k-means objective acceptance (within 1% of the oracle's) on one point of each head dim.
SWEEP_KMEANS = {"sweep_d128_s16384": (2,), "sweep_d64_s65536": (2,)}


@pytest.mark.parametrize("name", ["sweep_d64_s4096", "sweep_d128_s16384", "sweep_d64_s65536", "sweep_d128_s131072"])
def test_sweep_points(m, name):
    check_fullsize(m, synth.config(name), rows_per_head=3, prep_heads=(1,), kmeans_heads=SWEEP_KMEANS.get(name, ()))


def test_wan_fullsize_repair(m):
    """The Open-VC configuration at the benchmark size: no V-Smooth, one V scale per head, the 0.5% of
    tokens with the largest residual energy repaired ("Open-VC Attention", "Why V residual repair").
    Selection, copied keys and repair codes bit-exact on two heads; sampled rows of every head within
    the acceptance bound of the oracle run on the GPU's plan."""
    cfg = synth.config("wan")
    S, H = cfg["S"], cfg["H"]
    n = m.repair_rows_for(S, 0.005)
    Q, K, V = synth.make_inputs(cfg, seed=1, device="cuda")
    plan = m.vc_attn_prepare_repair(Q, K, V, n)
    O = m.vc_attn_forward(plan, flags=m.VC_EXPCAST | m.VC_MIDWINDOW)
    torch.cuda.synchronize()
    assert m.vc_plan_status(plan)[0] == 0
    allp = gpu_plan_all(m, plan)
    get = lambda what: m.vc_plan_get(plan, what).cpu().numpy()
    idx, kc, sk, vt = (get(w) for w in (m.VC_PLAN_REPAIR_IDX, m.VC_PLAN_REPAIR_KCODES, m.VC_PLAN_REPAIR_KSCALES,
                                        m.VC_PLAN_REPAIR_VCODES))
    rng = np.random.default_rng(11)
    for h in range(H):
        g = head_of(allp, 0, h)
        rep = {"n": n, "kc": kc[0, h], "sk": sk[0, h], "rc": vt[0, h].T}
        if h in (0, 17):
            o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(V[0, h]), 1, 1, vsmooth=False, n_repair=n)
            compare_prep(g, o, S)
            for key, want in (("idx", o["repair"]["idx"]), ("kc", o["repair"]["kc"]), ("sk", o["repair"]["sk"]),
                              ("rc", o["repair"]["rc"])):
                got = idx[0, h] if key == "idx" else rep[key]
                assert np.array_equal(got, want), f"head {h}: repair {key}"
        rows = np.unique(np.concatenate([rng.choice(S, 6, replace=False), [S - 1]]))
        ref = oracle.attention_quant(g["qc"], g["sq"], g["kc"], g["sk"], g["rc"], g["sv"], None, S, rows, repair=rep)[0]
        assert_within(f64(O[0, h])[rows], ref, float(np.abs(f64(V[0, h])).max()), f"repair head {h}")
    plan.destroy()


def test_wan_fullsize_channel_scale_and_k_centering(m):
    """V-Smooth with one V scale per channel and centred keys at the benchmark size: prepare outputs
    bit-exact on one head (the oracle fed the GPU's permutation), sampled rows of every head."""
    cfg = synth.config("wan")
    S, H = cfg["S"], cfg["H"]
    Q, K, V = synth.make_inputs(cfg, seed=2, device="cuda")
    plan = m.vc_attn_prepare_ex(Q, K, V, cfg["k"], cfg["iters"],
                                flags=m.VC_VSMOOTH | m.VC_VSCALE_CHANNEL | m.VC_KCENTER)
    O = m.vc_attn_forward(plan)
    torch.cuda.synchronize()
    assert m.vc_plan_status(plan)[0] == 0
    allp = gpu_plan_all(m, plan)
    svc = m.vc_plan_get(plan, m.VC_PLAN_VCHSCALES).cpu().numpy()
    mt = u16(m.vc_plan_get(plan, m.VC_PLAN_MEANS_T))
    nkb = (S + 127) // 128
    rng = np.random.default_rng(12)
    for h in range(H):
        g = head_of(allp, 0, h)
        if h == 5:
            o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(V[0, h]), cfg["k"], cfg["iters"], perm=g["perm"],
                                    kcenter=True, vscale_channel=True)
            for key in ("qc", "sq", "kc", "sk", "mub", "rc"):
                assert np.array_equal(g[key], o[key]), f"head {h}: {key}"
            assert np.array_equal(svc[0, h], o["sv"]) and np.array_equal(mt[0, h, :, :nkb].T, o["mut"])
        rows = np.unique(np.concatenate([rng.choice(S, 6, replace=False), [0]]))
        ref = oracle.attention_quant(g["qc"], g["sq"], g["kc"], g["sk"], g["rc"], svc[0, h], g["mub"], S, rows,
                                     mut=mt[0, h, :, :nkb].T)[0]
        assert_within(f64(O[0, h])[rows], ref, float(np.abs(f64(V[0, h])).max()), f"channel head {h}")
    plan.destroy()


def test_maximum_sequence_length_past_two_gig_elements(m):
    """The largest S and k the boundary accepts (2^20 tokens, 1024 clusters), with enough heads that every
    per-tensor element count passes 2^31 (17 * 2^20 * 128): the last head's codes, means and output sit past
    the 32-bit offset range. Inputs are seeded Gaussians drawn on the device (q, k std 0.5, v std 1) with one
    token in 200 of V scaled by 30, as outlier rows."""
    S, H, D, k = 1 << 20, 17, 128, 1024
    gen = torch.Generator(device="cuda").manual_seed(11)
    Q = (0.5 * torch.randn(1, H, S, D, device="cuda", generator=gen)).to(torch.bfloat16)
    K = (0.5 * torch.randn(1, H, S, D, device="cuda", generator=gen)).to(torch.bfloat16)
    V = torch.randn(1, H, S, D, device="cuda", generator=gen)
    V[:, :, torch.randperm(S, device="cuda", generator=gen)[:S // 200]] *= 30.0
    V = V.to(torch.bfloat16)
    plan = m.vc_attn_prepare(Q, K, V, k, 1)
    O = m.vc_attn_forward(plan)
    torch.cuda.synchronize()
    assert m.vc_plan_status(plan) == (0, 0)
    rng = np.random.default_rng(12)
    for h, prep in ((H - 1, True), (0, False)):
        g = gpu_plan_one_head(m, plan, 0, h)
        assert np.array_equal(g["perm"], oracle.stable_argsort(g["labels"], k)), f"head {h}"
        if prep:
            o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(V[0, h]), k, 1, perm=g["perm"])
            compare_prep(g, o, S)
        rows = np.unique(np.concatenate([rng.choice(S, 3, replace=False), [S - 1]]))
        ref = oracle_forward_from_plan(g, S, rows)
        got = f64(O[0, h][torch.as_tensor(rows, device=O.device)])
        assert_within(got, ref, float(V[0, h].float().abs().max()), f"max-S head {h}")
    plan.destroy()
