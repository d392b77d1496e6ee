"""GPU parity through the C ABI against the CPU oracle on seeded synthetic inputs.

The forward follows "VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention"
(Eq. 1, 3-7) and "Open-VC Attention" ("Scheduling around ExpCast"). Acceptance: ExpCast codes and
argsort permutations bit-exact; O within rel-L2 1e-2 and max-abs 3e-2 max|V| per head against the
quantised oracle fed the GPU's permutation; the k-means objective within 1% of the oracle's.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import (assert_within, compare_prep, errors, f64, gpu_plan_all, gpu_plan_head, head_of,
                         oracle_forward_from_plan, u16, vc)

pytestmark = pytest.mark.gpu

# Forward-only comparison (oracle run on the GPU's own codes): the two sides differ only by the
# tensor core's fp32 accumulation order for S and PV, ex2.approx for the rescale factor, the
# rank-16 mean update in fp32 and the final bf16 rounding (2^-9 relative), so a much tighter bound
# than the end-to-end acceptance applies.
FWD_ONLY_REL = 4e-3


@pytest.fixture(scope="module")
def m():
    return vc()


def test_expcast_encode_bit_exact(m):
    rng = np.random.default_rng(0)
    n = 1 << 20
    M = rng.normal(0, 300, n).astype(np.float32)
    a = rng.uniform(1e-3, 2.0, n).astype(np.float32)
    s = (M / a + rng.normal(0, 40, n)).astype(np.float32)
    b = (np.float32(119.65) - M).astype(np.float32)
    s[:8] = [0, -0.0, 1e30, -1e30, 3.4e38, -3.4e38, 1e-40, -1e-40]
    want = oracle.expcast_codes(s, a, b)
    got = m.vc_expcast_encode(*(torch.from_numpy(x).cuda() for x in (s, a, b))).cpu().numpy()
    assert np.array_equal(got, want)
    assert (want == 120).any() and (want == 0).any() and ((want > 0) & (want < 120)).mean() > 0.3


def test_expcast_fast_path_bytes_need_no_clamp(m):
    """The forward writes its codes without the clamp at 120 while |M| < 2^22 (M the running max in code
    units, every score of the row with fl(s*a) <= M). The unclamped export is that exact code path: on
    such (s, a, M) its bytes must equal the clipped codes of Eq. 7 ("VC-Attention" Sec. 3.3), including
    the row maxima themselves (fl(s*a) == M -> 120) and M at the edge of the range."""
    rng = np.random.default_rng(3)
    n = 1 << 20
    a = rng.uniform(1e-3, 2.0, n).astype(np.float32)
    lim = np.float32(4194304.0)
    top = rng.uniform(-1.0, 1.0, n) * rng.choice([30.0, 3e3, 4.19e6], n)   # fl(s*a) of the row max
    s = (top / a).astype(np.float32)
    sa = (s * a).astype(np.float32)                                       # fp32 product, one rounding
    gap = np.where(rng.random(n) < 0.25, 0.0, np.abs(rng.normal(0, 40, n)))  # 25%: the score is the max
    M = (sa + gap).astype(np.float32)
    M = np.maximum(M, sa)                                                 # fl(s*a) <= M after rounding too
    keep = np.abs(M) < lim
    s, a, M = s[keep], a[keep], M[keep]
    b = (np.float32(119.65) - M).astype(np.float32)
    assert np.all((s * a).astype(np.float32) <= M)
    want = oracle.expcast_codes(s, a, b)
    got = m.vc_expcast_encode(*(torch.from_numpy(x).cuda() for x in (s, a, b)), clamp=False).cpu().numpy()
    assert np.array_equal(got, want)
    assert (want == 120).mean() > 0.2 and (want == 0).any() and np.abs(M).max() > 4e6


def run(m, cfg, seed=0, vsmooth=True, perm=None):
    Q, K, V = synth.make_inputs(cfg, seed=seed, device="cuda")
    plan = m.vc_attn_prepare_ex(Q, K, V, cfg["k"], cfg["iters"], perm=perm, flags=m.VC_VSMOOTH if vsmooth else 0)
    torch.cuda.synchronize()
    return Q, K, V, plan


def check_config(m, cfg, rows_per_head=None, kmeans_heads=None, seed=0):
    Q, K, V, plan = run(m, cfg, seed)
    O = m.vc_attn_forward(plan)
    torch.cuda.synchronize()
    assert m.vc_plan_status(plan)[0] == 0
    S = cfg["S"]
    rng = np.random.default_rng(seed + 1)
    allp = gpu_plan_all(m, plan)
    for b in range(cfg["B"]):
        for h in range(cfg["H"]):
            g = head_of(allp, b, h)
            qh, kh, vh = u16(Q[b, h]), u16(K[b, h]), u16(V[b, h])
            # argsort: bit-exact given the GPU's labels
            assert np.array_equal(g["perm"], oracle.stable_argsort(g["labels"], cfg["k"]))
            if kmeans_heads is None or h in kmeans_heads:
                _, _, J = oracle.kmeans(vh, cfg["k"], cfg["iters"])
                Jg = oracle.kmeans_objective(vh, cfg["k"], g["labels"])
                assert abs(Jg - J[-1]) <= 0.01 * J[-1], f"head {h}: J_gpu {Jg} vs J_oracle {J[-1]}"
            o = oracle.prepare_head(qh, kh, vh, cfg["k"], cfg["iters"], perm=g["perm"])
            compare_prep(g, o, S)
            if rows_per_head is None:
                rows = np.arange(S)
            else:
                tiles = rng.choice((S + 127) // 128, size=min(2, (S + 127) // 128), replace=False)
                rows = np.unique(np.concatenate([np.arange(t * 128, min(S, t * 128 + 128)) for t in tiles] +
                                                [rng.choice(S, rows_per_head, replace=False), [0, S - 1]]))
            ref, _, _ = oracle.forward_head(o, rows)
            got = f64(O[b, h])[rows]
            vmax = float(np.abs(f64(V[b, h])).max())
            assert_within(got, ref, vmax, f"head {h}")
            rel_f, _ = errors(got, oracle_forward_from_plan(g, S, rows))
            assert rel_f <= FWD_ONLY_REL, f"head {h}: forward-only rel-L2 {rel_f:.3e}"
    plan.destroy()


def test_tiny_config_all_rows(m):
    check_config(m, synth.config("tiny"))


def test_small_config_sampled_rows(m):
    check_config(m, synth.config("small"), rows_per_head=64, kmeans_heads={0, 5})


@pytest.mark.parametrize("S,D", [(1, 128), (127, 128), (129, 64), (255, 128), (300, 64), (1000, 128), (2049, 64)])
def test_ragged_shapes(m, S, D):
    cfg = synth.custom(S, D=D, H=2, k=max(1, min(S, S // 100 + 1)), iters=2)
    check_config(m, cfg)


@pytest.mark.parametrize("S,D", [(300, 64), (257, 128)])
def test_batch_dimension(m, S, D):
    """B > 1: every (b, h) pair is its own head in the plan and in the output."""
    cfg = synth.custom(S, D=D, H=3, B=2, k=3, iters=2)
    check_config(m, cfg)


@pytest.mark.parametrize("expcast,midwindow,vsmooth", [(False, True, True), (True, False, True),
                                                       (True, True, False), (False, False, False)])
def test_ablations(m, expcast, midwindow, vsmooth):
    cfg = synth.custom(700, D=128, H=2, k=6, iters=3, outlier_frac=0.01)
    Q, K, V, plan = run(m, cfg, seed=3, vsmooth=vsmooth)
    flags = (m.VC_EXPCAST if expcast else 0) | (m.VC_MIDWINDOW if midwindow else 0) | m.VC_VSMOOTH
    O = m.vc_attn_forward(plan, flags=flags)
    torch.cuda.synchronize()
    allp = gpu_plan_all(m, plan)
    for h in range(2):
        g = head_of(allp, 0, h)
        o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(V[0, h]), 6, 3, vsmooth=vsmooth,
                                perm=g["perm"] if vsmooth else None)
        compare_prep(g, o, 700)
        rows = np.arange(700)
        ref, _, _ = oracle.forward_head(o, rows, expcast=expcast, midwindow=midwindow)
        assert_within(f64(O[0, h]), ref, float(np.abs(f64(V[0, h])).max()), f"head {h}")


def test_explicit_permutation_and_plan_reuse(m):
    cfg = synth.custom(513, D=128, H=2, k=5, iters=2)
    Q, K, V = synth.make_inputs(cfg, seed=4, device="cuda")
    perm = torch.stack([torch.randperm(513, generator=torch.Generator().manual_seed(i)) for i in range(2)])
    perm = perm.to(torch.int32).reshape(1, 2, 513).cuda().contiguous()
    plan = m.vc_attn_prepare_ex(Q, K, V, 5, 2, perm=perm)
    O1 = m.vc_attn_forward(plan).clone()
    plan2 = m.vc_attn_prepare_ex(Q, K, V, 5, 2, perm=perm, plan=plan)  # reuse: no allocation
    assert plan2 is plan
    O2 = m.vc_attn_forward(plan)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2)
    for h in range(2):
        o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(V[0, h]), 5, 2, perm=perm[0, h].cpu().numpy())
        ref, _, _ = oracle.forward_head(o, np.arange(513))
        assert_within(f64(O1[0, h]), ref, float(np.abs(f64(V[0, h])).max()))
    # a plan of another shape is refused and left intact
    Q2, K2, V2 = (t[:, :, :256].contiguous() for t in (Q, K, V))
    with pytest.raises(m.VCError) as e:
        m.vc_attn_prepare(Q2, K2, V2, 5, 2, plan=plan)
    assert e.value.rc == m.VC_ERR_PLAN_MISMATCH
    O3 = m.vc_attn_forward(plan)
    torch.cuda.synchronize()
    assert torch.equal(O1, O3)
    plan.destroy()


def test_forced_timeout_reports_status_and_recovers(m):
    cfg = synth.custom(384, D=128, H=1, k=3, iters=2)
    Q, K, V, plan = run(m, cfg, seed=5)
    m.vc_attn_forward(plan, flags=m.VC_FLAGS_DEFAULT | m.VC_DEBUG_TIMEOUT)
    rc, bits = m.vc_plan_status(plan)
    assert rc == m.VC_ERR_TIMEOUT and bits != 0
    O = m.vc_attn_forward(plan)  # the context is still usable and the next call is clean
    rc, bits = m.vc_plan_status(plan)
    assert rc == 0 and bits == 0
    g = gpu_plan_head(m, plan, 0, 0)
    ref = oracle_forward_from_plan(g, 384, np.arange(384))
    rel, _ = errors(f64(O[0, 0]), ref)
    assert rel <= FWD_ONLY_REL
    plan.destroy()


def test_forward_is_deterministic(m):
    """The forward has no data races: the same plan gives bitwise identical outputs."""
    cfg = synth.config("small")
    Q, K, V, plan = run(m, cfg, seed=9)
    O1 = m.vc_attn_forward(plan).clone()
    for _ in range(3):
        O2 = m.vc_attn_forward(plan)
        torch.cuda.synchronize()
        assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    plan.destroy()


@pytest.mark.parametrize("D", [64, 128])
def test_repeated_launches_never_stall(m, D):
    """Many back-to-back launches over every flag combination finish without a wait running out.

    The softmax groups, the MMA thread and the two load warps hand tiles around through mbarrier
    phases; a parity wait that could see its barrier two phases ahead would stall only under some
    interleavings, so the check is statistical: 4 flag sets x 12 launches on a 256-tile sequence.
    """
    S = 32768
    cfg = synth.custom(S=S, D=D, H=4, k=S // 128, iters=2)
    Q, K, V = synth.make_inputs(cfg, seed=21, device="cuda")
    plan = m.vc_attn_prepare(Q, K, V, cfg["k"], cfg["iters"])
    base = m.VC_EXPCAST | m.VC_VSMOOTH | m.VC_MIDWINDOW
    for flags in (base, base & ~m.VC_MIDWINDOW, base & ~m.VC_VSMOOTH, m.VC_EXPCAST):
        ref = None
        for rep in range(12):
            O = m.vc_attn_forward(plan, flags=flags)
            rc, bits = m.vc_plan_status(plan)
            assert rc == 0 and bits == 0, f"flags {flags} launch {rep}: status bits {bits}"
            if ref is None:
                ref = O.clone()
            else:
                assert torch.equal(ref.view(torch.int16), O.view(torch.int16)), f"flags {flags} launch {rep}"
    plan.destroy()


def test_huge_scores_take_the_clamped_code_path(m):
    """Row maxima far beyond 2^22 code units: the forward's byte-wise clip at 120 ("VC-Attention", Sec. 3.3
    Eq. 7) is exercised. Q = K = +-224 per element, so every row's own key scores 224^2 * sqrt(128) ~ 5.7e5,
    i.e. ~6.5e6 code units, while every other key scores far lower: P is one-hot and O is close to V of the
    row's own token."""
    S, D, H = 1024, 128, 2
    assert 224.0**2 * D / math.sqrt(D) * 8.0 / math.log(2.0) > 2.0**22
    gen = torch.Generator().manual_seed(31)
    signs = torch.randint(0, 2, (1, H, S, D), generator=gen).float() * 2 - 1
    Q = (224.0 * signs).to(torch.bfloat16).cuda()
    K = Q.clone()
    V = torch.randn(1, H, S, D, generator=gen).to(torch.bfloat16).cuda()
    plan = m.vc_attn_prepare(Q, K, V, 8, 2)
    O = m.vc_attn_forward(plan)
    assert m.vc_plan_status(plan) == (0, 0)
    allp = gpu_plan_all(m, plan)
    rows = np.arange(S)
    for h in range(H):
        g = head_of(allp, 0, h)
        rel, _ = errors(f64(O[0, h]), oracle_forward_from_plan(g, S, rows))
        assert rel <= FWD_ONLY_REL, f"head {h}: rel-L2 {rel:.3e}"
    plan.destroy()


@pytest.mark.parametrize("S,D", [(3000, 64), (2049, 128)])
def test_k_centering(m, S, D):
    """VC_KCENTER ("VC-Attention", Sec. 3.4 "Fused preprocessing", App. B): keys with large per-channel
    offsets. The GPU's channel centre and every prepare output are bit-exact against the oracle fed the
    GPU's permutation, and the forward meets the acceptance bound."""
    cfg = synth.custom(S, D=D, H=2, k=max(1, S // 128), iters=2)
    Q, K, V = synth.make_inputs(cfg, seed=11, device="cuda")
    gen = torch.Generator().manual_seed(12)
    offset = (torch.randn(D, generator=gen) * 8.0).cuda()
    K = (K.float() + offset).to(torch.bfloat16).contiguous()
    plan = m.vc_attn_prepare_ex(Q, K, V, cfg["k"], cfg["iters"], flags=m.VC_VSMOOTH | m.VC_KCENTER)
    O = m.vc_attn_forward(plan)
    assert m.vc_plan_status(plan) == (0, 0)
    allp = gpu_plan_all(m, plan)
    kmu = u16(m.vc_plan_get(plan, m.VC_PLAN_KCENTER))
    rows = np.arange(S)
    for h in range(2):
        g = head_of(allp, 0, h)
        o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(V[0, h]), cfg["k"], cfg["iters"], perm=g["perm"],
                                kcenter=True)
        assert np.array_equal(kmu[0, h], o["kmu"]), f"head {h}: channel centre"
        compare_prep(g, o, S)
        ref, _, _ = oracle.forward_head(o, rows)
        got = f64(O[0, h])
        assert_within(got, ref, float(np.abs(f64(V[0, h])).max()), f"head {h}")
        rel_f, _ = errors(got, oracle_forward_from_plan(g, S, rows))
        assert rel_f <= FWD_ONLY_REL, f"head {h}: forward-only rel-L2 {rel_f:.3e}"
    plan.destroy()


@pytest.mark.gpu
@pytest.mark.parametrize("S,D,vsmooth", [(3000, 64, True), (2049, 128, True), (1000, 128, False)])
def test_per_channel_v_scale(m, S, D, vsmooth):
    """VC_VSCALE_CHANNEL ("VC-Attention", Sec. 3.2 "Block demeaning", App. B): values with a few outlier
    channels 2^12 wider than the rest. Channel scales, residual codes and the scaled means the forward
    reads are bit-exact against the oracle fed the GPU's permutation; the forward meets the acceptance
    rule on every channel separately (max-abs against that channel's own max |V|)."""
    cfg = synth.custom(S, D=D, H=2, k=max(1, S // 128), iters=2)
    Q, K, V = synth.make_inputs(cfg, seed=21, device="cuda")
    gen = torch.Generator().manual_seed(22)
    wide = torch.randperm(D, generator=gen)[:3]
    gain = torch.ones(D)
    gain[wide] = 4096.0
    V = (V.float() * gain.cuda()).to(torch.bfloat16).contiguous()
    flags = (m.VC_VSMOOTH if vsmooth else 0) | m.VC_VSCALE_CHANNEL
    plan = m.vc_attn_prepare_ex(Q, K, V, cfg["k"], cfg["iters"], flags=flags)
    O = m.vc_attn_forward(plan)
    assert m.vc_plan_status(plan) == (0, 0)
    allp = gpu_plan_all(m, plan)
    svc = m.vc_plan_get(plan, m.VC_PLAN_VCHSCALES).cpu().numpy()
    mt = u16(m.vc_plan_get(plan, m.VC_PLAN_MEANS_T))
    nkb = (S + 127) // 128
    rows = np.arange(S)
    for h in range(2):
        g = head_of(allp, 0, h)
        o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(V[0, h]), cfg["k"], cfg["iters"],
                                vsmooth=vsmooth, perm=g["perm"] if vsmooth else None, vscale_channel=True)
        assert np.array_equal(svc[0, h], o["sv"]), f"head {h}: channel scales"
        assert g["sv"] == np.float32(o["sv"].max()), f"head {h}: head scale"
        assert np.array_equal(g["rc"], o["rc"]), f"head {h}: residual codes"
        assert np.array_equal(g["mub"], o["mub"]), f"head {h}: block means"
        for key in ("qc", "sq", "kc", "sk"):
            assert np.array_equal(g[key], o[key]), f"head {h}: {key}"
        assert np.array_equal(mt[0, h, :, :nkb].T, o["mut"]), f"head {h}: scaled means"
        assert not mt[0, h, :, nkb:].any()
        ref, _, _ = oracle.forward_head(o, rows)
        got = f64(O[0, h])
        Vh = np.abs(f64(V[0, h]))
        for d in range(D):
            rel, mx = errors(got[:, d], ref[:, d])
            assert rel <= 1e-2 and mx <= 3e-2 * Vh[:, d].max(), f"head {h} channel {d}: rel {rel:.3e} max {mx:.3e}"
        fwd = oracle.attention_quant(g["qc"], g["sq"], g["kc"], g["sk"], g["rc"], svc[0, h], g["mub"] if vsmooth
                                     else None, S, rows, mut=mt[0, h, :, :nkb].T if vsmooth else None)[0]
        rel_f, _ = errors(got, fwd)
        assert rel_f <= FWD_ONLY_REL, f"head {h}: forward-only rel-L2 {rel_f:.3e}"
    plan.destroy()


@pytest.mark.gpu
def test_per_head_plan_reports_equal_channel_scales(m):
    cfg = synth.custom(700, D=64, H=1, k=5, iters=2)
    Q, K, V = synth.make_inputs(cfg, seed=23, device="cuda")
    plan = m.vc_attn_prepare(Q, K, V, cfg["k"], cfg["iters"])
    sv = m.vc_plan_get(plan, m.VC_PLAN_VSCALES).cpu().numpy()
    svc = m.vc_plan_get(plan, m.VC_PLAN_VCHSCALES).cpu().numpy()
    assert np.array_equal(svc[0, 0], np.full(64, sv[0, 0], dtype=np.float32))
    mt = u16(m.vc_plan_get(plan, m.VC_PLAN_MEANS_T))
    mub = u16(m.vc_plan_get(plan, m.VC_PLAN_MEANS))
    assert np.array_equal(mt[0, 0, :, :6].T, mub[0, 0])  # true units without per-channel scales
    plan.destroy()


@pytest.mark.gpu
@pytest.mark.parametrize("S,D,kcenter", [(3000, 128, False), (2049, 64, True)])
def test_qk_hadamard(m, S, D, kcenter):
    """VC_QK_HADAMARD ("VC-Attention", Sec. 3.4 "Fused preprocessing", App. B): Q and K rows rotated by the
    Walsh-Hadamard butterfly before their quantisation. Codes and scales bit-exact against the oracle fed
    the GPU's permutation; the forward within the acceptance bound, and against the oracle on its plan."""
    cfg = synth.custom(S, D=D, H=2, k=max(1, S // 128), iters=2)
    Q, K, V = synth.make_inputs(cfg, seed=31, device="cuda")
    flags = m.VC_VSMOOTH | m.VC_QK_HADAMARD | (m.VC_KCENTER if kcenter else 0)
    plan = m.vc_attn_prepare_ex(Q, K, V, cfg["k"], cfg["iters"], flags=flags)
    O = m.vc_attn_forward(plan)
    assert m.vc_plan_status(plan) == (0, 0)
    allp = gpu_plan_all(m, plan)
    rows = np.arange(S)
    fl = oracle.EXPCAST | oracle.MIDWINDOW | oracle.HADAMARD
    for h in range(2):
        g = head_of(allp, 0, h)
        o = oracle.prepare_head(u16(Q[0, h]), u16(K[0, h]), u16(V[0, h]), cfg["k"], cfg["iters"], perm=g["perm"],
                                kcenter=kcenter, hadamard=True)
        compare_prep(g, o, S)
        ref, _, _ = oracle.forward_head(o, rows)
        got = f64(O[0, h])
        assert_within(got, ref, float(np.abs(f64(V[0, h])).max()), f"head {h}")
        fwd = oracle.attention_quant(g["qc"], g["sq"], g["kc"], g["sk"], g["rc"], g["sv"], g["mub"], S, rows, fl)[0]
        rel_f, _ = errors(got, fwd)
        assert rel_f <= FWD_ONLY_REL, f"head {h}: forward-only rel-L2 {rel_f:.3e}"
    plan.destroy()
