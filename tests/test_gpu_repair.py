"""GPU parity of the V residual repair ("Open-VC Attention", "Why V residual repair") through the C ABI.

The energies, the selected tokens, the copied keys' codes and scales and the repair residual codes are
compared bit for bit with the oracle; the forward meets the acceptance rule against the oracle's
quantised forward with repair, and the forward kernel alone is compared with the oracle run on the
GPU's own plan tensors.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_within, compare_prep, errors, f64, gpu_plan_all, head_of, u16, vc

FWD_ONLY_REL = 4e-3


@pytest.fixture(scope="module")
def m():
    return vc()


def heavy_inputs(S, D, H, seed, B=1):
    cfg = synth.custom(S, D=D, H=H, B=B, k=max(1, S // 128), iters=1)
    Q, K, V = synth.make_inputs(cfg, seed=seed, device="cuda")
    gen = torch.Generator().manual_seed(seed + 1)
    gain = torch.ones(S)
    gain[torch.randperm(S, generator=gen)[:max(1, S // 50)]] = 12.0
    V = (V.float() * gain.cuda()[None, None, :, None]).to(torch.bfloat16).contiguous()
    return Q, K, V


def plan_repair(m, plan):
    get = lambda what: m.vc_plan_get(plan, what).cpu().numpy()
    torch.cuda.synchronize()
    return {"idx": get(m.VC_PLAN_REPAIR_IDX), "energy": get(m.VC_PLAN_REPAIR_ENERGY),
            "kc": get(m.VC_PLAN_REPAIR_KCODES), "sk": get(m.VC_PLAN_REPAIR_KSCALES),
            "vt": get(m.VC_PLAN_REPAIR_VCODES)}


@pytest.mark.gpu
@pytest.mark.parametrize("S,D,n,flags", [
    (3000, 64, 15, 0),                 # one ragged repair tile (0.5% of S)
    (2049, 128, 200, "kcenter"),       # two repair tiles, copied keys centred
    (1000, 128, 130, "channel"),       # per-channel residual scales
    (300, 64, 300, 0),                 # every token repaired
    (1, 64, 1, 0),                     # one token: one key tile and one repair tile
    (129, 128, 129, "channel"),        # two ragged key tiles, two repair tiles, every token repaired
    (1000, 64, 50, "hadamard"),        # rotated Q and K, the copied keys rotated alike
    (700, 128, 20, "batch"),           # B = 2: each batch-head selects its own tokens
    (500, 64, 9, "batch"),
])
def test_repair_parity(m, S, D, n, flags):
    H, B = 2, 2 if flags == "batch" else 1
    Q, K, V = heavy_inputs(S, D, H, seed=S + n, B=B)
    f = {"kcenter": m.VC_KCENTER, "channel": m.VC_VSCALE_CHANNEL, "hadamard": m.VC_QK_HADAMARD}.get(flags, 0)
    plan = m.vc_attn_prepare_repair(Q, K, V, n, flags=f)
    assert plan.n_repair == n
    O = m.vc_attn_forward(plan, flags=m.VC_EXPCAST | m.VC_MIDWINDOW)
    assert m.vc_plan_status(plan) == (0, 0)
    allp = gpu_plan_all(m, plan)
    rp = plan_repair(m, plan)
    svc = m.vc_plan_get(plan, m.VC_PLAN_VCHSCALES).cpu().numpy()
    rows = np.arange(S)
    for b, h in ((b, h) for b in range(B) for h in range(H)):
        g = head_of(allp, b, h)
        o = oracle.prepare_head(u16(Q[b, h]), u16(K[b, h]), u16(V[b, h]), 1, 1, vsmooth=False,
                                kcenter=flags == "kcenter", vscale_channel=flags == "channel", n_repair=n,
                                hadamard=flags == "hadamard")
        if flags == "channel":
            assert np.array_equal(svc[b, h], o["sv"])
            assert np.array_equal(g["rc"], o["rc"]) and np.array_equal(g["qc"], o["qc"])
        else:
            compare_prep(g, o, S)
        orp = o["repair"]
        assert np.array_equal(rp["energy"][b, h], orp["energy"]), f"head {h}: energies"
        assert np.array_equal(rp["idx"][b, h], orp["idx"]), f"head {h}: selected tokens"
        assert np.array_equal(rp["kc"][b, h], orp["kc"]), f"head {h}: copied key codes"
        assert np.array_equal(rp["sk"][b, h], orp["sk"]), f"head {h}: copied key scales"
        assert np.array_equal(rp["vt"][b, h].T, orp["rc"]), f"head {h}: repair residual codes"
        ref, _, _ = oracle.forward_head(o, rows)
        got = f64(O[b, h])
        assert_within(got, ref, float(np.abs(f64(V[b, h])).max()), f"head {h}")
        sv = svc[b, h] if flags == "channel" else g["sv"]
        fl = oracle.EXPCAST | oracle.MIDWINDOW | (oracle.HADAMARD if flags == "hadamard" else 0)
        fwd = oracle.attention_quant(g["qc"], g["sq"], g["kc"], g["sk"], g["rc"], sv, None, S, rows, fl,
                                     repair={"n": n, "kc": rp["kc"][b, h], "sk": rp["sk"][b, h],
                                             "rc": rp["vt"][b, h].T})[0]
        rel_f, _ = errors(got, fwd)
        assert rel_f <= FWD_ONLY_REL, f"head {h}: forward-only rel-L2 {rel_f:.3e}"
    plan.destroy()


@pytest.mark.gpu
def test_repair_rows_are_applied(m):
    """Without repair rows the plan is the plain one, bit for bit; with every token repaired the GPU's
    output follows the oracle's repaired forward, not the unrepaired one."""
    S, D = 1500, 128
    Q, K, V = heavy_inputs(S, D, 1, seed=7)
    fl = m.VC_EXPCAST | m.VC_MIDWINDOW
    p0 = m.vc_attn_prepare_repair(Q, K, V, 0)
    assert p0.n_repair == 0
    pl = m.vc_attn_prepare_ex(Q, K, V, 1, 1, flags=0)
    O0 = m.vc_attn_forward(p0, flags=fl)
    assert torch.equal(O0, m.vc_attn_forward(pl, flags=fl))
    p1 = m.vc_attn_prepare_repair(Q, K, V, S)
    O1 = m.vc_attn_forward(p1, flags=fl)
    assert m.vc_plan_status(p1) == (0, 0)
    rows = np.arange(0, S, 5)
    q, k, v = u16(Q[0, 0]), u16(K[0, 0]), u16(V[0, 0])
    ref1, _, _ = oracle.forward_head(oracle.prepare_head(q, k, v, 1, 1, vsmooth=False, n_repair=S), rows)
    ref0, _, _ = oracle.forward_head(oracle.prepare_head(q, k, v, 1, 1, vsmooth=False), rows)
    e1, _ = errors(f64(O1[0, 0])[rows], ref1)
    e0, _ = errors(f64(O0[0, 0])[rows], ref1)
    assert e1 < 0.5 * e0, (e1, e0)  # the repair term is ~3x the bf16 rounding of O here
    assert errors(f64(O0[0, 0])[rows], ref0)[0] < 0.5 * e0
    for p in (p0, pl, p1):
        p.destroy()


@pytest.mark.gpu
def test_repair_plan_shape_is_fixed(m):
    S, D = 600, 64
    Q, K, V = heavy_inputs(S, D, 1, seed=9)
    p = m.vc_attn_prepare_repair(Q, K, V, 10)
    with pytest.raises(m.VCError):
        m.vc_attn_prepare_repair(Q, K, V, 11, plan=p)
    with pytest.raises(m.VCError):
        m.vc_attn_prepare_repair(Q, K, V, 10, flags=m.VC_VSMOOTH, plan=p)
    m.vc_attn_prepare_repair(Q, K, V, 10, plan=p)  # same shape: reused without allocation
    p.destroy()
