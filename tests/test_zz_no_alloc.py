"""The allocation-free entry point agrees with the regular prepare step and with the oracle.

vc_residual_pack_noalloc serves callers that must not allocate device memory (for instance a
framework whose pool already owns the whole device): its only scratch is a fixed array inside the
library. These tests call it through the C ABI twice in a row -- first on a large-magnitude V, then
on a small one, so a residual maximum left over from the first call would corrupt the second -- and
compare the means, residual codes and scales bit for bit with what vc_attn_prepare writes into a
plan for the same V and permutation, and with the oracle's demeaning of the same rows. Both head
dims are covered, and so is the identity permutation (perm = NULL). This file is collected last on
purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import u16, vc

pytestmark = pytest.mark.gpu


def _noalloc(m, V, perm, means, codes, scales):
    B, H, S, D = V.shape
    rc = m.lib().vc_residual_pack_noalloc(V.data_ptr(), None if perm is None else perm.data_ptr(), B, H, S, D,
                                          means.data_ptr(), codes.data_ptr(), scales.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
    assert rc == 0, m.vc_strerror(rc)
    torch.cuda.synchronize()


def _check_against_oracle(V, perm, means, codes, scales):
    """Every head against the oracle's gather + block means + per-head residual codes."""
    B, H, S, D = V.shape
    g_means, g_codes, g_scales = u16(means), codes.cpu().numpy(), scales.cpu().numpy()
    for b in range(B):
        for h in range(H):
            p = None if perm is None else perm[b, h].cpu().numpy()
            o = oracle.demean(V[b, h].cpu(), p)
            assert np.array_equal(g_means[b, h], o["mub"]), f"head {b},{h}: block means differ from the oracle"
            assert np.array_equal(np.ascontiguousarray(g_codes[b, h].T), o["rc"]), \
                f"head {b},{h}: residual codes differ from the oracle"
            assert g_scales[b, h] == np.float32(o["sv"]), f"head {b},{h}: V scale differs from the oracle"


@pytest.mark.parametrize("D", [128, 64])
def test_noalloc_matches_prepare_and_oracle_on_two_calls_in_a_row(D):
    m = vc()
    cfg = synth.custom(1000, D=D, H=3, k=7, iters=2, outlier_frac=0.01)
    Q, K, V0 = synth.make_inputs(cfg, seed=21, device="cuda")
    for scale in (8.0, 0.5):
        V = (V0.float() * scale).to(torch.bfloat16).contiguous()
        plan = m.vc_attn_prepare(Q, K, V, cfg["k"], cfg["iters"])
        perm = m.vc_plan_get(plan, m.VC_PLAN_PERM)
        ref_means = m.vc_plan_get(plan, m.VC_PLAN_MEANS)
        ref_codes = m.vc_plan_get(plan, m.VC_PLAN_VCODES)
        ref_scales = m.vc_plan_get(plan, m.VC_PLAN_VSCALES)
        means = torch.full_like(ref_means, 7.0)
        codes = torch.full_like(ref_codes, 0x55)
        scales = torch.full_like(ref_scales, -1.0)
        torch.cuda.synchronize()
        _noalloc(m, V, perm, means, codes, scales)
        assert torch.equal(means.view(torch.int16), ref_means.view(torch.int16))
        assert torch.equal(codes, ref_codes)
        assert torch.equal(scales, ref_scales)
        _check_against_oracle(V, perm, means, codes, scales)
        plan.destroy()


@pytest.mark.parametrize("D", [128, 64])
def test_noalloc_identity_permutation(D):
    """perm = NULL is the identity: equal to the plan path given an explicit identity permutation."""
    m = vc()
    cfg = synth.custom(777, D=D, H=2, k=5, iters=1, outlier_frac=0.01)
    Q, K, V = synth.make_inputs(cfg, seed=5, device="cuda")
    B, H, S, _ = V.shape
    ident = torch.arange(S, dtype=torch.int32, device="cuda").repeat(B * H, 1).view(B, H, S).contiguous()
    plan = m.vc_attn_prepare_ex(Q, K, V, cfg["k"], cfg["iters"], perm=ident, flags=m.VC_VSMOOTH)
    ref_means = m.vc_plan_get(plan, m.VC_PLAN_MEANS)
    ref_codes = m.vc_plan_get(plan, m.VC_PLAN_VCODES)
    ref_scales = m.vc_plan_get(plan, m.VC_PLAN_VSCALES)
    for _ in range(2):
        means = torch.full_like(ref_means, -3.0)
        codes = torch.full_like(ref_codes, 0x11)
        scales = torch.full_like(ref_scales, -1.0)
        _noalloc(m, V, None, means, codes, scales)
        assert torch.equal(means.view(torch.int16), ref_means.view(torch.int16))
        assert torch.equal(codes, ref_codes)
        assert torch.equal(scales, ref_scales)
    _check_against_oracle(V, None, means, codes, scales)
    plan.destroy()


def test_noalloc_rejects_bad_arguments_before_touching_memory():
    m = vc()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the argument checks come first
    L = m.lib()
    rc = L.vc_residual_pack_noalloc(fake, None, 1, m.VC_NOALLOC_MAX_HEADS + 1, 128, 128, fake, fake, fake, None)
    assert rc == m.VC_ERR_UNSUPPORTED
    misaligned = ctypes.c_void_p((1 << 20) + 2)
    rc = L.vc_residual_pack_noalloc(fake, misaligned, 1, 1, 128, 128, fake, fake, fake, None)
    assert rc == m.VC_ERR_INVALID_ARG
