"""The allocation-free entry point agrees with the regular prepare step.

vc_residual_pack_noalloc serves callers that must not allocate device memory (for instance a
framework whose pool already owns the whole device): its only scratch is a fixed array inside the
library. This test calls it through the C ABI twice in a row -- first on a large-magnitude V, then
on a small one, so a residual maximum left over from the first call would corrupt the second -- and
compares the means, residual codes and scales bit for bit with what vc_attn_prepare writes into a
plan for the same V and permutation. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import synth
from gpu_helpers import vc

pytestmark = pytest.mark.gpu


def test_noalloc_matches_prepare_on_two_calls_in_a_row():
    m = vc()
    L = m.lib()
    cfg = synth.custom(1000, D=128, H=3, k=7, iters=2, outlier_frac=0.01)
    Q, K, V0 = synth.make_inputs(cfg, seed=21, device="cuda")
    B, H, S, D = V0.shape
    stream = torch.cuda.current_stream()
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
        rc = L.vc_residual_pack_noalloc(V.data_ptr(), perm.data_ptr(), B, H, S, D, means.data_ptr(),
                                        codes.data_ptr(), scales.data_ptr(), stream.cuda_stream)
        assert rc == 0, m.vc_strerror(rc)
        torch.cuda.synchronize()
        assert torch.equal(means.view(torch.int16), ref_means.view(torch.int16))
        assert torch.equal(codes, ref_codes)
        assert torch.equal(scales, ref_scales)
        plan.destroy()


def test_noalloc_rejects_more_heads_than_its_scratch():
    m = vc()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    rc = m.lib().vc_residual_pack_noalloc(fake, None, 1, m.VC_NOALLOC_MAX_HEADS + 1, 128, 128, fake, fake, fake,
                                          None)
    assert rc == m.VC_ERR_UNSUPPORTED
