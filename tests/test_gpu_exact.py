"""The GPU forward against exact fp64 attention on the bf16 inputs ("VC-Attention" Sec. 3.1): the
quantised method's own error, measured on the oracle (i), is all the GPU shows -- the kernel adds only
its bf16 output rounding and fp32 accumulation order on top."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import errors, f64, head_of, gpu_plan_all, u16, vc

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,heads", [("tiny", (0,)), ("small", (0, 5))])
def test_error_against_exact_attention_is_the_methods_own(name, heads):
    m = vc()
    cfg = synth.config(name)
    Q, K, V = synth.make_inputs(cfg, seed=4, device="cuda")
    plan = m.vc_attn_prepare(Q, K, V, cfg["k"], cfg["iters"])
    O = m.vc_attn_forward(plan)
    torch.cuda.synchronize()
    assert m.vc_plan_status(plan) == (0, 0)
    allp = gpu_plan_all(m, plan)
    S = cfg["S"]
    rows = np.unique(np.random.default_rng(9).choice(S, min(S, 96), replace=False))
    for h in heads:
        q, k, v = u16(Q[0, h]), u16(K[0, h]), u16(V[0, h])
        exact = oracle.attention_exact(q, k, v, rows)
        o = oracle.prepare_head(q, k, v, cfg["k"], cfg["iters"], perm=head_of(allp, 0, h)["perm"])
        quant, _, _ = oracle.forward_head(o, rows)
        e_gpu, _ = errors(f64(O[0, h])[rows], exact)
        e_orc, _ = errors(quant, exact)
        assert e_gpu <= 0.08, f"head {h}: rel-L2 against exact attention {e_gpu:.4f}"
        assert abs(e_gpu - e_orc) <= 0.05 * e_orc + 2e-3, f"head {h}: GPU {e_gpu:.5f} vs oracle {e_orc:.5f}"
    plan.destroy()
