"""A prepare into an existing plan and the forward allocate nothing and are stream-ordered, so a CUDA graph
can capture both; replaying it on new inputs gives the same bits as eager calls on a fresh plan."""
import pytest
import torch

import synth
from gpu_helpers import vc

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D,vsmooth", [(128, True), (64, True), (128, False)])
def test_prepare_and_forward_replay_in_a_cuda_graph(D, vsmooth):
    m = vc()
    cfg = synth.custom(2049, D=D, H=2, k=16, iters=2)
    flags = m.VC_VSMOOTH if vsmooth else 0
    Q, K, V = synth.make_inputs(cfg, seed=1, device="cuda")
    Qs, Ks, Vs = Q.clone(), K.clone(), V.clone()
    O = torch.empty_like(Q)
    plan = m.vc_attn_prepare_ex(Qs, Ks, Vs, cfg["k"], cfg["iters"], flags=flags)
    m.vc_attn_forward(plan, O)  # eager first call: launch attributes are set outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        m.vc_attn_prepare_ex(Qs, Ks, Vs, cfg["k"], cfg["iters"], flags=flags, plan=plan)
        m.vc_attn_forward(plan, O)
    for seed in (2, 3):
        Q2, K2, V2 = synth.make_inputs(cfg, seed=seed, device="cuda")
        Qs.copy_(Q2)
        Ks.copy_(K2)
        Vs.copy_(V2)
        graph.replay()
        torch.cuda.synchronize()
        assert m.vc_plan_status(plan) == (0, 0)
        fresh = m.vc_attn_prepare_ex(Q2, K2, V2, cfg["k"], cfg["iters"], flags=flags)
        ref = m.vc_attn_forward(fresh)
        torch.cuda.synchronize()
        assert torch.equal(O, ref), f"seed {seed}"
        fresh.destroy()
    plan.destroy()


def test_step_kernel_count_is_counted_from_the_captured_graph():
    """bench.py reports gpu_launches from the kernel nodes of the captured prepare and forward; they match the
    step's structure: Q quantisation, k-means initialisation, five kernels per Lloyd round (assignment, label
    histogram, scan, scatter, update), K' quantisation, block means, residual pack, and the forward."""
    import bench

    m = vc()
    cfg = synth.custom(4096, D=128, H=2, k=32, iters=3)
    Q, K, V = synth.make_inputs(cfg, seed=3, device="cuda")
    plan = m.vc_attn_prepare(Q, K, V, cfg["k"], cfg["iters"])
    O = m.vc_attn_forward(plan)
    torch.cuda.synchronize()
    n_prep = bench.count_kernels(lambda: m.vc_attn_prepare(Q, K, V, cfg["k"], cfg["iters"], plan=plan))
    n_fwd = bench.count_kernels(lambda: m.vc_attn_forward(plan, O))
    assert n_fwd == 1
    assert n_prep + n_fwd == bench.launches_per_step(cfg)
    plan.destroy()
