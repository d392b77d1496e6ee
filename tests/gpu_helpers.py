"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI, run the CPU
oracle on the same inputs, and compare with the acceptance rule of the forward.

Acceptance (per batch-head, over the compared rows): relative L2 error <= 1e-2 and max-abs error
<= 3e-2 * max|V|, with the oracle fed the GPU's permutation. ExpCast codes, the argsort
permutation and (expected) every prepare output are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

REL_L2 = 1e-2
MAX_ABS_FRAC = 3e-2


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def vc():
    from bit_fp8_attention_gb300 import build

    build.build()
    import bit_fp8_attention_gb300 as mod

    return mod


def plan_host(m, plan, what) -> np.ndarray:
    t = m.vc_plan_get(plan, what)
    torch.cuda.synchronize()
    if t.dtype == torch.bfloat16:
        return u16(t)
    return t.cpu().numpy()


def gpu_plan_all(m, plan) -> dict:
    """Every prepare output of a plan copied to the host once."""
    return {"perm": plan_host(m, plan, m.VC_PLAN_PERM), "labels": plan_host(m, plan, m.VC_PLAN_LABELS),
            "qc": plan_host(m, plan, m.VC_PLAN_QCODES), "sq": plan_host(m, plan, m.VC_PLAN_QSCALES),
            "kc": plan_host(m, plan, m.VC_PLAN_KCODES), "sk": plan_host(m, plan, m.VC_PLAN_KSCALES),
            "vt": plan_host(m, plan, m.VC_PLAN_VCODES), "sv": plan_host(m, plan, m.VC_PLAN_VSCALES),
            "mub": plan_host(m, plan, m.VC_PLAN_MEANS)}


def head_of(a: dict, b: int, h: int) -> dict:
    """One batch-head of gpu_plan_all(), in the oracle's layouts (residual codes [S_pad, D])."""
    g = {key: a[key][b, h] for key in ("perm", "labels", "qc", "sq", "kc", "sk", "mub")}
    g["rc"] = np.ascontiguousarray(a["vt"][b, h].T)
    g["sv"] = float(a["sv"][b, h])
    return g


def gpu_plan_one_head(m, plan, b, h) -> dict:
    """The prepare outputs of one batch-head, sliced on the device before the copy (large plans)."""
    def get(what):
        t = m.vc_plan_get(plan, what)[b, h]
        torch.cuda.synchronize()
        return u16(t) if t.dtype == torch.bfloat16 else t.cpu().numpy()

    g = {key: get(what) for key, what in (("perm", m.VC_PLAN_PERM), ("labels", m.VC_PLAN_LABELS),
                                          ("qc", m.VC_PLAN_QCODES), ("sq", m.VC_PLAN_QSCALES),
                                          ("kc", m.VC_PLAN_KCODES), ("sk", m.VC_PLAN_KSCALES),
                                          ("mub", m.VC_PLAN_MEANS))}
    g["rc"] = np.ascontiguousarray(get(m.VC_PLAN_VCODES).T)
    g["sv"] = float(get(m.VC_PLAN_VSCALES))
    return g


def gpu_plan_head(m, plan, b, h) -> dict:
    """The GPU's prepare outputs for one batch-head (copies the whole plan: small plans only)."""
    return head_of(gpu_plan_all(m, plan), b, h)


def compare_prep(g: dict, o: dict, S: int):
    """Bit-exact comparison of the GPU and oracle prepare outputs of one head."""
    assert np.array_equal(g["qc"], o["qc"]), "Q codes differ"
    assert np.array_equal(g["sq"], o["sq"]), "Q scales differ"
    assert np.array_equal(g["kc"], o["kc"]), "K' codes differ"
    assert np.array_equal(g["sk"], o["sk"]), "K' scales differ"
    assert np.array_equal(g["mub"], o["mub"]), "block means differ"
    assert g["sv"] == np.float32(o["sv"]), "V scale differs"
    assert np.array_equal(g["rc"], o["rc"]), "residual codes differ"


def errors(gpu_rows: np.ndarray, ref_rows: np.ndarray) -> tuple[float, float]:
    d = gpu_rows - ref_rows
    return float(np.linalg.norm(d) / max(np.linalg.norm(ref_rows), 1e-300)), float(np.abs(d).max())


def assert_within(gpu_rows, ref_rows, vmax, what=""):
    rel, mx = errors(gpu_rows, ref_rows)
    assert rel <= REL_L2, f"{what} rel-L2 {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS_FRAC * vmax, f"{what} max-abs {mx:.3e} > {MAX_ABS_FRAC} * {vmax:.3e}"
    return rel, mx


def oracle_forward_from_plan(g: dict, S: int, rows, expcast=True, midwindow=True, with_mean=True):
    """Oracle (i) on the GPU's own plan tensors: isolates the forward kernel."""
    return oracle.attention_quant(g["qc"], g["sq"], g["kc"], g["sk"], g["rc"], g["sv"],
                                  g["mub"] if with_mean else None, S, rows,
                                  (oracle.EXPCAST if expcast else 0) | (oracle.MIDWINDOW if midwindow else 0))[0]
