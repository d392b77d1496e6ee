"""CPU oracle for the ExpCast-FP8 + V-Smooth FP8 attention forward.

TEST INFRASTRUCTURE. This package is the plain, slow reference the CUDA path is checked against.
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it;
the product package never does. It shares no code with the CUDA library: the arithmetic lives in
``vc_oracle.c`` (plain C, fp64 where the pages fix no precision), built with gcc by ``build()``.

Every function cites the passage it follows (page title and section/equation):
  [VC]  "VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention"
  [OVC] "Open-VC Attention: an open-source, error-tunable variant of VC-Attention" (MachGen blog)

Parity pins for every function live in ``tests/test_oracle_*.py``. Nothing here is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vc_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libvc_oracle.so")
_lock = threading.Lock()
_lib = None

BLOCK = 128
EXPCAST = 1
MIDWINDOW = 2
HADAMARD = 4  # Q and K were rotated (reading R19)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc. -ffp-contract=off keeps every fp32 step unfused on any host."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(t):
    return ctypes.POINTER(t)


def lib():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        L = ctypes.CDLL(build())
        u8, u16, i32, i64, f32, f64 = (_p(ctypes.c_uint8), _p(ctypes.c_uint16), _p(ctypes.c_int32),
                                       _p(ctypes.c_int64), _p(ctypes.c_float), _p(ctypes.c_double))
        sig = {
            "orc_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "orc_e4m3_decode_n": (None, [u8, ctypes.c_int64, f64]),
            "orc_e4m3_encode_n": (None, [f32, ctypes.c_int64, u8]),
            "orc_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
            "orc_f64_to_bf16_n": (None, [f64, ctypes.c_int64, u16]),
            "orc_expcast_code": (ctypes.c_int, [ctypes.c_float, ctypes.c_float, ctypes.c_float]),
            "orc_expcast_unclipped": (ctypes.c_int, [ctypes.c_float, ctypes.c_float, ctypes.c_float]),
            "orc_expcast_codes": (None, [f32, f32, f32, ctypes.c_int64, u8]),
            "orc_exp_then_cast": (ctypes.c_uint8, [ctypes.c_double]),
            "orc_expcast_of_u": (ctypes.c_int, [ctypes.c_double]),
            "orc_quant_blocks": (None, [u16, ctypes.c_int64, ctypes.c_int, u8, f32]),
            "orc_quant_blocks_centered": (None, [u16, ctypes.c_int64, ctypes.c_int, u16, u8, f32]),
            "orc_quant_blocks_rot": (None, [u16, ctypes.c_int64, ctypes.c_int, u16, ctypes.c_int, u8, f32]),
            "orc_fwht_f32": (None, [f32, ctypes.c_int]),
            "orc_code_scale_rot": (ctypes.c_float, [ctypes.c_int]),
            "orc_kmeans_from": (None, [u16, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32, f64, f64]),
            "orc_schedule_action": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
            "orc_channel_mean_bf16": (None, [u16, ctypes.c_int64, ctypes.c_int, u16]),
            "orc_kmeans_objective": (ctypes.c_double, [u16, ctypes.c_int64, ctypes.c_int, ctypes.c_int, i32]),
            "orc_kmeans": (None, [u16, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32, f64, f64]),
            "orc_stable_argsort": (None, [i32, ctypes.c_int64, ctypes.c_int, i32]),
            "orc_demean": (None, [u16, i32, ctypes.c_int64, ctypes.c_int, ctypes.c_int, f64, u16, f32, u8, f32, f32]),
            "orc_demean_ex": (None, [u16, i32, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, f64, u16, u16,
                                     f32, u8, f32, f32]),
            "orc_gather_rows": (None, [u16, i32, ctypes.c_int64, ctypes.c_int, u16]),
            "orc_visit_order": (None, [ctypes.c_int, ctypes.c_int, ctypes.c_int, i32]),
            "orc_code_scale": (ctypes.c_float, [ctypes.c_int]),
            "orc_attention_quant": (None, [u8, f32, u8, f32, u8, ctypes.c_float, u16, ctypes.c_int64, ctypes.c_int,
                                           ctypes.c_int, i64, ctypes.c_int64, f64, f64, f32]),
            "orc_attention_quant_ex": (None, [u8, f32, u8, f32, u8, ctypes.c_float, f32, u16, u16, ctypes.c_int64,
                                              ctypes.c_int, ctypes.c_int, i64, ctypes.c_int64, f64, f64, f32]),
            "orc_repair_select": (None, [u16, ctypes.c_int64, ctypes.c_int, f32, ctypes.c_int64, i32, f32, u8]),
            "orc_attention_quant_rep": (None, [u8, f32, u8, f32, u8, ctypes.c_float, f32, u16, u16, u8, f32, u8,
                                               ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int, i64,
                                               ctypes.c_int64, f64, f64, f32]),
            "orc_attention_exact": (None, [u16, u16, u16, ctypes.c_int64, ctypes.c_int, i64, ctypes.c_int64, f64]),
            "orc_attention_demeaned_exact": (None, [f64, f64, f64, ctypes.c_int64, ctypes.c_int, ctypes.c_int, i64,
                                                    ctypes.c_int64, f64]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def _ptr(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(t))


def _u16(x) -> np.ndarray:
    """bf16 tensor or uint16/int16 array -> C-contiguous uint16 bit pattern array."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            assert x.dtype == torch.bfloat16
            return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if x.dtype == np.int16:
        x = x.view(np.uint16)
    assert x.dtype == np.uint16
    return np.ascontiguousarray(x)


def nkb_of(S: int) -> int:
    return (S + BLOCK - 1) // BLOCK


# ----------------------------------------------------------------------------------------------
# E4M3 codec  ([VC] §3.3: v = 2^(e-7)(1+m/8); OCP subnormals/NaN/saturation by reading)
# ----------------------------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    lib().orc_e4m3_decode_n(_ptr(c, ctypes.c_uint8), c.size, _ptr(out, ctypes.c_double))
    return out


def e4m3_encode(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(a.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_n(_ptr(a, ctypes.c_float), a.size, _ptr(out, ctypes.c_uint8))
    return out


def f64_to_bf16(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(a.shape, dtype=np.uint16)
    lib().orc_f64_to_bf16_n(_ptr(a, ctypes.c_double), a.size, _ptr(out, ctypes.c_uint16))
    return out


def bf16_to_f64(u16) -> np.ndarray:
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------------------------
# ExpCast-FP8  ([VC] §3.3 Eq. 7; [OVC] "Scheduling around ExpCast": one FMA per score)
# ----------------------------------------------------------------------------------------------
def expcast_codes(s, a, b) -> np.ndarray:
    s = np.ascontiguousarray(np.asarray(s, dtype=np.float32))
    a = np.ascontiguousarray(np.broadcast_to(np.asarray(a, dtype=np.float32), s.shape))
    b = np.ascontiguousarray(np.broadcast_to(np.asarray(b, dtype=np.float32), s.shape))
    out = np.empty(s.shape, dtype=np.uint8)
    lib().orc_expcast_codes(_ptr(s, ctypes.c_float), _ptr(a, ctypes.c_float), _ptr(b, ctypes.c_float), s.size,
                            _ptr(out, ctypes.c_uint8))
    return out


def expcast_code(s: float, a: float, b: float) -> int:
    return int(lib().orc_expcast_code(s, a, b))


def expcast_unclipped(s: float, a: float, b: float) -> int:
    return int(lib().orc_expcast_unclipped(s, a, b))


def expcast_of_u(u: float) -> int:
    """Eq. 7 as a function of the log2-domain score u alone."""
    return int(lib().orc_expcast_of_u(u))


def exp_then_cast(u: float) -> int:
    """The conventional path ExpCast replaces: 2^(u+8) cast to E4M3 ([VC] §3.3, Fig. 5a)."""
    return int(lib().orc_exp_then_cast(u))


def code_scale(D: int) -> float:
    """fp32(8 log2(e) / sqrt(D)): log2 e, the factor 8 and the softmax scale folded together."""
    return float(lib().orc_code_scale(D))


# ----------------------------------------------------------------------------------------------
# Preparation steps
# ----------------------------------------------------------------------------------------------
def quant_blocks(x, center=None, rotate: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Per-128-token block E4M3 quantisation ([OVC] "Scheduling around ExpCast").

    x: [S, D] bf16. center: None, or [D] bf16 subtracted (fp32) from every row first. rotate: apply
    the fp32 Walsh-Hadamard butterfly to every row first (reading R19, see fwht).
    Returns codes [S_pad, D] uint8 and scales [nkb] float32.
    """
    x = _u16(x)
    S, D = x.shape
    nkb = nkb_of(S)
    codes = np.empty((nkb * BLOCK, D), dtype=np.uint8)
    scales = np.empty(nkb, dtype=np.float32)
    c = None if center is None else np.ascontiguousarray(_u16(center).reshape(D))
    lib().orc_quant_blocks_rot(_ptr(x, ctypes.c_uint16), S, D, None if c is None else _ptr(c, ctypes.c_uint16),
                               1 if rotate else 0, _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_float))
    return codes, scales


def fwht(x) -> np.ndarray:
    """The unnormalised Walsh-Hadamard transform of each row of x, as the fp32 butterfly of reading R19."""
    a = np.array(x, dtype=np.float32, order="C", copy=True)  # never the caller's array
    rows = a.reshape(-1, a.shape[-1])
    for r in rows:
        lib().orc_fwht_f32(_ptr(r, ctypes.c_float), r.size)
    return a


def channel_mean_bf16(x) -> np.ndarray:
    """K channel centering statistic ([VC] §3.4 "Fused preprocessing", App. B): bf16 of the fp64 mean
    of every channel over the head's tokens. x: [S, D] bf16. Returns [D] bf16 bits (uint16)."""
    x = _u16(x)
    S, D = x.shape
    mu = np.empty(D, dtype=np.uint16)
    lib().orc_channel_mean_bf16(_ptr(x, ctypes.c_uint16), S, D, _ptr(mu, ctypes.c_uint16))
    return mu


def kmeans(v, k: int, iters: int, init=None):
    """Lloyd k-means over value tokens ([VC] §3.2 "Value-guided permutation", "Unbalanced clusters").

    init: None (centroid i starts as row floor(i*S/k)), or [k, D] starting centroids (warm start from a
    previous grouping, "Unbalanced clusters cost little").
    Returns labels [S] int32, centroids [k, D] float64, objective of each round [iters].
    """
    v = _u16(v)
    S, D = v.shape
    labels = np.empty(S, dtype=np.int32)
    J = np.empty(max(iters, 1), dtype=np.float64)
    if init is None:
        cent = np.empty((k, D), dtype=np.float64)
        lib().orc_kmeans(_ptr(v, ctypes.c_uint16), S, D, k, iters, _ptr(labels, ctypes.c_int32),
                         _ptr(cent, ctypes.c_double), _ptr(J, ctypes.c_double))
    else:
        cent = np.array(init, dtype=np.float64, copy=True).reshape(k, D)
        lib().orc_kmeans_from(_ptr(v, ctypes.c_uint16), S, D, k, iters, _ptr(labels, ctypes.c_int32),
                              _ptr(cent, ctypes.c_double), _ptr(J, ctypes.c_double))
    return labels, cent, J[:iters]


GROUP, GROUP_WARM, REUSE, PLAIN = 0, 1, 2, 3


def schedule_action(step: int, n_steps: int, reuse: int = 4) -> int:
    """Grouping schedule ([VC] §3.4 "Amortized grouping schedule", App. A "Grouping schedule"):
    GROUP / GROUP_WARM / REUSE / PLAIN for one denoising step."""
    return int(lib().orc_schedule_action(step, n_steps, reuse))


def kmeans_objective(v, k: int, labels) -> float:
    """J(z) = sum_t ||x_t - mean_{z_t}||^2 in fp64, from the labels alone."""
    v = _u16(v)
    S, D = v.shape
    z = np.ascontiguousarray(np.asarray(labels, dtype=np.int32))
    return float(lib().orc_kmeans_objective(_ptr(v, ctypes.c_uint16), S, D, k, _ptr(z, ctypes.c_int32)))


def stable_argsort(z, k: int) -> np.ndarray:
    """pi = argsort(z), ties in token order ([VC] §3.2 Eq. 3)."""
    z = np.ascontiguousarray(np.asarray(z, dtype=np.int32))
    perm = np.empty(z.size, dtype=np.int32)
    lib().orc_stable_argsort(_ptr(z, ctypes.c_int32), z.size, k, _ptr(perm, ctypes.c_int32))
    return perm


def gather_rows(x, perm) -> np.ndarray:
    x = _u16(x)
    S, D = x.shape
    p = np.ascontiguousarray(np.asarray(perm, dtype=np.int32))
    out = np.empty_like(x)
    lib().orc_gather_rows(_ptr(x, ctypes.c_uint16), _ptr(p, ctypes.c_int32), S, D, _ptr(out, ctypes.c_uint16))
    return out


def demean(v, perm=None, subtract_mean: bool = True, per_channel: bool = False) -> dict:
    """Gather by pi, 128-row block means, residual and its E4M3 quantisation.

    [VC] §3.2 "Block demeaning" Eq. 4. per_channel=False: one V scale per head ([OVC]); "amax" and
    "sv" are floats. per_channel=True: one scale per channel ([VC] §3.2, App. B); "amax" and "sv" are
    [D] float32 arrays and "mut" holds the means divided by the channel scales (bf16 bits).
    """
    v = _u16(v)
    S, D = v.shape
    nkb = nkb_of(S)
    p = None if perm is None else np.ascontiguousarray(np.asarray(perm, dtype=np.int32))
    mu = np.empty((nkb, D), dtype=np.float64)
    mub = np.empty((nkb, D), dtype=np.uint16)
    mut = np.zeros((nkb, D), dtype=np.uint16)
    resid = np.empty((nkb * BLOCK, D), dtype=np.float32)
    rc = np.empty((nkb * BLOCK, D), dtype=np.uint8)
    amax = np.zeros(D, dtype=np.float32)
    sv = np.zeros(D, dtype=np.float32)
    lib().orc_demean_ex(_ptr(v, ctypes.c_uint16), None if p is None else _ptr(p, ctypes.c_int32), S, D,
                        1 if subtract_mean else 0, 1 if per_channel else 0, _ptr(mu, ctypes.c_double),
                        _ptr(mub, ctypes.c_uint16), _ptr(mut, ctypes.c_uint16), _ptr(resid, ctypes.c_float),
                        _ptr(rc, ctypes.c_uint8), _ptr(amax, ctypes.c_float), _ptr(sv, ctypes.c_float))
    out = {"mu": mu, "mub": mub, "resid": resid, "rc": rc}
    if per_channel:
        out.update(amax=amax, sv=sv, mut=mut)
    else:
        out.update(amax=float(amax[0]), sv=float(sv[0]))
    return out


def visit_order(nkb: int, qt: int, midwindow: bool = True) -> np.ndarray:
    """Mid-window key traversal ([OVC] "Scheduling around ExpCast"); linear when midwindow is off."""
    out = np.empty(nkb, dtype=np.int32)
    lib().orc_visit_order(nkb, qt, 1 if midwindow else 0, _ptr(out, ctypes.c_int32))
    return out


# ----------------------------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------------------------
def attention_quant(qc, sq, kc, sk, rc, sv, mub, S: int, rows, flags: int = EXPCAST | MIDWINDOW, mut=None,
                    repair=None):
    """(i) The quantised forward for the given query rows of one batch-head.

    [VC] §3.1 Eq. 1, §3.2 Eq. 6, §3.3 Eq. 7; [OVC] true-score max, consistent denominator, order.
    sv is a float (one residual scale per head; mub the means) or a [D] array of per-channel scales,
    then with mut the means divided by them ([VC] App. B). repair: None or the dict repair_rows()
    returns ([OVC] V residual repair: numerator-only rows visited last).
    Returns (out [n, D] fp64 = sv*A/l, l [n], M [n] float32 final running max in code units).
    """
    qc = np.ascontiguousarray(qc, dtype=np.uint8)
    kc = np.ascontiguousarray(kc, dtype=np.uint8)
    rc = np.ascontiguousarray(rc, dtype=np.uint8)
    sq = np.ascontiguousarray(sq, dtype=np.float32)
    sk = np.ascontiguousarray(sk, dtype=np.float32)
    D = qc.shape[1]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.size
    out = np.empty((n, D), dtype=np.float64)
    l = np.empty(n, dtype=np.float64)
    m = np.empty(n, dtype=np.float32)
    svc = None
    if np.ndim(sv) > 0:
        svc = np.ascontiguousarray(sv, dtype=np.float32)
        assert svc.shape == (D,)
        sv = 1.0
    mub_keep = None if mub is None else np.ascontiguousarray(mub, dtype=np.uint16)
    mut_keep = None if mut is None else np.ascontiguousarray(mut, dtype=np.uint16)
    if svc is not None and mub_keep is not None:
        assert mut_keep is not None, "per-channel scales need the scaled means"
    n_rep = 0
    kr = sr = rr = None
    if repair is not None and repair["n"] > 0:
        n_rep = int(repair["n"])
        kr = np.ascontiguousarray(repair["kc"], dtype=np.uint8)
        sr = np.ascontiguousarray(repair["sk"], dtype=np.float32)
        rr = np.ascontiguousarray(repair["rc"], dtype=np.uint8)
        assert kr.shape == rr.shape == (nkb_of(n_rep) * BLOCK, D) and sr.shape == (nkb_of(n_rep),)
    lib().orc_attention_quant_rep(_ptr(qc, ctypes.c_uint8), _ptr(sq, ctypes.c_float), _ptr(kc, ctypes.c_uint8),
                                  _ptr(sk, ctypes.c_float), _ptr(rc, ctypes.c_uint8), float(sv),
                                  None if svc is None else _ptr(svc, ctypes.c_float),
                                  None if mub_keep is None else _ptr(mub_keep, ctypes.c_uint16),
                                  None if (svc is None or mut_keep is None) else _ptr(mut_keep, ctypes.c_uint16),
                                  None if kr is None else _ptr(kr, ctypes.c_uint8),
                                  None if sr is None else _ptr(sr, ctypes.c_float),
                                  None if rr is None else _ptr(rr, ctypes.c_uint8), n_rep,
                                  S, D, flags, _ptr(rows, ctypes.c_int64), n, _ptr(out, ctypes.c_double),
                                  _ptr(l, ctypes.c_double), _ptr(m, ctypes.c_float))
    return out, l, m


def repair_select(v, amax, n_rep: int):
    """[OVC] "Why V residual repair": the n_rep tokens of largest residual energy (reading R18).

    v: [S, D] bf16 (no V-Smooth: R = V); amax: [D] float32 residual max per channel (all equal for
    one scale per head). Returns (idx [n_rep] int32 ascending, energy [S] float32, rep [R_pad, D]
    uint8 E4M3 codes of the kept tokens' rounding residuals in the main codes' units).
    """
    v = _u16(v)
    S, D = v.shape
    n_rep = int(n_rep)
    assert 0 <= n_rep <= S
    a = np.ascontiguousarray(np.broadcast_to(np.asarray(amax, dtype=np.float32), (D,)))
    idx = np.zeros(max(n_rep, 1), dtype=np.int32)
    energy = np.empty(max(S, 1), dtype=np.float32)
    rep = np.zeros((max(nkb_of(n_rep), 1) * BLOCK, D), dtype=np.uint8)
    lib().orc_repair_select(_ptr(v, ctypes.c_uint16), S, D, _ptr(a, ctypes.c_float), n_rep,
                            _ptr(idx, ctypes.c_int32), _ptr(energy, ctypes.c_float), _ptr(rep, ctypes.c_uint8))
    return idx[:n_rep], energy[:S], rep[:nkb_of(n_rep) * BLOCK]


def repair_rows(k, v, amax, n_rep: int, kcenter=None, rotate: bool = False) -> dict:
    """The repair rows of one head: the selected tokens, their keys copied and quantised as extra
    128-row blocks (minus the K centre when given, rotated like every key when asked), and their
    residual codes."""
    idx, energy, rep = repair_select(v, amax, n_rep)
    out = {"n": int(n_rep), "idx": idx, "energy": energy, "rc": rep}
    if n_rep > 0:
        out["kc"], out["sk"] = quant_blocks(_u16(k)[idx], center=kcenter, rotate=rotate)
    else:
        out["kc"], out["sk"] = np.zeros((0, _u16(k).shape[1]), dtype=np.uint8), np.zeros(0, dtype=np.float32)
    return out


def attention_exact(q, k, v, rows) -> np.ndarray:
    """(ii) Exact fp64 softmax attention on the bf16 inputs in token order ([VC] §3.1)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    S, D = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.size, D), dtype=np.float64)
    lib().orc_attention_exact(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16), S, D,
                              _ptr(rows, ctypes.c_int64), rows.size, _ptr(out, ctypes.c_double))
    return out


def attention_demeaned_exact(q, k, v, rows, midwindow: bool = True) -> np.ndarray:
    """Tiled recurrence with demeaned fp64 values and exact exp ([VC] §3.2 "Online mean restoration")."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    S, D = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.size, D), dtype=np.float64)
    lib().orc_attention_demeaned_exact(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                       _ptr(v, ctypes.c_double), S, D, MIDWINDOW if midwindow else 0,
                                       _ptr(rows, ctypes.c_int64), rows.size, _ptr(out, ctypes.c_double))
    return out


# ----------------------------------------------------------------------------------------------
# Whole-path conveniences for one batch-head
# ----------------------------------------------------------------------------------------------
def prepare_head(q, k, v, k_clusters: int, iters: int, vsmooth: bool = True, perm=None,
                 kcenter: bool = False, vscale_channel: bool = False, n_repair: int = 0,
                 hadamard: bool = False) -> dict:
    """Everything the prepare step produces for one batch-head, computed on the CPU.

    vsmooth=False: identity permutation, no means (R = V). perm given: use it instead of k-means
    (the parity tests feed the GPU's permutation here, as the acceptance rule says).
    kcenter: subtract the keys' channel mean before their quantisation (see channel_mean_bf16).
    vscale_channel: one residual scale per channel instead of one per head (see demean).
    n_repair: V residual repair rows (without V-Smooth only; see repair_rows).
    hadamard: rotate Q and K rows before their quantisation (reading R19, see fwht).
    """
    assert n_repair == 0 or not vsmooth, "V residual repair is defined without V-Smooth"
    q, k, v = _u16(q), _u16(k), _u16(v)
    S, D = q.shape
    out = {"S": S, "D": D}
    labels = None
    if vsmooth and perm is None:
        labels, cent, J = kmeans(v, k_clusters, iters)
        perm = stable_argsort(labels, k_clusters)
        out.update(labels=labels, centroids=cent, J_rounds=J)
    if perm is None:
        perm = np.arange(S, dtype=np.int32)
    perm = np.asarray(perm, dtype=np.int32)
    out["perm"] = perm
    out["qc"], out["sq"] = quant_blocks(q, rotate=hadamard)
    kp = gather_rows(k, perm)
    kmu = channel_mean_bf16(k) if kcenter else None
    out["kmu"] = kmu
    out["kc"], out["sk"] = quant_blocks(kp, center=kmu, rotate=hadamard)
    dm = demean(v, perm, subtract_mean=vsmooth, per_channel=vscale_channel)
    out.update(rc=dm["rc"], sv=dm["sv"], amax=dm["amax"], mub=dm["mub"], mu=dm["mu"], resid=dm["resid"],
               mut=dm.get("mut"))
    out["vsmooth"] = vsmooth
    out["vscale_channel"] = vscale_channel
    out["hadamard"] = hadamard
    out["repair"] = None
    if n_repair > 0:
        amax = dm["amax"] if vscale_channel else np.full(D, dm["amax"], dtype=np.float32)
        out["repair"] = repair_rows(k, v, amax, n_repair, kcenter=kmu, rotate=hadamard)
    return out


def forward_head(prep: dict, rows, expcast: bool = True, midwindow: bool = True):
    flags = (EXPCAST if expcast else 0) | (MIDWINDOW if midwindow else 0) | (HADAMARD if prep.get("hadamard") else 0)
    mub = prep["mub"] if prep["vsmooth"] else None
    return attention_quant(prep["qc"], prep["sq"], prep["kc"], prep["sk"], prep["rc"], prep["sv"], mub,
                           prep["S"], rows, flags, mut=prep.get("mut") if prep["vsmooth"] else None,
                           repair=prep.get("repair"))


def num_threads() -> int:
    """Threads the OpenMP loops use (OMP_NUM_THREADS or the host's cores)."""
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else (os.cpu_count() or 1)
