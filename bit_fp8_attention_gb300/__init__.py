"""Python binding of the sm_103a ExpCast-FP8 + V-Smooth attention library (include/vc_attn.h).

Argument marshalling only: every step of the computation runs in the library's CUDA kernels.
The functions carry the C ABI's names. PyTorch provides device memory and streams. There is no
CPU fallback: if the shared library is missing, calls raise instead of computing elsewhere.

    plan = vc_attn_prepare(Q, K, V, k_clusters, iters)      # k-means, pi, means, FP8 codes
    O = vc_attn_forward(plan)                               # fused FP8 attention -> bf16
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libvc_attn.so")

VC_OK = 0
VC_ERR_INVALID_ARG = -1
VC_ERR_UNSUPPORTED = -2
VC_ERR_CUDA = -3
VC_ERR_TIMEOUT = -4
VC_ERR_PLAN_MISMATCH = -5
VC_ERR_OOM = -6
VC_ERR_NO_DEVICE = -7

VC_EXPCAST = 1
VC_VSMOOTH = 2
VC_MIDWINDOW = 4
VC_KCENTER = 8
VC_WARM_START = 16
VC_REUSE_PERM = 32
VC_VSCALE_CHANNEL = 64
VC_QK_HADAMARD = 128
VC_DEBUG_TIMEOUT = 1 << 16
VC_FLAGS_DEFAULT = VC_EXPCAST | VC_VSMOOTH | VC_MIDWINDOW

VC_PLAN_LABELS = 1
VC_PLAN_PERM = 2
VC_PLAN_QCODES = 3
VC_PLAN_QSCALES = 4
VC_PLAN_KCODES = 5
VC_PLAN_KSCALES = 6
VC_PLAN_VCODES = 7
VC_PLAN_VSCALES = 8
VC_PLAN_MEANS = 9
VC_PLAN_CENTROIDS = 10
VC_PLAN_KCENTER = 11
VC_PLAN_VCHSCALES = 12
VC_PLAN_MEANS_T = 13
VC_PLAN_REPAIR_IDX = 14
VC_PLAN_REPAIR_ENERGY = 15
VC_PLAN_REPAIR_KCODES = 16
VC_PLAN_REPAIR_KSCALES = 17
VC_PLAN_REPAIR_VCODES = 18
VC_NOALLOC_MAX_HEADS = 4096
VC_STEP_GROUP, VC_STEP_GROUP_WARM, VC_STEP_REUSE, VC_STEP_PLAIN = 0, 1, 2, 3

EXPORTS = ("vc_attn_prepare", "vc_attn_prepare_ex", "vc_attn_prepare_repair", "vc_attn_forward", "vc_plan_size",
           "vc_plan_get", "vc_plan_status", "vc_plan_shape", "vc_plan_destroy", "vc_expcast_encode",
           "vc_expcast_encode_unclamped",
           "vc_schedule_action",
           "vc_strerror", "vc_version")


class VCError(RuntimeError):
    def __init__(self, rc: int, what: str):
        super().__init__(f"{what}: {vc_strerror(rc)} ({rc})")
        self.rc = rc


_lib = None


def lib() -> ctypes.CDLL:
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m bit_fp8_attention_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, u, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
    sigs = {
        "vc_attn_prepare": (i, [vp, vp, vp, i, i, i, i, i, i, vp, ctypes.POINTER(vp)]),
        "vc_attn_prepare_ex": (i, [vp, vp, vp, i, i, i, i, i, i, vp, u, vp, ctypes.POINTER(vp)]),
        "vc_attn_prepare_repair": (i, [vp, vp, vp, i, i, i, i, i, u, vp, ctypes.POINTER(vp)]),
        "vc_attn_forward": (i, [vp, vp, u, vp]),
        "vc_plan_size": (sz, [vp, i]),
        "vc_plan_get": (i, [vp, i, vp, sz, vp]),
        "vc_plan_status": (i, [vp, vp, ctypes.POINTER(i)]),
        "vc_plan_shape": (i, [vp] + [ctypes.POINTER(i)] * 5),
        "vc_plan_destroy": (None, [vp]),
        "vc_expcast_encode": (i, [vp, vp, vp, ctypes.c_int64, vp, vp]),
        "vc_expcast_encode_unclamped": (i, [vp, vp, vp, ctypes.c_int64, vp, vp]),
        "vc_residual_pack_noalloc": (i, [vp, vp, i, i, i, i, vp, vp, vp, vp]),
        "vc_schedule_action": (i, [i, i, i]),
        "vc_strerror": (ctypes.c_char_p, [i]),
        "vc_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(rc: int, what: str):
    if rc != VC_OK:
        raise VCError(rc, what)


def vc_schedule_action(step: int, n_steps: int, reuse: int = 4) -> int:
    """VC_STEP_* action of a denoising step (see include/vc_attn.h); raises on invalid arguments."""
    rc = lib().vc_schedule_action(step, n_steps, reuse)
    if rc < 0:
        raise VCError(rc, "vc_schedule_action")
    return rc


# Prepare flags of each schedule action (include/vc_attn.h, grouping schedule).
STEP_PREPARE_FLAGS = {VC_STEP_GROUP: VC_VSMOOTH, VC_STEP_GROUP_WARM: VC_VSMOOTH | VC_WARM_START,
                      VC_STEP_REUSE: VC_VSMOOTH | VC_REUSE_PERM, VC_STEP_PLAIN: VC_REUSE_PERM}


def vc_strerror(rc: int) -> str:
    return lib().vc_strerror(rc).decode()


def vc_version() -> str:
    return lib().vc_version().decode()


class Plan:
    """Owns a vc_plan* (device buffers of the prepare step); freed by destroy() or on collection."""

    def __init__(self, handle: ctypes.c_void_p):
        self.handle = handle
        dims = [ctypes.c_int() for _ in range(5)]
        _check(lib().vc_plan_shape(handle, *[ctypes.byref(d) for d in dims]), "vc_plan_shape")
        self.B, self.H, self.S, self.D, self.k = (d.value for d in dims)
        self.nkb = (self.S + 127) // 128
        self.S_pad = self.nkb * 128
        # repair rows per head (a plan from vc_attn_prepare_repair); 0 otherwise
        self.n_repair = lib().vc_plan_size(handle, VC_PLAN_REPAIR_IDX) // (4 * self.B * self.H)
        self.R_pad = (self.n_repair + 127) // 128 * 128

    def destroy(self):
        if self.handle is not None and self.handle.value:
            lib().vc_plan_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def _qkv_args(Q, K, V):
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
                and t.dim() == 4):
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [B, H, S, D]")
    if not (Q.shape == K.shape == V.shape):
        raise ValueError("Q, K, V must have the same shape")
    return Q.shape


def vc_attn_prepare_ex(Q, K, V, k_clusters: int, iters: int, perm=None, flags: int = VC_VSMOOTH, stream=None,
                       plan: Plan | None = None) -> Plan:
    B, H, S, D = _qkv_args(Q, K, V)
    pp = None
    if perm is not None:
        if not (perm.is_cuda and perm.dtype == torch.int32 and perm.is_contiguous() and perm.numel() == B * H * S):
            raise ValueError("perm must be a contiguous CUDA int32 tensor [B, H, S]")
        pp = perm.data_ptr()
    h = ctypes.c_void_p(plan.handle.value if plan is not None else None)
    rc = lib().vc_attn_prepare_ex(Q.data_ptr(), K.data_ptr(), V.data_ptr(), B, H, S, D, k_clusters, iters, pp,
                                  flags, _stream(stream), ctypes.byref(h))
    _check(rc, "vc_attn_prepare_ex")
    return plan if plan is not None else Plan(h)


def repair_rows_for(S: int, rho: float = 0.005) -> int:
    """The repair budget as a row count: ceil(rho * S) (the pages' operating point rho = 0.5%)."""
    return min(S, math.ceil(rho * S))


def vc_attn_prepare_repair(Q, K, V, n_repair: int, flags: int = 0, stream=None, plan: Plan | None = None) -> Plan:
    B, H, S, D = _qkv_args(Q, K, V)
    h = ctypes.c_void_p(plan.handle.value if plan is not None else None)
    rc = lib().vc_attn_prepare_repair(Q.data_ptr(), K.data_ptr(), V.data_ptr(), B, H, S, D, n_repair, flags,
                                      _stream(stream), ctypes.byref(h))
    _check(rc, "vc_attn_prepare_repair")
    return plan if plan is not None else Plan(h)


def vc_attn_prepare(Q, K, V, k_clusters: int, iters: int, stream=None, plan: Plan | None = None) -> Plan:
    B, H, S, D = _qkv_args(Q, K, V)
    h = ctypes.c_void_p(plan.handle.value if plan is not None else None)
    rc = lib().vc_attn_prepare(Q.data_ptr(), K.data_ptr(), V.data_ptr(), B, H, S, D, k_clusters, iters,
                               _stream(stream), ctypes.byref(h))
    _check(rc, "vc_attn_prepare")
    return plan if plan is not None else Plan(h)


def vc_attn_forward(plan: Plan, O=None, flags: int = VC_FLAGS_DEFAULT, stream=None):
    if O is None:
        O = torch.empty((plan.B, plan.H, plan.S, plan.D), dtype=torch.bfloat16, device="cuda")
    if not (O.is_cuda and O.dtype == torch.bfloat16 and O.is_contiguous()
            and tuple(O.shape) == (plan.B, plan.H, plan.S, plan.D)):
        raise ValueError("O must be a contiguous CUDA bf16 tensor [B, H, S, D]")
    _check(lib().vc_attn_forward(plan.handle, O.data_ptr(), flags, _stream(stream)), "vc_attn_forward")
    return O


_PLAN_DTYPES = {
    VC_PLAN_LABELS: (torch.int32, lambda p: (p.B, p.H, p.S)),
    VC_PLAN_PERM: (torch.int32, lambda p: (p.B, p.H, p.S)),
    VC_PLAN_QCODES: (torch.uint8, lambda p: (p.B, p.H, p.S_pad, p.D)),
    VC_PLAN_QSCALES: (torch.float32, lambda p: (p.B, p.H, p.nkb)),
    VC_PLAN_KCODES: (torch.uint8, lambda p: (p.B, p.H, p.S_pad, p.D)),
    VC_PLAN_KSCALES: (torch.float32, lambda p: (p.B, p.H, p.nkb)),
    VC_PLAN_VCODES: (torch.uint8, lambda p: (p.B, p.H, p.D, p.S_pad)),
    VC_PLAN_VSCALES: (torch.float32, lambda p: (p.B, p.H)),
    VC_PLAN_MEANS: (torch.bfloat16, lambda p: (p.B, p.H, p.nkb, p.D)),
    VC_PLAN_CENTROIDS: (torch.float32, lambda p: (p.B, p.H, p.k, p.D)),
    VC_PLAN_KCENTER: (torch.bfloat16, lambda p: (p.B, p.H, p.D)),
    VC_PLAN_VCHSCALES: (torch.float32, lambda p: (p.B, p.H, p.D)),
    VC_PLAN_MEANS_T: (torch.bfloat16, lambda p: (p.B, p.H, p.D, (p.nkb + 15) // 16 * 16)),
    VC_PLAN_REPAIR_IDX: (torch.int32, lambda p: (p.B, p.H, p.n_repair)),
    VC_PLAN_REPAIR_ENERGY: (torch.float32, lambda p: (p.B, p.H, p.S)),
    VC_PLAN_REPAIR_KCODES: (torch.uint8, lambda p: (p.B, p.H, p.R_pad, p.D)),
    VC_PLAN_REPAIR_KSCALES: (torch.float32, lambda p: (p.B, p.H, p.R_pad // 128)),
    VC_PLAN_REPAIR_VCODES: (torch.uint8, lambda p: (p.B, p.H, p.D, p.R_pad)),
}


def vc_plan_size(plan: Plan, what: int) -> int:
    return int(lib().vc_plan_size(plan.handle, what))


def vc_plan_get(plan: Plan, what: int, out=None, stream=None):
    """Copy one plan tensor into `out` (a new CUDA tensor by default) on `stream`."""
    dt, shape = _PLAN_DTYPES[what]
    if out is None:
        out = torch.empty(shape(plan), dtype=dt, device="cuda")
    nbytes = out.numel() * out.element_size()
    _check(lib().vc_plan_get(plan.handle, what, out.data_ptr(), nbytes, _stream(stream)), "vc_plan_get")
    return out


def vc_plan_status(plan: Plan, stream=None) -> tuple[int, int]:
    """(status code, error bits) of the plan's kernels since the last call; synchronises the stream."""
    bits = ctypes.c_int(0)
    rc = lib().vc_plan_status(plan.handle, _stream(stream), ctypes.byref(bits))
    return rc, bits.value


def vc_plan_shape(plan: Plan) -> tuple[int, int, int, int, int]:
    """(B, H, S, D, k_clusters) of a plan."""
    return plan.B, plan.H, plan.S, plan.D, plan.k


def vc_plan_destroy(plan: Plan):
    plan.destroy()


def vc_residual_pack_noalloc(V, perm, means, vcodes, vscales, stream=None):
    """Value-side preparation into caller-provided tensors, with no device allocation.

    For callers that must not allocate device memory: the library's only scratch is a fixed
    in-library array of VC_NOALLOC_MAX_HEADS words per GPU. V: bf16 [B, H, S, D]; perm: int32
    [B, H, S] or None (identity); means: bf16 [B, H, nkb, D]; vcodes: uint8 [B, H, D, S_pad];
    vscales: fp32 [B, H] -- the layouts of VC_PLAN_MEANS / VC_PLAN_VCODES / VC_PLAN_VSCALES.
    Calls that overlap on the GPU share that scratch and must be serialised by the caller.
    """
    if not (V.is_cuda and V.dtype == torch.bfloat16 and V.is_contiguous() and V.dim() == 4):
        raise ValueError("V must be a contiguous CUDA bf16 tensor [B, H, S, D]")
    B, H, S, D = V.shape
    nkb = (S + 127) // 128
    for t, dt, shape in ((means, torch.bfloat16, (B, H, nkb, D)), (vcodes, torch.uint8, (B, H, D, nkb * 128)),
                         (vscales, torch.float32, (B, H))):
        if not (t.is_cuda and t.dtype == dt and t.is_contiguous() and tuple(t.shape) == shape):
            raise ValueError(f"output must be a contiguous CUDA {dt} tensor {shape}")
    pp = None
    if perm is not None:
        if not (perm.is_cuda and perm.dtype == torch.int32 and perm.is_contiguous() and perm.numel() == B * H * S):
            raise ValueError("perm must be a contiguous CUDA int32 tensor [B, H, S]")
        pp = perm.data_ptr()
    _check(lib().vc_residual_pack_noalloc(V.data_ptr(), pp, B, H, S, D, means.data_ptr(), vcodes.data_ptr(),
                                          vscales.data_ptr(), _stream(stream)), "vc_residual_pack_noalloc")


def vc_expcast_encode(s, a, b, stream=None, clamp: bool = True):
    """ExpCast-FP8 codes clip[0,120](rne(fmaf(s, a, b))) through the forward kernel's code path.

    clamp=False: vc_expcast_encode_unclamped, the bytes of the forward's fast path (no clamp at 120)."""
    for t in (s, a, b):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and t.numel() == s.numel()):
            raise ValueError("s, a, b must be contiguous CUDA float32 tensors of equal size")
    out = torch.empty(s.shape, dtype=torch.uint8, device=s.device)
    fn = lib().vc_expcast_encode if clamp else lib().vc_expcast_encode_unclamped
    _check(fn(s.data_ptr(), a.data_ptr(), b.data_ptr(), s.numel(), out.data_ptr(), _stream(stream)),
           "vc_expcast_encode" if clamp else "vc_expcast_encode_unclamped")
    return out


def vc_expcast_encode_unclamped(s, a, b, stream=None):
    """The forward's fast-path bytes: the code path of vc_expcast_encode without the clamp at 120."""
    return vc_expcast_encode(s, a, b, stream=stream, clamp=False)
