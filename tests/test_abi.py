"""The C-ABI library loads, exports every function include/vc_attn.h declares, and rejects bad
arguments before touching a device (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from bit_fp8_attention_gb300 import build

    build.build()
    import bit_fp8_attention_gb300 as vc

    return vc.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "vc_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:[\w\s\*]+?)\b(vc_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("vc_attn_prepare", "vc_attn_forward", "vc_attn_prepare_ex", "vc_plan_get", "vc_plan_destroy",
                 "vc_expcast_encode", "vc_strerror"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_python_binding_names_match_abi():
    import bit_fp8_attention_gb300 as vc

    for name in declared_functions():
        assert hasattr(vc, name), name


def test_python_constants_match_header():
    """Every flag, plan-tensor id, error code and step action the header defines has the same value
    in the binding."""
    import bit_fp8_attention_gb300 as vc

    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "vc_attn.h")).read(), flags=re.S)
    consts = re.findall(r"\b(VC_[A-Z0-9_]+)\s*=\s*(-?\d+)u?(?:\s*<<\s*(\d+))?", text)
    assert len(consts) >= 30
    for name, val, sh in consts:
        want = int(val) << int(sh) if sh else int(val)
        assert getattr(vc, name) == want, name


def test_strerror_and_version(L):
    import bit_fp8_attention_gb300 as vc

    assert vc.vc_strerror(0) == "ok"
    assert "timed out" in vc.vc_strerror(vc.VC_ERR_TIMEOUT)
    assert "sm_103a" in vc.vc_version()


def test_invalid_arguments_rejected_without_device(L):
    vp = ctypes.c_void_p
    plan = vp(None)
    fake = vp(4096)  # never dereferenced: validation fails first
    # null pointers
    assert L.vc_attn_prepare(None, fake, fake, 1, 1, 128, 128, 1, 1, None, ctypes.byref(plan)) == -1
    assert L.vc_attn_prepare(fake, fake, fake, 1, 1, 128, 128, 1, 1, None, None) == -1
    # misaligned
    assert L.vc_attn_prepare(vp(4097), fake, fake, 1, 1, 128, 128, 1, 1, None, ctypes.byref(plan)) == -1
    # unsupported head dim, k > S, S too large
    assert L.vc_attn_prepare(fake, fake, fake, 1, 1, 128, 96, 1, 1, None, ctypes.byref(plan)) == -2
    assert L.vc_attn_prepare(fake, fake, fake, 1, 1, 16, 128, 17, 1, None, ctypes.byref(plan)) == -2
    assert L.vc_attn_prepare(fake, fake, fake, 1, 1, (1 << 20) + 1, 128, 1, 1, None, ctypes.byref(plan)) == -2
    # non-positive sizes, grouping without iterations
    assert L.vc_attn_prepare(fake, fake, fake, 0, 1, 128, 128, 1, 1, None, ctypes.byref(plan)) == -1
    assert L.vc_attn_prepare(fake, fake, fake, 1, 1, 128, 128, 1, 0, None, ctypes.byref(plan)) == -1
    # a warm start or a permutation reuse needs a plan that has been grouped / prepared before
    assert L.vc_attn_prepare_ex(fake, fake, fake, 1, 1, 128, 128, 1, 2, None, 2 | 16, None, ctypes.byref(plan)) == -1
    assert L.vc_attn_prepare_ex(fake, fake, fake, 1, 1, 128, 128, 1, 2, None, 2 | 32, None, ctypes.byref(plan)) == -1
    assert L.vc_attn_prepare_ex(fake, fake, fake, 1, 1, 128, 128, 1, 2, fake, 2 | 32, None, ctypes.byref(plan)) == -1
    # repair rows: count within [0, S], never with V-Smooth or a reused permutation
    assert L.vc_attn_prepare_repair(fake, fake, fake, 1, 1, 128, 128, -1, 0, None, ctypes.byref(plan)) == -1
    assert L.vc_attn_prepare_repair(fake, fake, fake, 1, 1, 128, 128, 129, 0, None, ctypes.byref(plan)) == -1
    assert L.vc_attn_prepare_repair(fake, fake, fake, 1, 1, 128, 128, 4, 2, None, ctypes.byref(plan)) == -1
    assert L.vc_attn_prepare_repair(fake, fake, fake, 1, 1, 128, 128, 4, 32, None, ctypes.byref(plan)) == -1
    assert L.vc_attn_prepare_repair(None, fake, fake, 1, 1, 128, 128, 4, 0, None, ctypes.byref(plan)) == -1
    assert plan.value is None
    # forward / plan calls on a null plan
    assert L.vc_attn_forward(None, fake, 7, None) == -1
    assert L.vc_plan_size(None, 1) == 0
    assert L.vc_plan_get(None, 1, fake, 1 << 20, None) == -1
    assert L.vc_plan_shape(None, None, None, None, None, None) == -1
    L.vc_plan_destroy(None)
    assert L.vc_expcast_encode(None, None, None, 5, None, None) == -1
    assert L.vc_expcast_encode(None, None, None, -1, None, None) == -1
    assert L.vc_expcast_encode_unclamped(None, None, None, 5, None, None) == -1
    assert L.vc_expcast_encode_unclamped(None, None, None, -1, None, None) == -1


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """No fallback: without the built library every call raises instead of computing anything."""
    import bit_fp8_attention_gb300 as vc

    monkeypatch.setattr(vc, "_lib", None)
    monkeypatch.setattr(vc, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(ImportError):
        vc.lib()
    with pytest.raises(ImportError):
        vc.vc_schedule_action(0, 40, 4)
