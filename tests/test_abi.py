"""The C-ABI library builds for sm_103a, loads, and exports every entry
point that include/megamoe.h declares; host-side argument checks that run
before any CUDA call behave as documented.  No GPU needed."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    from moe_layer_serving_gb300 import build
    return build.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "megamoe.h")).read()
    return sorted(set(re.findall(r"^MM_API\s+[\w\s\*]+?\b(mm_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("mm_create", "mm_set_eplb_map", "mm_forward", "mm_read_counts", "mm_set_weights",
                     "mm_bind_layer", "mm_set_recording", "mm_set_route", "mm_reserve", "mm_destroy"):
        assert required in names


def test_library_exports_every_declared_symbol(built):
    lib = C.CDLL(built)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_debug_library_exports_every_declared_symbol(built):
    # the build with device-side bounds checks: the same entry points
    from moe_layer_serving_gb300 import build
    assert os.path.exists(build.DEBUG_LIB)
    lib = C.CDLL(build.DEBUG_LIB)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_exposes_c_names(built):
    import moe_layer_serving_gb300 as mm
    for n in _declared():
        assert callable(getattr(mm, n)), n


def test_library_targets_sm103a(built):
    # the fatbin carries sm_103a code only (checked from the build command, not the binary)
    from moe_layer_serving_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


@pytest.mark.parametrize("args", [(0, 8, 2, 256, 128), (8, 4, 2, 256, 128), (8, 8, 0, 256, 128),
                                  (8, 8, 9, 256, 128), (4, 4, 5, 256, 128), (8, 8, 2, 200, 128),
                                  (8, 8, 2, 256, 96), (600, 600, 2, 256, 128)])
def test_create_rejects_unsupported_shapes_before_touching_cuda(built, args):
    import moe_layer_serving_gb300 as mm
    h = C.c_void_p()
    assert mm.lib().mm_create(*args, C.byref(h)) == mm.MM_ERR_UNSUPPORTED
    assert not h.value


def test_null_handle_calls_are_invalid(built):
    import moe_layer_serving_gb300 as mm
    L = mm.lib()
    assert L.mm_forward(None, None, None, None, None, 1, None) == mm.MM_ERR_INVALID_ARG
    assert L.mm_bind_layer(None, 0) == mm.MM_ERR_INVALID_ARG
    assert L.mm_reserve(None, 16) == mm.MM_ERR_INVALID_ARG
    assert L.mm_set_shared_experts(None, 1) == mm.MM_ERR_INVALID_ARG
    assert L.mm_set_activation_format(None, 0) == mm.MM_ERR_INVALID_ARG
    assert L.mm_destroy(None) == mm.MM_OK
    assert L.mm_status_string(4) == b"token count above capacity"


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import moe_layer_serving_gb300 as mm
    monkeypatch.setattr(mm, "library_path", str(tmp_path / "absent.so"))
    monkeypatch.setattr(mm, "debug_library_path", str(tmp_path / "absent_debug.so"))
    monkeypatch.setattr(mm, "_libs", {})
    with pytest.raises(RuntimeError, match="missing"):
        mm.lib()
    with pytest.raises(RuntimeError, match="missing"):
        mm.lib(debug=True)
