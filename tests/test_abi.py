"""The C-ABI library loads and exports every symbol include/*.h declares;
host-side argument checks that need no GPU."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def native():
    from realtime_transformer_gb300 import build
    build.build()
    from realtime_transformer_gb300 import _native
    return _native


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(frt_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["frt_ffn_plan_create", "frt_ffn_plan_destroy", "frt_ffn_load_weights", "frt_ffn_calibrate",
                     "frt_ffn_get_scales", "frt_ffn_set_scales", "frt_ffn_forward", "frt_ffn_graph_capture",
                     "frt_ffn_graph_replay", "frt_ffn_debug_trace", "frt_ffn_last_error"]:
        assert required in names


def test_library_exports_every_declared_symbol(native):
    lib = ctypes.CDLL(native.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(native.SIGNATURES), "binding and header disagree"


def test_null_plan_is_rejected_without_touching_the_gpu(native):
    L = native.lib()
    assert L.frt_ffn_forward(None, None, None, None, 1, None) == 1
    assert L.frt_ffn_graph_replay(None, 1, None) == 1
    assert L.frt_ffn_graph_autotune(None, None, None, None, 1, 3, 10, None, None, None) == 1
    assert L.frt_ffn_set_scales(None, None, None) == 1
    assert L.frt_ffn_plan_destroy(None) == 0
    assert "null plan" in native.frt_ffn_last_error()


def test_plan_create_validates_shapes_before_any_cuda_call(native):
    L = native.lib()
    out = ctypes.c_void_p()
    assert L.frt_ffn_plan_create(100, 1024, 0, 8, 1, ctypes.byref(out)) == 1
    assert "multiples of 128" in native.frt_ffn_last_error()
    assert L.frt_ffn_plan_create(256, 1024, 7, 8, 1, ctypes.byref(out)) == 1
    assert L.frt_ffn_plan_create(256, 1024, 0, 0, 1, ctypes.byref(out)) == 1
    assert L.frt_ffn_plan_create(256, 1024, 0, 8, 0, ctypes.byref(out)) == 1
    assert out.value is None


def test_errors_raise_with_the_library_message(native):
    with pytest.raises(native.FrtError) as ei:
        native.frt_ffn_plan_create(256, 1000, 0, 8, 1)
    assert ei.value.name == "FRT_ERR_INVALID_ARG"


def test_product_package_does_not_import_the_oracle():
    import ast
    pkg = os.path.join(ROOT, "realtime_transformer_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.py"), recursive=True):
        tree = ast.parse(open(path).read())
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                mods = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                mods = [node.module or ""]
            else:
                continue
            assert not any(m.split(".")[0] in ("oracle", "synthetic") for m in mods), path


def test_nvfp4_entry_points_check_arguments_before_any_cuda_call(native):
    L = native.lib()
    out = ctypes.c_void_p()
    assert L.frt_fp4_plan_create(1000, 4096, 0, 8, 1, ctypes.byref(out)) == 1
    assert "multiples of 256" in native.frt_ffn_last_error()
    assert L.frt_fp4_plan_create(1024, 4096, 5, 8, 1, ctypes.byref(out)) == 1
    assert L.frt_fp4_plan_create(1024, 4096, 0, 0, 1, ctypes.byref(out)) == 1
    assert L.frt_fp4_forward(None, None, None, None, 1, None) == 1
    assert L.frt_fp4_set_scales(None, None) == 1
    assert L.frt_fp4_device_status(None, None) == 1
    assert L.frt_fp4_debug_stall(None, 8, None) == 1
    assert L.frt_fp4_forward_profile(None, None, None, None, 8, 1, None, None, None) == 1
    assert L.frt_fp4_debug_trace_from(None, 0, None, None, None, None, None, None, None, None, None, None, None,
                                      None, None, 8, None) == 1
    assert L.frt_fp4_debug_trace(None, 0, None, None, None, None, None, None, None, None, None, None, None, None,
                                 8, None) == 1
    assert L.frt_fp4_debug_weights(None, 0, 0, None, None, None) == 1
    assert L.frt_fp4_plan_destroy(None) == 0
    # the diagnostic GEMM rejects shapes its tiles do not cover
    assert L.frt_nvfp4_gemm(None, None, None, None, 8, 128, 256, ctypes.c_float(1.0), None, 1, None, None, None,
                            None) == 1
