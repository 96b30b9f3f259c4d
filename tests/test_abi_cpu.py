"""CPU-only checks of the C ABI: the library loads, exports every function the
header declares, and its host-side validation answers without a GPU."""
import ctypes
import os
import re

import pytest

import decode_sampling_tail_gb300 as dst
from decode_sampling_tail_gb300 import build as dbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tail.h")


@pytest.fixture(scope="module")
def L():
    dbuild.build()
    return dst.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|void|const char\*)\s+(tail_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    assert set(declared_functions()) == set(dst.EXPORTS)


def test_library_exports_every_declared_function(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} missing from libtail.so"


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5):
        assert L.tail_status_string(code)
    assert b"unknown" in L.tail_status_string(42)


def test_config_validation_without_gpu(L):
    h = ctypes.c_void_p()
    def create(**kw):
        base = dict(H=256, hidden_actual=0, V=4096, k=16, gbs_max=4, eps=1e-5, hidden_dtype=0,
                    zero_interleaved_pad=1, deferred_rms=1, path=0)
        base.update(kw)
        cfg = dst.tail_config(*[base[f[0]] for f in dst.tail_config._fields_])
        return L.tail_create(ctypes.byref(cfg), 0, ctypes.byref(h))
    assert create(H=0) == dst.TAIL_ERR_INVALID_ARG
    assert create(k=0) == dst.TAIL_ERR_INVALID_ARG
    assert create(k=5000) == dst.TAIL_ERR_INVALID_ARG
    assert create(k=64, V=32) == dst.TAIL_ERR_INVALID_ARG          # k > V
    assert create(hidden_actual=300) == dst.TAIL_ERR_INVALID_ARG   # H_u > H
    assert create(gbs_max=0) == dst.TAIL_ERR_INVALID_ARG
    assert create(hidden_dtype=7) == dst.TAIL_ERR_INVALID_ARG
    assert create(eps=-1.0) == dst.TAIL_ERR_INVALID_ARG
    assert create(H=100) == dst.TAIL_ERR_UNSUPPORTED               # H % 16
    assert create(V=4100) == dst.TAIL_ERR_UNSUPPORTED              # V % 16
    assert create(path=3) == dst.TAIL_ERR_INVALID_ARG
    assert create(path=-1) == dst.TAIL_ERR_INVALID_ARG
    assert L.tail_create(None, 0, ctypes.byref(h)) == dst.TAIL_ERR_INVALID_ARG
    assert h.value is None


def test_null_handle_calls(L):
    assert L.tail_run(None, None, None, None, None, 4, 1, None, None, None) == dst.TAIL_ERR_INVALID_ARG
    assert L.tail_run_ex(None, None, None, None, None, 4, 1, None, None, None, None, None) == \
        dst.TAIL_ERR_INVALID_ARG
    assert L.tail_run_host(None, None, None, None, None, 4, 1, None, None, None) == dst.TAIL_ERR_INVALID_ARG
    assert L.tail_check(None) == dst.TAIL_ERR_INVALID_ARG
    assert L.tail_get_info(None, None) == dst.TAIL_ERR_INVALID_ARG
    assert L.tail_prepare_weight(None, None, None) == dst.TAIL_ERR_INVALID_ARG
    L.tail_destroy(None)


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(dst, "_lib", None)
    with pytest.raises(dst.TailLibraryMissing):
        dst.lib(str(tmp_path / "absent.so"))


def header_struct_fields(name):
    """Field names of `typedef struct { ... } name;` in include/tail.h, in order."""
    import re
    text = open(HEADER).read()
    body = re.search(r"typedef struct \{([^{}]*)\}\s*" + name + ";", text).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    return re.findall(r"\b(\w+);", body)


def test_python_structs_mirror_the_header():
    assert [f[0] for f in dst.tail_config._fields_] == header_struct_fields("tail_config")
    assert [f[0] for f in dst.tail_info._fields_] == header_struct_fields("tail_info")


def test_path_constants_mirror_the_header():
    import re
    text = open(HEADER).read()
    for key, name in (("auto", "AUTO"), ("gemv", "GEMV"), ("tensor", "TENSOR")):
        assert int(re.search(r"TAIL_PATH_" + name + r"\s*=\s*(\d+)", text).group(1)) == dst.PATHS[key]
    assert int(re.search(r"#define TAIL_TC_ALL_ROWS_MAX_V (\d+)", text).group(1)) == dst.TC_ALL_ROWS_MAX_V
