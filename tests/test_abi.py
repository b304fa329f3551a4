"""The C-ABI library builds for sm_103a, loads, and exports what the header
declares; the device translation units are compiled without contraction.
No compute call is made here (no GPU needed)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "seqsum.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(seqsum_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def libpath():
    from parity_binade_chunked_gb300 import build
    return build.build()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["seqsum_f64", "seqsum_f64_batched", "seqsum_f64_batched_sized", "seqsum_get_stats",
                     "seqsum_strerror", "seqsum_release_workspace"]:
        assert required in names, names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in seqsum.h but not exported"


def test_strerror_and_version_without_gpu(libpath):
    lib = ctypes.CDLL(libpath)
    lib.seqsum_strerror.restype = ctypes.c_char_p
    lib.seqsum_version.restype = ctypes.c_char_p
    assert lib.seqsum_strerror(0) == b"ok"
    assert b"invalid" in lib.seqsum_strerror(-1)
    assert b"sm_103a" in lib.seqsum_version()


def test_argument_errors_need_no_gpu(libpath):
    lib = ctypes.CDLL(libpath)
    lib.seqsum_f64.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p,
                               ctypes.c_void_p]
    # n < 0 and a null out are rejected before any CUDA call
    assert lib.seqsum_f64(None, -1, 0.0, ctypes.c_void_p(8), None) == -1
    assert lib.seqsum_f64(None, 0, 0.0, None, None) == -1
    assert lib.seqsum_f64(None, 5, 0.0, ctypes.c_void_p(8), None) == -1
    lib.seqsum_f64_batched.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int32] + [ctypes.c_void_p] * 3
    assert lib.seqsum_f64_batched(None, None, -1, None, None, None) == -1
    assert lib.seqsum_f64_batched(None, None, 0, None, None, None) == 0
    # a plan is host state until its first call; bad arguments are refused first
    lib.seqsum_plan_create.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
    lib.seqsum_plan_destroy.argtypes = [ctypes.c_void_p]
    lib.seqsum_f64_planned.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int64, ctypes.c_double] + [ctypes.c_void_p] * 2
    assert lib.seqsum_plan_create(None) == -1
    h = ctypes.c_void_p()
    assert lib.seqsum_plan_create(ctypes.byref(h)) == 0 and h.value
    assert lib.seqsum_f64_planned(None, None, 0, 0.0, ctypes.c_void_p(8), None) == -1
    assert lib.seqsum_f64_planned(h, None, 5, 0.0, ctypes.c_void_p(8), None) == -1
    assert lib.seqsum_f64_planned(h, None, -1, 0.0, ctypes.c_void_p(8), None) == -1
    assert lib.seqsum_f64_planned(h, None, 0, 0.0, None, None) == -1
    lib.seqsum_plan_destroy(h)
    lib.seqsum_plan_destroy(None)


def test_device_code_is_built_strict_fp():
    """Research-1433 / ADR-1391: the device translation units build with
    --fmad=false (no contraction on the device path)."""
    from parity_binade_chunked_gb300 import build
    assert "--fmad=false" in build.NVCC_FLAGS
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)
    import oracle
    for flag in ["-ffp-contract=off", "-fno-fast-math", "-fno-tree-vectorize"]:
        assert flag in oracle.CFLAGS


def test_product_has_no_oracle_or_cpu_fallback():
    """The product path never imports the oracle, and the binding has no CPU
    path: its only compute entry points call into libseqsum."""
    pkg = os.path.join(ROOT, "parity_binade_chunked_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "seqsum_oracle" not in text, f
