"""The C-ABI library builds, loads without a GPU and exports what sc.h declares.

Only host-side logic is exercised here (argument checks and handle
bookkeeping that return before any CUDA call); compute needs a GPU and lives
in test_gpu_*.py.
"""
import ctypes

import pytest

import sparse_voxel_convolution_coord_b300 as sc
from sparse_voxel_convolution_coord_b300 import build_lib


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return sc.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = sc.header_symbols()
    assert len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name


def test_deterministic_switch_checks_its_argument(lib):
    assert lib.sc_set_deterministic(2) == sc.SC_ERR_INVALID_ARG
    assert lib.sc_set_deterministic(1) == sc.SC_OK
    assert lib.sc_set_deterministic(0) == sc.SC_OK


def test_release_cached_memory_without_pools(lib):
    # no map built in this process: no pool exists, nothing to trim
    assert lib.sc_release_cached_memory() == sc.SC_OK


def test_launch_counter_is_exported(lib):
    assert sc.sc_kernel_launches() >= 0


def test_version(lib):
    assert "sm_103a" in sc.sc_version()


def test_build_rejects_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    assert lib.sc_build_map(None, -1, 4, None) is None
    assert sc.sc_last_error() == sc.SC_ERR_INVALID_ARG
    assert lib.sc_build_map(None, 10, 0, None) is None
    assert sc.sc_last_error() == sc.SC_ERR_INVALID_ARG
    assert lib.sc_build_map(None, 10, (1 << 20) + 1, None) is None
    assert sc.sc_last_error() == sc.SC_ERR_INVALID_ARG
    assert lib.sc_build_map(None, 10, 8, None) is None          # NULL coords
    assert sc.sc_last_error() == sc.SC_ERR_INVALID_ARG
    assert lib.sc_build_map(P(0x1004), 10, 8, None) is None     # not 16-byte aligned
    assert sc.sc_last_error() == sc.SC_ERR_INVALID_ARG
    assert lib.sc_build_map(None, 1 << 31, 8, None) is None
    assert sc.sc_last_error() == sc.SC_ERR_INVALID_ARG


def test_dead_handles_are_caught(lib):
    bogus = ctypes.c_void_p(0xdeadbeef0)
    assert lib.sc_free_map(bogus, None) == sc.SC_ERR_BAD_HANDLE
    assert lib.sc_map_size(bogus) == -1
    assert sc.sc_last_error() == sc.SC_ERR_BAD_HANDLE
    assert lib.sc_map_pairs(bogus) == -1
    assert lib.sc_forward(bogus, None, None, None, None, 16, 16, 1, None) == sc.SC_ERR_BAD_HANDLE
    assert lib.sc_get_neighbor_table(bogus, None, None) == sc.SC_ERR_BAD_HANDLE
    assert lib.sc_device_status(bogus, None) == sc.SC_ERR_BAD_HANDLE
    assert lib.sc_free_map(None, None) == sc.SC_OK


def test_allocator_pairs_must_match(lib):
    f = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p)(
        lambda b, s, c: None)
    lib.sc_set_allocator.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.sc_set_allocator(ctypes.cast(f, ctypes.c_void_p), None, None) == \
        sc.SC_ERR_INVALID_ARG
    assert lib.sc_set_allocator(None, None, None) == sc.SC_OK


def test_no_cpu_fallback_in_binding():
    """The binding never imports the oracle: the product path has no CPU route."""
    import inspect
    src = inspect.getsource(sc)
    assert "oracle" not in src.replace("no CPU fallback", "")


def test_header_is_plain_c(lib, tmp_path):
    """include/sc.h compiles as C99 and a C program links against libsc.so
    (no C++ in the ABI's declarations)."""
    import os
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "use_sc.c"
    src.write_text(
        '#include "sc.h"\n'
        "#include <stdio.h>\n"
        "int main(void) {\n"
        "  sc_handle h = sc_build_map(0, -1, 4, 0);\n"
        "  sc_activation a = SC_ACT_SILU;\n"
        "  sc_dtype d = SC_F16;\n"
        "  printf(\"%d %d %d %s\\n\", h == 0, (int)a, (int)d, sc_version());\n"
        "  return sc_last_error() == SC_ERR_INVALID_ARG ? 0 : 1;\n"
        "}\n")
    exe = tmp_path / "use_sc"
    libdir = os.path.dirname(sc.library_path())
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lsc",
                    "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("1 2 2 ")


def test_noalloc_source_calls_no_allocator():
    """The allocation-free entry point's file calls no allocating routine
    (comments aside): its scratch is the static device array, its status
    read-back a stack buffer."""
    import os
    import re
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = open(os.path.join(root, "sparse_voxel_convolution_coord_b300", "csrc",
                            "sc_noalloc.cu")).read()
    code = re.sub(r"//[^\n]*", "", src)
    for name in ("cudaMalloc", "cudaHostAlloc", "cudaMallocHost", "cudaFree",
                 "status_readback_buffer", "new ", "malloc("):
        assert name not in code, name
    assert "static __device__ __align__(256)" in code
