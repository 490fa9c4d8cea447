"""The allocation-free neighbour-table entry point agrees with sc_build_map.

sc_build_neighbor_table_noalloc serves callers that cannot let a library
allocate device memory (fixed-budget plugin runtimes, loops that cannot absorb
cudaMalloc's implicit synchronisation, fully pre-reserved deployments).  It
keeps its hash table in a static device array shared by all calls, so this
test calls it twice in a row on different voxel sets (the second smaller than
the first, so stale slots from the first call would show) and compares each
result bit for bit with the allocating path: sc_build_map followed by
sc_get_neighbor_table.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

from sparse_voxel_convolution_coord_b300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_voxel_convolution_coord_b300 as sc
    from sparse_voxel_convolution_coord_b300 import build_lib
    build_lib.build()
    lib = sc.load_library()
    lib.sc_build_neighbor_table_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                                    ctypes.c_int32, ctypes.c_void_p,
                                                    ctypes.c_void_p, ctypes.c_void_p]
    lib.sc_build_neighbor_table_noalloc.restype = ctypes.c_int
    return lib


def noalloc_table(lib, coords_dev, res):
    n = coords_dev.shape[0]
    nbr = torch.full((max(n, 1), 27), 7, dtype=torch.int32, device="cuda")
    pairs = ctypes.c_int64(-1)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.sc_build_neighbor_table_noalloc(ctypes.c_void_p(coords_dev.data_ptr()), n, res,
                                             ctypes.c_void_p(nbr.data_ptr()),
                                             ctypes.byref(pairs), stream)
    return rc, nbr[:n].cpu().numpy(), pairs.value


def allocating_table(coords_dev, res):
    import sparse_voxel_convolution_coord_b300 as sc
    m = sc.sc_build_map(coords_dev, res)
    nbr = sc.sc_get_neighbor_table(m).cpu().numpy()
    pairs = sc.sc_map_pairs(m)
    m.free()
    return nbr, pairs


def test_noalloc_matches_allocating_path_twice(lib):
    import sparse_voxel_convolution_coord_b300 as sc
    for key in (5, 3, 2):     # 395,775, 29,850, then 20,236 voxels over the same scratch
        p = synth.make_problem(key)
        coords = torch.from_numpy(p.coords).cuda()
        rc, nbr, pairs = noalloc_table(lib, coords, p.res)
        assert rc == sc.SC_OK, sc.sc_last_error_msg()
        want, want_pairs = allocating_table(coords, p.res)
        np.testing.assert_array_equal(nbr, want)
        assert pairs == want_pairs


def test_noalloc_key_space_retry(lib):
    """Batch indices beyond the 32-bit key space at res 64 (>= 16383) make the
    build retry with 64-bit keys; the table still matches the allocating path."""
    import sparse_voxel_convolution_coord_b300 as sc
    rng = np.random.default_rng(11)
    rows = []
    for b in (0, 16383, 20000):
        xyz = np.argwhere(rng.random((64, 64, 64)) < 0.01)
        rows.append(np.concatenate([np.full((len(xyz), 1), b), xyz], axis=1))
    # argwhere's rows are column-major: make them C-contiguous for the raw call
    coords = torch.from_numpy(np.ascontiguousarray(np.concatenate(rows), dtype=np.int32)).cuda()
    rc, nbr, pairs = noalloc_table(lib, coords, 64)
    assert rc == sc.SC_OK, sc.sc_last_error_msg()
    want, want_pairs = allocating_table(coords, 64)
    np.testing.assert_array_equal(nbr, want)
    assert pairs == want_pairs


def test_noalloc_rejects_beyond_limit_and_reports_errors(lib):
    import sparse_voxel_convolution_coord_b300 as sc
    coords = torch.zeros((4, 4), dtype=torch.int32, device="cuda")
    out = torch.empty((4, 27), dtype=torch.int32, device="cuda")
    rc = lib.sc_build_neighbor_table_noalloc(ctypes.c_void_p(coords.data_ptr()), (1 << 19) + 1,
                                             16, ctypes.c_void_p(out.data_ptr()), None, None)
    assert rc == sc.SC_ERR_UNSUPPORTED
    assert "static scratch limit" in sc.sc_last_error_msg()
    dup = torch.tensor([[0, 1, 1, 1], [0, 1, 1, 1]], dtype=torch.int32, device="cuda")
    rc, _, _ = noalloc_table(lib, dup, 4)
    assert rc == sc.SC_ERR_DUPLICATE


_FRESH_PROCESS = r"""
import ctypes, json, sys, threading
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import sparse_voxel_convolution_coord_b300 as sc
from sparse_voxel_convolution_coord_b300 import synth

lib = sc.load_library()
lib.sc_build_neighbor_table_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
p = synth.make_problem(2)
coords = torch.from_numpy(p.coords).cuda()
outs = [torch.full((p.n, 27), 7, dtype=torch.int32, device="cuda") for _ in range(2)]
torch.cuda.synchronize()
got = {}


def call(i):
    pairs = ctypes.c_int64(-1)
    got[i] = (lib.sc_build_neighbor_table_noalloc(ctypes.c_void_p(coords.data_ptr()), p.n, p.res,
                                                  ctypes.c_void_p(outs[i].data_ptr()),
                                                  ctypes.byref(pairs), None), pairs.value)


# the first call into the library in this process, from a thread that never called it
t = threading.Thread(target=call, args=(0,))
t.start()
t.join()
torch.cuda.synchronize()
# a second call, from another fresh thread, with the device's free memory read around it
free0 = torch.cuda.mem_get_info()[0]
t = threading.Thread(target=call, args=(1,))
t.start()
t.join()
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
m = sc.sc_build_map(coords, p.res)
want = sc.sc_get_neighbor_table(m).cpu().numpy()
print(json.dumps({"rc": [got[0][0], got[1][0]], "pairs": [got[0][1], got[1][1]],
                  "want_pairs": m.pairs, "free": [free0, free1],
                  "equal": [bool(np.array_equal(o.cpu().numpy(), want)) for o in outs]}))
m.free()
"""


def test_noalloc_first_call_from_a_fresh_thread_of_a_fresh_process(lib):
    """In a new process, the first call into the library is the no-alloc entry,
    made from a new host thread: its table equals the allocating path's.  A
    second call from another new thread leaves the device's free memory
    unchanged (no allocation on the device), and the status read-back uses the
    calling thread's stack (no pinned host buffer)."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH_PROCESS, root], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["rc"] == [0, 0]
    assert d["equal"] == [True, True]
    assert d["pairs"] == [d["want_pairs"]] * 2
    assert d["free"][0] == d["free"][1]
