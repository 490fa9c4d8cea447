"""The C ABI's boundary and failure paths on the device.

* sc_forward rejects operands that are not this GPU's own device memory, and
  outputs that overlap their inputs, on the host, with nothing launched;
* sc_set_allocator routes every map buffer through a caller's allocator (here
  PyTorch's caching allocator, through ctypes callbacks);
* sc_set_probe_limit makes the hash insert's bounded probe loop give up, so
  that SC_ERR_TABLE_FULL is reported (and nothing faults);
* sc_build_map_async builds the same map as sc_build_map without a host
  synchronisation, and reports the device-found errors later.
"""
import ctypes

import numpy as np
import pytest

import oracle
from sparse_voxel_convolution_coord_b300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


@pytest.fixture(scope="module")
def sc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_voxel_convolution_coord_b300 as m
    from sparse_voxel_convolution_coord_b300 import build_lib
    build_lib.build()
    m.load_library()
    return m


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(dtype) if dtype is not None else t


def table(sc, m):
    return sc.sc_get_neighbor_table(m).cpu().numpy()


# ---------------------------------------------------------------------------
# operand memory

def test_foreign_operand_memory_is_rejected_before_launch(sc):
    p = synth.make_problem(3)          # C=256: the kernel with the W multicast
    m = sc.sc_build_map(dev(p.coords), p.res)
    lib = sc.load_library()
    f = dev(p.feats, torch.bfloat16)
    w = dev(p.weight, torch.bfloat16)
    out = torch.empty((p.n, 256), device="cuda")
    w_pinned = torch.from_numpy(p.weight).to(torch.bfloat16).pin_memory()
    w_pageable = torch.from_numpy(p.weight).to(torch.bfloat16)
    bias_pinned = torch.from_numpy(p.bias).pin_memory()
    out_pinned = torch.empty((p.n, 256)).pin_memory()
    c0 = sc.sc_kernel_launches()
    cases = [
        (f.data_ptr(), w_pinned.data_ptr(), None, out.data_ptr()),      # pinned host W
        (f.data_ptr(), w_pageable.data_ptr(), None, out.data_ptr()),    # pageable host W
        (f.data_ptr(), w.data_ptr(), bias_pinned.data_ptr(), out.data_ptr()),
        (f.data_ptr(), w.data_ptr(), None, out_pinned.data_ptr()),
    ]
    for fp, wp, bp, op in cases:
        rc = lib.sc_forward(P(m.ptr), P(fp), P(wp), None if bp is None else P(bp), P(op),
                            256, 256, sc.SC_BF16, None)
        assert rc == sc.SC_ERR_INVALID_ARG
        assert "device memory" in sc.sc_last_error_msg()
    assert sc.sc_kernel_launches() == c0      # nothing was launched
    # the same call on device memory runs
    assert lib.sc_forward(P(m.ptr), P(f.data_ptr()), P(w.data_ptr()), None, P(out.data_ptr()),
                          256, 256, sc.SC_BF16, None) == sc.SC_OK
    sc.sc_device_status(m)
    m.free()


def test_output_overlapping_inputs_is_rejected(sc):
    p = synth.make_problem(2)
    m = sc.sc_build_map(dev(p.coords), p.res)
    lib = sc.load_library()
    f = dev(p.feats, torch.bfloat16)
    w = dev(p.weight, torch.bfloat16)
    big = torch.zeros((2 * p.n, 64), device="cuda")
    c0 = sc.sc_kernel_launches()
    # out on top of the features (fp32 out over bf16 feats: any overlap counts)
    assert lib.sc_forward(P(m.ptr), P(f.data_ptr()), P(w.data_ptr()), None, P(f.data_ptr()),
                          64, 64, sc.SC_BF16, None) == sc.SC_ERR_INVALID_ARG
    # a residual shifted by one row against out
    assert lib.sc_forward_ex(P(m.ptr), P(f.data_ptr()), P(w.data_ptr()), None,
                             P(big.data_ptr() + 64 * 4), P(big.data_ptr()), 64, 64, sc.SC_BF16,
                             sc.SC_ACT_NONE, sc.SC_F32, None) == sc.SC_ERR_INVALID_ARG
    assert sc.sc_kernel_launches() == c0
    m.free()


# ---------------------------------------------------------------------------
# installed allocator

def test_allocator_routes_every_map_buffer(sc):
    """A counting allocator over PyTorch's caching allocator: a build, a
    forward and the pair lists go through it, the map matches the default
    path bit for bit, and every allocation is returned by sc_free_map."""
    lib = sc.load_library()
    ALLOC = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p)
    FREE = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)
    live, log = {}, []

    def _alloc(nbytes, stream, ctx):
        ptr = torch.cuda.caching_allocator_alloc(int(nbytes), stream=int(stream or 0))
        live[ptr] = nbytes
        log.append(("alloc", nbytes))
        return ptr

    def _free(ptr, stream, ctx):
        assert ptr in live
        del live[ptr]
        log.append(("free", 0))
        torch.cuda.caching_allocator_delete(ptr)

    a_cb, f_cb = ALLOC(_alloc), FREE(_free)
    lib.sc_set_allocator.argtypes = [P, P, P]
    p = synth.make_problem(2)
    coords = dev(p.coords)
    ref = sc.sc_build_map(coords, p.res)
    want = table(sc, ref)
    want_pairs = ref.pairs
    ref.free()
    assert lib.sc_set_allocator(ctypes.cast(a_cb, P), ctypes.cast(f_cb, P), None) == sc.SC_OK
    try:
        m = sc.sc_build_map(coords, p.res)
        assert len(live) == 1                      # the map's one block
        np.testing.assert_array_equal(table(sc, m), want)
        assert m.pairs == want_pairs
        off, pin, pout = sc.sc_get_pairs(m)        # its scratch also comes from the allocator
        assert int(off[27]) == want_pairs
        out = sc.sc_forward(m, dev(p.feats, torch.bfloat16), dev(p.weight, torch.bfloat16),
                            dev(p.bias))
        sc.sc_device_status(m)
        m.free()
        torch.cuda.synchronize()
        assert not live, "allocations not returned: %s" % live
        assert sum(1 for k, _ in log if k == "alloc") == 2
    finally:
        lib.sc_set_allocator(None, None, None)
    got = out.cpu().numpy().astype(np.float64)
    ref_out = oracle.conv(oracle.build_neighbor_table(p.coords, p.res), p.feats, p.weight, p.bias)
    assert np.linalg.norm(got - ref_out) / np.linalg.norm(ref_out) <= 2e-3


# ---------------------------------------------------------------------------
# bounded probe loop

def test_probe_limit_reports_table_full(sc):
    """With one probe allowed, any key whose home slot is taken by another key
    fails the insertion: the build returns SC_ERR_TABLE_FULL (64^3, ~20k
    voxels: brick groups collide), and works again once the limit is lifted."""
    p = synth.make_problem(2)
    coords = dev(p.coords)
    sc.sc_set_probe_limit(1)
    try:
        with pytest.raises(sc.ScError) as e:
            sc.sc_build_map(coords, p.res)
        assert e.value.code == sc.SC_ERR_TABLE_FULL
        m = sc.sc_build_map_async(coords, p.res, 1)
        with pytest.raises(sc.ScError) as e:
            sc.sc_map_status(m)
        assert e.value.code == sc.SC_ERR_TABLE_FULL
        assert sc.load_library().sc_map_pairs(P(m.ptr)) == -1
        m.free()
        with pytest.raises(sc.ScError) as e:
            sc.sc_build_neighbor_table_noalloc(coords, p.res)
        assert e.value.code == sc.SC_ERR_TABLE_FULL
        # a voxel set with no collision at all passes under the same limit
        one = dev(np.array([[0, 3, 4, 5]], np.int32))
        sc.sc_build_map(one, 8).free()
    finally:
        sc.sc_set_probe_limit(0)
    m = sc.sc_build_map(coords, p.res)
    np.testing.assert_array_equal(table(sc, m), oracle.build_neighbor_table(p.coords, p.res))
    m.free()
    assert sc.load_library().sc_set_probe_limit(-1) == sc.SC_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# asynchronous build

@pytest.mark.parametrize("key", [1, 2, 3, 4, 5])
def test_async_build_matches_oracle(sc, key):
    p = synth.make_problem(key)
    coords = dev(p.coords)
    c0 = sc.sc_kernel_launches()
    m = sc.sc_build_map_async(coords, p.res, int(p.coords[:, 0].max()) + 1)
    assert sc.sc_kernel_launches() - c0 == 3    # init, insert, query; no synchronisation
    want = oracle.build_neighbor_table(p.coords, p.res)
    np.testing.assert_array_equal(table(sc, m), want)
    sc.sc_map_status(m)
    assert m.pairs == int((want >= 0).sum())
    m.free()


@pytest.mark.parametrize("res,nbatch,density", [(1, 3, 1.0), (2, 2, 0.7), (33, 4, 0.2),
                                               (31, 1, 0.5), (64, 6, 0.05)])
def test_async_build_small_and_odd_grids(sc, res, nbatch, density):
    """Asynchronous builds on small and odd grids: cells on the grid's faces,
    res 1 and 2, res not a multiple of 32, an empty batch element, unused
    batch indices below nbatch and shuffled rows: the map equals the
    oracle's."""
    rng = np.random.default_rng(res * 100 + nbatch)
    rows = []
    for b in range(nbatch):
        if nbatch > 2 and b == 1:
            continue                                   # an empty batch element
        xyz = np.argwhere(rng.random((res, res, res)) < density)
        rows.append(np.concatenate([np.full((len(xyz), 1), b), xyz], axis=1))
    c = np.concatenate(rows).astype(np.int32)
    c = np.ascontiguousarray(c[rng.permutation(len(c))])
    m = sc.sc_build_map_async(dev(c), res, nbatch + 1)
    np.testing.assert_array_equal(table(sc, m), oracle.build_neighbor_table(c, res))
    sc.sc_map_status(m)
    m.free()


def test_async_build_then_forward_without_status_read(sc):
    """A forward enqueued right after the asynchronous build, before anything
    reads the build's status, sees the finished map (stream order)."""
    p = synth.make_problem(3)
    m = sc.sc_build_map_async(dev(p.coords), p.res, 1)
    out = sc.sc_forward(m, dev(p.feats, torch.bfloat16), dev(p.weight, torch.bfloat16),
                        dev(p.bias))
    got = out.cpu().numpy().astype(np.float64)
    sc.sc_device_status(m)
    m.free()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.arange(0, 128), np.arange(p.n - 300, p.n),
                                     rng.choice(p.n, size=1500, replace=False)]))
    ref = oracle.conv(oracle.build_neighbor_table(p.coords, p.res)[rows], p.feats, p.weight,
                      p.bias)
    err = got[rows] - ref
    assert np.linalg.norm(err) / np.linalg.norm(ref) <= 2e-3
    assert np.abs(err).max() <= 1e-2 * np.linalg.norm(ref) / np.sqrt(ref.size)


def test_async_build_wide_keys_and_shuffled_rows(sc):
    """nbatch beyond the 32-bit key space at res 64 selects 64-bit keys up
    front; rows in random order.  The map still equals the oracle's."""
    rng = np.random.default_rng(9)
    rows = []
    for b in (0, 16383, 20000):
        xyz = np.argwhere(rng.random((64, 64, 64)) < 0.01)
        rows.append(np.concatenate([np.full((len(xyz), 1), b), xyz], axis=1))
    c = np.concatenate(rows).astype(np.int32)
    c = np.ascontiguousarray(c[rng.permutation(len(c))])
    m = sc.sc_build_map_async(dev(c), 64, 20001)
    np.testing.assert_array_equal(table(sc, m), oracle.build_neighbor_table(c, 64))
    sc.sc_map_status(m)
    m.free()


@pytest.mark.parametrize("coords,res,nbatch,code", [
    ([[0, 0, 0, 8]], 8, 1, 2),                       # x/y/z == res
    ([[-1, 0, 0, 0]], 8, 1, 2),                      # negative batch
    ([[3, 1, 1, 1]], 8, 3, 2),                       # batch >= nbatch
    ([[0, 1, 2, 3], [0, 4, 4, 4], [0, 1, 2, 3]], 8, 1, 3),  # duplicate
])
def test_async_build_reports_device_errors_later(sc, coords, res, nbatch, code):
    m = sc.sc_build_map_async(dev(np.array(coords, np.int32)), res, nbatch)
    with pytest.raises(sc.ScError) as e:
        sc.sc_map_status(m)
    assert e.value.code == code
    # the error stays with the map
    lib = sc.load_library()
    assert lib.sc_map_pairs(P(m.ptr)) == -1 and sc.sc_last_error() == code
    assert lib.sc_device_status(P(m.ptr), None) == code
    m.free()


def test_async_build_rejects_bad_nbatch(sc):
    lib = sc.load_library()
    c = dev(np.array([[0, 1, 1, 1]], np.int32))
    assert lib.sc_build_map_async(P(c.data_ptr()), 1, 8, 0, None) is None
    assert sc.sc_last_error() == sc.SC_ERR_INVALID_ARG
    # res = 2^20: res^3 = 2^60 in a 63-bit key (n = 1) leaves room for 8 batch elements
    assert lib.sc_build_map_async(P(c.data_ptr()), 1, 1 << 20, 1 << 10, None) is None
    assert sc.sc_last_error() == sc.SC_ERR_UNSUPPORTED
