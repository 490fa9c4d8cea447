"""CPU oracle for the 3x3x3 submanifold sparse convolution.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, fp64 statement of
what the CUDA library computes, written from the method's description and
sharing no code with the library.  Only ``tests/``, the package smoke check
and the benchmark's CPU-baseline leg may import it; the library itself never
does, and never falls back to it.

Sources followed (page title, section):
  * "Running TRELLIS.2 on a Mac (1/3)", "Swapping out the CUDA libraries one
    at a time" / Sparse 3D convolution -- spatial hash, per-offset gather,
    multiply, accumulate into the output site;
  * "Porting TRELLIS.2 From Python to Rust and Metal", section V -- neighbour
    table built once per level, gather-GEMM, bias in the same pass;
  * "FABLE_STARTUP_PACKET.md", section 5 -- weights (Co,Kd,Kh,Kw,Ci) viewed as
    (Kvol, Ci, Co).

Every function below is pinned by ``tests/test_oracle_pins.py`` against
routes that do not go through this code: brute-force neighbour search, a
dense index volume, a dense fp64 Conv3d, closed forms and invariants.
"""
import ctypes
import numpy as np

from . import build_oracle

OK, BAD_ARG, COORD_RANGE, DUPLICATE = 0, 1, 2, 3


class OracleError(RuntimeError):
    def __init__(self, code, what):
        super().__init__("oracle %s failed with status %d" % (what, code))
        self.code = code


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """The oracle functions bound to one build of ``sc_oracle.cpp``."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.oracle_displacement.argtypes = [ctypes.c_int, P, P, P]
        lib.oracle_build_neighbor_table.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P]
        lib.oracle_pairs.argtypes = [P, ctypes.c_int64, P, P, P]
        lib.oracle_pairs.restype = ctypes.c_int64
        lib.oracle_conv.argtypes = [P, ctypes.c_int64, P, ctypes.c_int64,
                                    ctypes.c_int32, P, ctypes.c_int32, P, P,
                                    ctypes.c_int32]
        lib.oracle_max_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def displacement(self, k):
        """(dx, dy, dz) of offset k."""
        d = [ctypes.c_int(), ctypes.c_int(), ctypes.c_int()]
        rc = self.lib.oracle_displacement(k, *[ctypes.byref(v) for v in d])
        if rc:
            raise OracleError(rc, "displacement")
        return tuple(v.value for v in d)

    def build_neighbor_table(self, coords, res):
        """int32 [n,27] neighbour table of int32 coords [n,4] = (b,x,y,z)."""
        coords = np.ascontiguousarray(coords, dtype=np.int32).reshape(-1, 4)
        n = coords.shape[0]
        nbr = np.empty((n, 27), dtype=np.int32)
        rc = self.lib.oracle_build_neighbor_table(_ptr(coords), n, int(res), _ptr(nbr))
        if rc:
            raise OracleError(rc, "build_neighbor_table")
        return nbr

    def pairs(self, nbr):
        """CSR pair lists: (off[28] int64, in[P] int32, out[P] int32)."""
        nbr = np.ascontiguousarray(nbr, dtype=np.int32).reshape(-1, 27)
        n = nbr.shape[0]
        p = self.lib.oracle_pairs(_ptr(nbr), n, None, None, None)
        off = np.empty(28, dtype=np.int64)
        pin = np.empty(p, dtype=np.int32)
        pout = np.empty(p, dtype=np.int32)
        self.lib.oracle_pairs(_ptr(nbr), n, _ptr(off), _ptr(pin), _ptr(pout))
        return off, pin, pout

    def conv(self, nbr, feats, weight, bias=None, threads=0):
        """fp64 [m,cout] = bias + sum_k gather(feats, nbr[:,k]) @ weight[k].

        nbr [m,27] may be the whole table or a subset of its rows (the output
        rows wanted).  feats [n,cin] and weight [27,cin,cout] are taken as
        float32 (a bf16 input must be widened to float32 first, which is
        exact); bias [cout] or None.
        """
        nbr = np.ascontiguousarray(nbr, dtype=np.int32).reshape(-1, 27)
        feats = np.ascontiguousarray(feats, dtype=np.float32)
        weight = np.ascontiguousarray(weight, dtype=np.float32)
        n, cin = feats.shape
        m = nbr.shape[0]
        assert weight.shape[:2] == (27, cin)
        cout = weight.shape[2]
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        out = np.empty((m, cout), dtype=np.float64)
        rc = self.lib.oracle_conv(_ptr(nbr), m, _ptr(feats), n, cin, _ptr(weight),
                                  cout, _ptr(b), _ptr(out), int(threads))
        if rc:
            raise OracleError(rc, "conv")
        return out

    def sparse_conv(self, coords, res, feats, weight, bias=None, threads=0):
        """Neighbour table then convolution: the whole method on the CPU."""
        return self.conv(self.build_neighbor_table(coords, res), feats, weight,
                         bias, threads)

    def max_threads(self):
        return int(self.lib.oracle_max_threads())


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build_oracle.build())
    return _default


def displacement(k):
    return default().displacement(k)


def build_neighbor_table(coords, res):
    return default().build_neighbor_table(coords, res)


def pairs(nbr):
    return default().pairs(nbr)


def conv(nbr, feats, weight, bias=None, threads=0):
    return default().conv(nbr, feats, weight, bias, threads)


def sparse_conv(coords, res, feats, weight, bias=None, threads=0):
    return default().sparse_conv(coords, res, feats, weight, bias, threads)


def max_threads():
    return default().max_threads()
