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
    (Kvol, Ci, Co);
  * "Porting TRELLIS.2 From Python to Rust and Metal", section V -- bias,
    rounding, activation and the residual add fused into the output pass
    (``epilogue`` and ``round_bf16`` below, plain numpy in fp64).

Every function below is pinned by ``tests/test_oracle_pins.py`` against
routes that do not go through this code: brute-force neighbour search, a
dense index volume, a dense fp64 Conv3d, closed forms and invariants.
"""
import ctypes
import numpy as np

from . import build_oracle

OK, BAD_ARG, COORD_RANGE, DUPLICATE = 0, 1, 2, 3
ACT_NONE, ACT_RELU, ACT_SILU = 0, 1, 2


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


# ---------------------------------------------------------------------------
# Fused epilogue ("Porting TRELLIS.2 From Python to Rust and Metal", section
# V: bias, rounding, activation and the residual add in the convolution's
# output pass).  The pages name neither the activation nor the order; the
# reading taken: out = act(conv + bias) + residual, then one rounding to the
# output type.


def activation(v, act):
    """fp64 activation: identity, ReLU max(v, 0), or SiLU v * sigmoid(v)."""
    v = np.asarray(v, dtype=np.float64)
    if act == ACT_NONE:
        return v.copy()
    if act == ACT_RELU:
        return np.where(v > 0.0, v, 0.0)
    if act == ACT_SILU:
        # v / (1 + e^-v); for v < 0 written as v e^v / (1 + e^v) so that
        # e^-v cannot overflow
        e = np.exp(-np.abs(v))
        return np.where(v >= 0.0, v / (1.0 + e), v * e / (1.0 + e))
    raise ValueError("unknown activation %r" % (act,))


def epilogue(conv_out, act=ACT_NONE, residual=None):
    """act(conv_out) + residual in fp64; conv_out already holds the bias."""
    y = activation(conv_out, act)
    if residual is not None:
        y = y + np.asarray(residual, dtype=np.float64)
    return y


def _round_to_format(v, sig_bits, e_min, max_finite):
    """Round fp64 values to a binary format with `sig_bits` significant bits,
    nearest with ties to even: v = m * 2^e with 0.5 <= |m| < 1 keeps m to
    sig_bits bits, i.e. v becomes a multiple of 2^(e - sig_bits); below the
    format's smallest normal (e < e_min) the spacing stays 2^(e_min -
    sig_bits).  Results past max_finite become infinities."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    nz = (v != 0.0) & np.isfinite(v)
    _, e = np.frexp(v[nz])
    step = np.ldexp(1.0, np.maximum(e, e_min) - sig_bits)
    q = np.rint(v[nz] / step) * step  # rint: round half to even
    big = np.abs(q) > max_finite
    q[big] = np.copysign(np.inf, q[big])
    out[nz] = q
    out[~nz] = v[~nz]
    return out


def round_bf16(v):
    """Round fp64 values to bfloat16 (8 significant bits, fp32's exponent
    range: smallest normal 2^-126, so the spacing below it is 2^-133; largest
    finite 0x1.fep127), nearest with ties to even; returned as fp64."""
    return _round_to_format(v, 8, -125, float.fromhex("0x1.fep127"))


def round_f16(v):
    """Round fp64 values to IEEE binary16 (11 significant bits, smallest
    normal 2^-14 so subnormal spacing 2^-24, largest finite 65504), nearest
    with ties to even; returned as fp64."""
    return _round_to_format(v, 11, -13, 65504.0)
