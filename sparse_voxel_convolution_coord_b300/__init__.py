"""B300 (sm_103a) 3x3x3 submanifold sparse convolution.

A thin ctypes binding over ``libsc.so`` (C ABI in ``include/sc.h``).  The
functions keep the C names and only marshal arguments: torch tensors supply
device pointers and the current CUDA stream; every step of the method runs in
the library's CUDA kernels.  There is no CPU fallback: if the library is
missing or no CUDA device is present, calls raise.

    coords : int32 [N,4] (batch, x, y, z) on the GPU
    m = sc_build_map(coords, res)                 # hash + neighbour map
    out = sc_forward(m, feats, weight, bias)      # bf16 or fp32 feats/weight
    sc_free_map(m)
"""
from __future__ import annotations

import ctypes
import os
import re

__all__ = [
    "ScError", "Map", "load_library", "library_path", "header_symbols",
    "sc_build_map", "sc_forward", "sc_free_map", "sc_map_size", "sc_map_pairs",
    "sc_get_neighbor_table", "sc_get_pairs", "sc_device_status", "sc_last_error",
    "sc_last_error_msg", "sc_version", "sc_set_deterministic", "sc_kernel_launches", "sc_release_cached_memory", "SC_OK", "SC_ERR_INVALID_ARG", "SC_ERR_COORD_RANGE",
    "SC_ERR_DUPLICATE", "SC_ERR_TABLE_FULL", "SC_ERR_UNSUPPORTED", "SC_ERR_ALLOC",
    "SC_ERR_CUDA", "SC_ERR_BAD_HANDLE", "SC_ERR_DEVICE_TIMEOUT", "SC_F32", "SC_BF16", "SC_F16",
    "SC_ACT_NONE", "SC_ACT_RELU", "SC_ACT_SILU", "sc_forward_ex",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
HEADER = os.path.join(_ROOT, "include", "sc.h")

(SC_OK, SC_ERR_INVALID_ARG, SC_ERR_COORD_RANGE, SC_ERR_DUPLICATE, SC_ERR_TABLE_FULL,
 SC_ERR_UNSUPPORTED, SC_ERR_ALLOC, SC_ERR_CUDA, SC_ERR_BAD_HANDLE,
 SC_ERR_DEVICE_TIMEOUT) = range(10)
SC_F32, SC_BF16, SC_F16 = 0, 1, 2
SC_ACT_NONE, SC_ACT_RELU, SC_ACT_SILU = 0, 1, 2
_ACTS = {"none": SC_ACT_NONE, "relu": SC_ACT_RELU, "silu": SC_ACT_SILU}

_lib = None


class ScError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("sc error %d: %s" % (code, msg))
        self.code = code


def library_path() -> str:
    return os.path.join(_HERE, "libsc.so")


def header_symbols():
    """Names of the functions include/sc.h declares."""
    text = open(HEADER).read()
    return re.findall(r"SC_API\s+[\w\s\*]+?\b(sc_\w+)\s*\(", text)


def load_library():
    """Load libsc.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError("libsc.so is not built (%s); run "
                           "python -m sparse_voxel_convolution_coord_b300.build_lib" % path)
    lib = ctypes.CDLL(path)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.sc_build_map.argtypes = [P, I64, I32, P]
    lib.sc_build_map.restype = P
    lib.sc_forward.argtypes = [P, P, P, P, P, I32, I32, ctypes.c_int, P]
    lib.sc_forward.restype = ctypes.c_int
    lib.sc_forward_ex.argtypes = [P, P, P, P, P, P, I32, I32, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, P]
    lib.sc_forward_ex.restype = ctypes.c_int
    lib.sc_free_map.argtypes = [P, P]
    lib.sc_free_map.restype = ctypes.c_int
    lib.sc_map_size.argtypes = [P]
    lib.sc_map_size.restype = I64
    lib.sc_map_pairs.argtypes = [P]
    lib.sc_map_pairs.restype = I64
    lib.sc_get_neighbor_table.argtypes = [P, P, P]
    lib.sc_get_neighbor_table.restype = ctypes.c_int
    lib.sc_get_pairs.argtypes = [P, P, P, P, P]
    lib.sc_get_pairs.restype = ctypes.c_int
    lib.sc_device_status.argtypes = [P, P]
    lib.sc_device_status.restype = ctypes.c_int
    lib.sc_last_error.restype = ctypes.c_int
    lib.sc_last_error_msg.restype = ctypes.c_char_p
    lib.sc_version.restype = ctypes.c_char_p
    lib.sc_set_deterministic.argtypes = [I32]
    lib.sc_set_deterministic.restype = ctypes.c_int
    lib.sc_kernel_launches.restype = ctypes.c_uint64
    lib.sc_release_cached_memory.restype = ctypes.c_int
    _lib = lib
    return lib


def sc_last_error() -> int:
    return int(load_library().sc_last_error())


def sc_last_error_msg() -> str:
    return load_library().sc_last_error_msg().decode()


def sc_version() -> str:
    return load_library().sc_version().decode()


def sc_kernel_launches() -> int:
    """Kernels the library has launched in this process (see sc.h)."""
    return int(load_library().sc_kernel_launches())


def sc_release_cached_memory() -> None:
    """Return the library pool's cached (freed) map memory to the device."""
    _check(load_library().sc_release_cached_memory())


def sc_set_deterministic(enable: bool) -> None:
    """Bit-identical repeated forwards (see sc_set_deterministic in sc.h)."""
    _check(load_library().sc_set_deterministic(1 if enable else 0))


def _check(rc: int):
    if rc != SC_OK:
        raise ScError(rc, sc_last_error_msg())


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_ptr(t, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


class Map:
    """A neighbour map built by sc_build_map (owns its device memory)."""

    def __init__(self, ptr: int, n: int, res: int, device):
        self.ptr = ptr
        self.n = n
        self.res = res
        self.device = device

    @property
    def pairs(self) -> int:
        return sc_map_pairs(self)

    def free(self, stream=None):
        if self.ptr:
            sc_free_map(self, stream)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.free()

    def __del__(self):
        try:
            if self.ptr:
                self.free()
        except Exception:
            pass


def sc_build_map(coords, res: int, stream=None) -> Map:
    """Hash table + neighbour map of int32 coords [N,4] (batch,x,y,z) on the GPU."""
    import torch
    if coords.dtype != torch.int32 or coords.dim() != 2 or coords.shape[1] != 4:
        raise ValueError("coords must be int32 [N,4]")
    lib = load_library()
    ptr = lib.sc_build_map(_dev_ptr(coords, "coords"), coords.shape[0], int(res),
                           _stream_ptr(stream))
    if not ptr:
        raise ScError(sc_last_error(), sc_last_error_msg())
    return Map(ptr, int(coords.shape[0]), int(res), coords.device)


def sc_free_map(m: Map, stream=None):
    lib = load_library()
    rc = lib.sc_free_map(ctypes.c_void_p(m.ptr), _stream_ptr(stream))
    m.ptr = 0
    _check(rc)


def sc_map_size(m: Map) -> int:
    v = load_library().sc_map_size(ctypes.c_void_p(m.ptr))
    if v < 0:
        raise ScError(sc_last_error(), sc_last_error_msg())
    return int(v)


def sc_map_pairs(m: Map) -> int:
    v = load_library().sc_map_pairs(ctypes.c_void_p(m.ptr))
    if v < 0:
        raise ScError(sc_last_error(), sc_last_error_msg())
    return int(v)


def _operand_dtype(feats):
    import torch
    codes = {torch.bfloat16: SC_BF16, torch.float16: SC_F16, torch.float32: SC_F32}
    if feats.dtype not in codes:
        raise ValueError("dtype must be bfloat16, float16 or float32")
    return codes[feats.dtype]


def sc_forward(m: Map, feats, weight, bias=None, out=None, stream=None):
    """out[N,cout] fp32 = bias + sum_k gather(feats, nbr[:,k]) @ weight[k].

    feats [N,cin] and weight [27,cin,cout] are both bf16 or both fp16
    (tensor-core path), or both fp32 (FFMA path); bias fp32 [cout] or None.
    Asynchronous.
    """
    import torch
    if feats.dtype != weight.dtype:
        raise ValueError("feats and weight must have the same dtype")
    dt = _operand_dtype(feats)
    n, cin = feats.shape
    if weight.dim() != 3 or weight.shape[0] != 27 or weight.shape[1] != cin:
        raise ValueError("weight must be [27, cin, cout]")
    cout = weight.shape[2]
    if n != m.n:
        raise ValueError("feats has %d rows, the map %d" % (n, m.n))
    if bias is not None and (bias.dtype != torch.float32 or bias.numel() != cout):
        raise ValueError("bias must be fp32 [cout]")
    if out is None:
        out = torch.empty((n, cout), dtype=torch.float32, device=feats.device)
    rc = load_library().sc_forward(ctypes.c_void_p(m.ptr), _dev_ptr(feats, "feats"),
                                   _dev_ptr(weight, "weight"), _dev_ptr(bias, "bias"),
                                   _dev_ptr(out, "out"), cin, cout, dt, _stream_ptr(stream))
    _check(rc)
    return out


def sc_forward_ex(m: Map, feats, weight, bias=None, residual=None, act="none",
                  out_dtype=None, out=None, stream=None):
    """Convolution with the fused epilogue: out = act(conv + bias) + residual.

    act is "none", "relu" or "silu"; out_dtype torch.float32 (default),
    torch.bfloat16 or torch.float16; residual [N,cout] in out_dtype or None.
    Asynchronous.
    """
    import torch
    if feats.dtype != weight.dtype:
        raise ValueError("feats and weight must have the same dtype")
    dt = _operand_dtype(feats)
    if act not in _ACTS:
        raise ValueError("act must be one of %s" % sorted(_ACTS))
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    odts = {torch.float32: SC_F32, torch.bfloat16: SC_BF16, torch.float16: SC_F16}
    if out_dtype not in odts:
        raise ValueError("out_dtype must be float32, bfloat16 or float16")
    odt = odts[out_dtype]
    n, cin = feats.shape
    if weight.dim() != 3 or weight.shape[0] != 27 or weight.shape[1] != cin:
        raise ValueError("weight must be [27, cin, cout]")
    cout = weight.shape[2]
    if n != m.n:
        raise ValueError("feats has %d rows, the map %d" % (n, m.n))
    if bias is not None and (bias.dtype != torch.float32 or bias.numel() != cout):
        raise ValueError("bias must be fp32 [cout]")
    if residual is not None and (residual.dtype != out_dtype or tuple(residual.shape) != (n, cout)):
        raise ValueError("residual must be [N, cout] in out_dtype")
    if out is None:
        out = torch.empty((n, cout), dtype=out_dtype, device=feats.device)
    elif out.dtype != out_dtype or tuple(out.shape) != (n, cout):
        raise ValueError("out must be [N, cout] in out_dtype")
    rc = load_library().sc_forward_ex(
        ctypes.c_void_p(m.ptr), _dev_ptr(feats, "feats"), _dev_ptr(weight, "weight"),
        _dev_ptr(bias, "bias"), _dev_ptr(residual, "residual"), _dev_ptr(out, "out"), cin, cout,
        dt, _ACTS[act], odt, _stream_ptr(stream))
    _check(rc)
    return out


def sc_get_neighbor_table(m: Map, out=None, stream=None):
    """int32 [N,27] neighbour table (device)."""
    import torch
    if out is None:
        out = torch.empty((m.n, 27), dtype=torch.int32, device=m.device)
    _check(load_library().sc_get_neighbor_table(ctypes.c_void_p(m.ptr), _dev_ptr(out, "out"),
                                                _stream_ptr(stream)))
    return out


def sc_get_pairs(m: Map, stream=None):
    """CSR pair lists: (off int64 [28] host tensor, in int32 [P], out int32 [P] device)."""
    import torch
    p = sc_map_pairs(m)
    off = torch.empty(28, dtype=torch.int64)
    pin = torch.empty(max(p, 1), dtype=torch.int32, device=m.device)
    pout = torch.empty(max(p, 1), dtype=torch.int32, device=m.device)
    _check(load_library().sc_get_pairs(ctypes.c_void_p(m.ptr), ctypes.c_void_p(off.data_ptr()),
                                       _dev_ptr(pin, "in"), _dev_ptr(pout, "out"),
                                       _stream_ptr(stream)))
    return off, pin[:p], pout[:p]


def sc_device_status(m: Map, stream=None):
    """Synchronise and raise if a kernel over this map recorded a device error."""
    _check(load_library().sc_device_status(ctypes.c_void_p(m.ptr), _stream_ptr(stream)))
