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
    "SC_ACT_NONE", "SC_ACT_RELU", "SC_ACT_SILU", "sc_forward_ex", "sc_set_probe_limit",
    "sc_build_neighbor_table_noalloc", "sc_build_map_async", "sc_map_status",
    "LevelMap", "sc_subdivide", "sc_channel_to_spatial", "sc_build_level_map",
    "sc_level_parents", "sc_get_level_map", "sc_conv_down", "sc_conv_up",
    "sc_level_device_status", "sc_free_level_map", "sc_dual_mesh_quads",
    "sc_dual_mesh_triangulate", "sc_map_order_rows",
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
    lib.sc_build_map_async.argtypes = [P, I64, I32, I32, P]
    lib.sc_build_map_async.restype = P
    lib.sc_map_status.argtypes = [P]
    lib.sc_map_status.restype = ctypes.c_int
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
    lib.sc_set_probe_limit.argtypes = [I32]
    lib.sc_set_probe_limit.restype = ctypes.c_int
    lib.sc_build_neighbor_table_noalloc.argtypes = [P, I64, I32, P, P, P]
    lib.sc_build_neighbor_table_noalloc.restype = ctypes.c_int
    lib.sc_subdivide.argtypes = [P, P, I64, I32, P, P, P, P, P, P]
    lib.sc_subdivide.restype = ctypes.c_int
    lib.sc_channel_to_spatial.argtypes = [P, P, P, I64, I32, ctypes.c_int, P, P]
    lib.sc_channel_to_spatial.restype = ctypes.c_int
    lib.sc_build_level_map.argtypes = [P, I64, I32, I32, P]
    lib.sc_build_level_map.restype = P
    lib.sc_level_parents.argtypes = [P]
    lib.sc_level_parents.restype = I64
    lib.sc_get_level_map.argtypes = [P, P, P, P, P]
    lib.sc_get_level_map.restype = ctypes.c_int
    for name in ("sc_conv_down", "sc_conv_up"):
        getattr(lib, name).argtypes = [P, P, P, P, P, P, I32, I32, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, P]
        getattr(lib, name).restype = ctypes.c_int
    lib.sc_level_device_status.argtypes = [P, P]
    lib.sc_level_device_status.restype = ctypes.c_int
    lib.sc_free_level_map.argtypes = [P, P]
    lib.sc_free_level_map.restype = ctypes.c_int
    lib.sc_map_order_rows.argtypes = [P, P]
    lib.sc_map_order_rows.restype = ctypes.c_int
    lib.sc_dual_mesh_quads.argtypes = [P, P, P, P, P]
    lib.sc_dual_mesh_quads.restype = ctypes.c_int
    lib.sc_dual_mesh_triangulate.argtypes = [P, I64, P, P, P]
    lib.sc_dual_mesh_triangulate.restype = ctypes.c_int
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


def sc_set_probe_limit(limit: int) -> None:
    """Cap on one key's insertion probes, for testing the bounded probe loop
    (0 = the table's capacity; see sc_set_probe_limit in sc.h)."""
    _check(load_library().sc_set_probe_limit(int(limit)))


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


def sc_build_neighbor_table_noalloc(coords, res: int, out=None, stream=None):
    """int32 [N,27] neighbour table built without any device allocation by the
    library (static scratch; N <= 2^19); returns (table, pair count)."""
    import torch
    if coords.dtype != torch.int32 or coords.dim() != 2 or coords.shape[1] != 4:
        raise ValueError("coords must be int32 [N,4]")
    n = coords.shape[0]
    if out is None:
        out = torch.empty((n, 27), dtype=torch.int32, device=coords.device)
    elif out.dtype != torch.int32 or tuple(out.shape) != (n, 27):
        raise ValueError("out must be int32 [N, 27]")
    pairs = ctypes.c_int64(0)
    _check(load_library().sc_build_neighbor_table_noalloc(
        _dev_ptr(coords, "coords"), n, int(res), _dev_ptr(out, "out"), ctypes.byref(pairs),
        _stream_ptr(stream)))
    return out, int(pairs.value)


def sc_build_map_async(coords, res: int, nbatch: int, stream=None) -> Map:
    """sc_build_map without a host synchronisation; batch indices must lie in
    [0, nbatch).  Device-found errors surface at sc_map_status / pairs."""
    import torch
    if coords.dtype != torch.int32 or coords.dim() != 2 or coords.shape[1] != 4:
        raise ValueError("coords must be int32 [N,4]")
    lib = load_library()
    ptr = lib.sc_build_map_async(_dev_ptr(coords, "coords"), coords.shape[0], int(res),
                                 int(nbatch), _stream_ptr(stream))
    if not ptr:
        raise ScError(sc_last_error(), sc_last_error_msg())
    return Map(ptr, int(coords.shape[0]), int(res), coords.device)


def sc_map_status(m: Map) -> None:
    """Wait for the map's build and raise its error, if any."""
    _check(load_library().sc_map_status(ctypes.c_void_p(m.ptr)))


def sc_map_order_rows(m: Map, stream=None) -> None:
    """Sort the map's rows by neighbour mask for the convolutions that follow
    (outputs still land in their own rows)."""
    _check(load_library().sc_map_order_rows(ctypes.c_void_p(m.ptr), _stream_ptr(stream)))


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


# ---------------------------------------------------------------------------
# level changes


class LevelMap:
    """A level map built by sc_build_level_map (owns its device memory)."""

    def __init__(self, ptr: int, n: int, np_: int, device):
        self.ptr = ptr
        self.n = n
        self.parents = np_
        self.device = device

    def free(self, stream=None):
        if self.ptr:
            sc_free_level_map(self, stream)

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


def _coords_arg(coords):
    import torch
    if coords.dtype != torch.int32 or coords.dim() != 2 or coords.shape[1] != 4:
        raise ValueError("coords must be int32 [N,4]")
    return _dev_ptr(coords, "coords")


def sc_subdivide(coords, res: int, mask=None, stream=None):
    """Children of each voxel under an 8-bit mask (None: all 8).  Returns
    (child_coords int32 [M,4], parent int32 [M], offset int32 [M], child_of
    int32 [N,8]) on the device."""
    import torch
    cp = _coords_arg(coords)
    n = coords.shape[0]
    if mask is not None and (mask.dtype != torch.uint8 or mask.numel() != n):
        raise ValueError("mask must be uint8 [N]")
    dev = coords.device
    cap = max(8 * n, 1)
    child = torch.empty((cap, 4), dtype=torch.int32, device=dev)
    parent = torch.empty(cap, dtype=torch.int32, device=dev)
    offset = torch.empty(cap, dtype=torch.int32, device=dev)
    child_of = torch.empty((max(n, 1), 8), dtype=torch.int32, device=dev)
    m = ctypes.c_int64(0)
    _check(load_library().sc_subdivide(cp, _dev_ptr(mask, "mask"), n, int(res),
                                       _dev_ptr(child, "child_coords"), _dev_ptr(parent, "parent"),
                                       _dev_ptr(offset, "offset"), _dev_ptr(child_of, "child_of"),
                                       ctypes.byref(m), _stream_ptr(stream)))
    M = int(m.value)
    return child[:M], parent[:M], offset[:M], child_of[:n]


def sc_channel_to_spatial(feats, parent, offset, stream=None):
    """Channel2Spatial: child (parent i, offset o) takes channels c*8 + o of
    feats[i] (feats [N, 8C]); returns [M, C] in feats' dtype."""
    import torch
    n, c8 = feats.shape
    if c8 % 8:
        raise ValueError("feats must have 8C channels")
    m = parent.numel()
    out = torch.empty((m, c8 // 8), dtype=feats.dtype, device=feats.device)
    _check(load_library().sc_channel_to_spatial(
        _dev_ptr(feats, "feats"), _dev_ptr(parent, "parent"), _dev_ptr(offset, "offset"), m,
        c8 // 8, _operand_dtype(feats), _dev_ptr(out, "out"), _stream_ptr(stream)))
    return out


def sc_build_level_map(coords, res: int, nbatch: int = 1, stream=None) -> LevelMap:
    """Parents (b, x>>1, y>>1, z>>1) of fine voxels, in (b,x,y,z) order, with
    their child tables; drives sc_conv_down / sc_conv_up."""
    lib = load_library()
    ptr = lib.sc_build_level_map(_coords_arg(coords), coords.shape[0], int(res), int(nbatch),
                                 _stream_ptr(stream))
    if not ptr:
        raise ScError(sc_last_error(), sc_last_error_msg())
    np_ = int(lib.sc_level_parents(ctypes.c_void_p(ptr)))
    return LevelMap(ptr, int(coords.shape[0]), np_, coords.device)


def sc_level_parents(lm: LevelMap) -> int:
    v = load_library().sc_level_parents(ctypes.c_void_p(lm.ptr))
    if v < 0:
        raise ScError(sc_last_error(), sc_last_error_msg())
    return int(v)


def sc_get_level_map(lm: LevelMap, stream=None):
    """(parent_coords int32 [P,4], child_of int32 [P,8], parent_of int32 [N])."""
    import torch
    P = lm.parents
    pc = torch.empty((max(P, 1), 4), dtype=torch.int32, device=lm.device)
    co = torch.empty((max(P, 1), 8), dtype=torch.int32, device=lm.device)
    po = torch.empty(max(lm.n, 1), dtype=torch.int32, device=lm.device)
    _check(load_library().sc_get_level_map(ctypes.c_void_p(lm.ptr), _dev_ptr(pc, "pc"),
                                           _dev_ptr(co, "co"), _dev_ptr(po, "po"),
                                           _stream_ptr(stream)))
    return pc[:P], co[:P], po[:lm.n]


def _level_conv(fn, lm, feats, weight, bias, residual, act, out_dtype, out, n_out, stream):
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
    cin = feats.shape[1]
    if weight.dim() != 3 or weight.shape[0] != 8 or weight.shape[1] != cin:
        raise ValueError("weight must be [8, cin, cout]")
    cout = weight.shape[2]
    if bias is not None and (bias.dtype != torch.float32 or bias.numel() != cout):
        raise ValueError("bias must be fp32 [cout]")
    if residual is not None and (residual.dtype != out_dtype or
                                 tuple(residual.shape) != (n_out, cout)):
        raise ValueError("residual must be [rows, cout] in out_dtype")
    if out is None:
        out = torch.empty((n_out, cout), dtype=out_dtype, device=feats.device)
    rc = fn(ctypes.c_void_p(lm.ptr), _dev_ptr(feats, "feats"), _dev_ptr(weight, "weight"),
            _dev_ptr(bias, "bias"), _dev_ptr(residual, "residual"), _dev_ptr(out, "out"), cin,
            cout, dt, _ACTS[act], odts[out_dtype], _stream_ptr(stream))
    _check(rc)
    return out


def sc_conv_down(lm: LevelMap, feats, weight, bias=None, residual=None, act="none",
                 out_dtype=None, out=None, stream=None):
    """2x2x2 stride-2 convolution to the parents: feats [N, cin] -> [P, cout]."""
    if feats.shape[0] != lm.n:
        raise ValueError("feats has %d rows, the level map %d fine rows" % (feats.shape[0], lm.n))
    return _level_conv(load_library().sc_conv_down, lm, feats, weight, bias, residual, act,
                       out_dtype, out, lm.parents, stream)


def sc_conv_up(lm: LevelMap, feats, weight, bias=None, residual=None, act="none",
               out_dtype=None, out=None, stream=None):
    """Its transpose: parent feats [P, cin] -> fine [N, cout]."""
    if feats.shape[0] != lm.parents:
        raise ValueError("feats has %d rows, the level map %d parents" % (feats.shape[0],
                                                                          lm.parents))
    return _level_conv(load_library().sc_conv_up, lm, feats, weight, bias, residual, act,
                       out_dtype, out, lm.n, stream)


def sc_level_device_status(lm: LevelMap, stream=None):
    _check(load_library().sc_level_device_status(ctypes.c_void_p(lm.ptr), _stream_ptr(stream)))


def sc_free_level_map(lm: LevelMap, stream=None):
    rc = load_library().sc_free_level_map(ctypes.c_void_p(lm.ptr), _stream_ptr(stream))
    lm.ptr = 0
    _check(rc)


# ---------------------------------------------------------------------------
# dual-grid mesh


def sc_dual_mesh_quads(m: Map, flags, stream=None):
    """int32 [Q,4] voxel rows of the quads of the map's flagged edges
    (flags uint8 [N], 6 bits per voxel)."""
    import torch
    if flags.dtype != torch.uint8 or flags.numel() != m.n:
        raise ValueError("flags must be uint8 [N]")
    quads = torch.empty((max(3 * m.n, 1), 4), dtype=torch.int32, device=m.device)
    q = ctypes.c_int64(0)
    _check(load_library().sc_dual_mesh_quads(ctypes.c_void_p(m.ptr), _dev_ptr(flags, "flags"),
                                             _dev_ptr(quads, "quads"), ctypes.byref(q),
                                             _stream_ptr(stream)))
    return quads[:int(q.value)]


def sc_dual_mesh_triangulate(quads, vertices, stream=None):
    """int32 [2Q,3] triangles of quads [Q,4] over fp32 vertices [N,3]."""
    import torch
    if vertices.dtype != torch.float32 or vertices.dim() != 2 or vertices.shape[1] != 3:
        raise ValueError("vertices must be fp32 [N,3]")
    nq = quads.shape[0]
    tris = torch.empty((max(2 * nq, 1), 3), dtype=torch.int32, device=quads.device)
    _check(load_library().sc_dual_mesh_triangulate(_dev_ptr(quads, "quads"), nq,
                                                   _dev_ptr(vertices, "vertices"),
                                                   _dev_ptr(tris, "tris"), _stream_ptr(stream)))
    return tris[:2 * nq]
