"""CPU oracle for the convolution forward pass -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  It shares no code with the CUDA library: it has its
own C source (``conv_oracle.c``, plain loops, fp64 accumulation), its own shape
normalisation and its own build step.

Every function here follows the definition on the page "composable_kernel
dispatcher/heuristics/LEARNINGS_GROUPED_CONV.md" (introduction: NHWGC x GKYXC ->
NHWGK; section 2: 3D shapes and dilation) and the shapes and GELU placement on the
page "[ET-VK] conv1d runs at ~3% of the GPU's matmul throughput ..." (sections
"Measurements" and "The conv2d path already solves this").  The pins that tie it
to something other than itself live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc.  FP contraction is off so x86 and Arm hosts agree."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        lib.oracle_out_len.restype = ctypes.c_int64
        lib.oracle_out_len.argtypes = [ctypes.c_int64] * 5
        lib.oracle_conv_fwd.restype = ctypes.c_int
        lib.oracle_conv_fwd.argtypes = [P(ctypes.c_int64), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_conv_fwd_points.restype = ctypes.c_int
        lib.oracle_conv_fwd_points.argtypes = [P(ctypes.c_int64), ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                               ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        for name in ("oracle_conv_bwd_data", "oracle_conv_bwd_weight"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [P(ctypes.c_int64), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                           ctypes.c_int]
        lib.oracle_conv_bwd_points.restype = ctypes.c_int
        lib.oracle_conv_bwd_points.argtypes = [P(ctypes.c_int64), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                               ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_gelu.restype = None
        lib.oracle_gelu.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        _lib = lib
    return _lib


class Geom:
    """A problem in the 3-spatial form: conv1d is D = H = 1, conv2d is D = 1."""

    def __init__(self, N, G, C, K, spatial, filt, stride, pad, dilation):
        nd = len(spatial)
        assert nd in (1, 2, 3) and len(filt) == len(stride) == len(pad) == len(dilation) == nd
        lift = lambda v, one: (one,) * (3 - nd) + tuple(int(a) for a in v)
        self.N, self.G, self.C, self.K = int(N), int(G), int(C), int(K)
        self.ndim = nd
        self.spatial = lift(spatial, 1)
        self.filt = lift(filt, 1)
        self.stride = lift(stride, 1)
        self.pad = lift(pad, 0)
        self.dilation = lift(dilation, 1)
        self.out_spatial = tuple(out_len(i, f, s, p, d) for i, f, s, p, d in
                                 zip(self.spatial, self.filt, self.stride, self.pad, self.dilation))

    def params(self) -> np.ndarray:
        return np.array([self.N, self.G, self.C, self.K, *self.spatial, *self.filt,
                         *self.stride, *self.pad, *self.dilation], dtype=np.int64)

    # channels-last shapes in the 3-spatial form
    def x_shape(self):
        return (self.N, *self.spatial, self.G, self.C)

    def w_shape(self):
        return (self.G, self.K, *self.filt, self.C)

    def y_shape(self):
        return (self.N, *self.out_spatial, self.G, self.K)

    def macs(self) -> int:
        """Multiply-adds counted over every tap, padded ones included."""
        return int(np.prod(self.y_shape())) * self.C * int(np.prod(self.filt))


def out_len(i, f, s, p, d) -> int:
    return int(_load().oracle_out_len(int(i), int(f), int(s), int(p), int(d)))


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def conv_fwd(geom: Geom, x, w, bias=None, gelu=False, nthreads=None):
    """Whole output (float64) and S = sum |x*w| per output (float64), in N Do Ho Wo G K."""
    lib = _load()
    x = _f32(x).reshape(geom.x_shape())
    w = _f32(w).reshape(geom.w_shape())
    b = None if bias is None else _f32(bias).reshape(geom.G * geom.K)
    if min(geom.out_spatial) <= 0:
        raise ValueError("empty output")
    out = np.empty(geom.y_shape(), dtype=np.float64)
    absum = np.empty(geom.y_shape(), dtype=np.float64)
    nt = nthreads or os.cpu_count() or 1
    p = geom.params()
    rc = lib.oracle_conv_fwd(p.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), x.ctypes.data,
                             w.ctypes.data, None if b is None else b.ctypes.data, int(bool(gelu)),
                             out.ctypes.data, absum.ctypes.data, int(nt))
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    return out, absum


def conv_fwd_points(geom: Geom, x, w, bias, gelu, idx):
    """Outputs at idx (rows of n, od, oh, ow, g, k) and their S."""
    lib = _load()
    x = _f32(x).reshape(geom.x_shape())
    w = _f32(w).reshape(geom.w_shape())
    b = None if bias is None else _f32(bias).reshape(geom.G * geom.K)
    idx = np.ascontiguousarray(idx, dtype=np.int64).reshape(-1, 6)
    out = np.empty(len(idx), dtype=np.float64)
    absum = np.empty(len(idx), dtype=np.float64)
    p = geom.params()
    rc = lib.oracle_conv_fwd_points(p.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), x.ctypes.data,
                                    w.ctypes.data, None if b is None else b.ctypes.data, int(bool(gelu)),
                                    idx.ctypes.data, len(idx), out.ctypes.data, absum.ctypes.data)
    if rc != 0:
        raise ValueError("bad problem or index")
    return out, absum


def gelu(v):
    lib = _load()
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty_like(v)
    lib.oracle_gelu(v.ctypes.data, out.ctypes.data, v.size)
    return out


def conv_bwd_data(geom: Geom, dy, w, nthreads=None):
    """Gradient with respect to x (float64, N D H W G C) of the conv's linear part, given dy
    (N Do Ho Wo G K), and S = sum |dy*w| per element (page "composable_kernel
    dispatcher/heuristics/LEARNINGS_GROUPED_CONV.md", section 6: the bwd_data variant)."""
    lib = _load()
    dy = _f32(dy).reshape(geom.y_shape())
    w = _f32(w).reshape(geom.w_shape())
    if min(geom.out_spatial) <= 0:
        raise ValueError("empty output")
    out = np.empty(geom.x_shape(), dtype=np.float64)
    absum = np.empty(geom.x_shape(), dtype=np.float64)
    p = geom.params()
    rc = lib.oracle_conv_bwd_data(p.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), dy.ctypes.data, w.ctypes.data,
                                  out.ctypes.data, absum.ctypes.data, int(nthreads or os.cpu_count() or 1))
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    return out, absum


def conv_bwd_weight(geom: Geom, x, dy, nthreads=None):
    """Gradient with respect to w (float64, G K Z Y X C) given x and dy, and S = sum |dy*x|
    per element (same page, section 6: the bwd_weight variant)."""
    lib = _load()
    x = _f32(x).reshape(geom.x_shape())
    dy = _f32(dy).reshape(geom.y_shape())
    if min(geom.out_spatial) <= 0:
        raise ValueError("empty output")
    out = np.empty(geom.w_shape(), dtype=np.float64)
    absum = np.empty(geom.w_shape(), dtype=np.float64)
    p = geom.params()
    rc = lib.oracle_conv_bwd_weight(p.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), x.ctypes.data,
                                    dy.ctypes.data, out.ctypes.data, absum.ctypes.data,
                                    int(nthreads or os.cpu_count() or 1))
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    return out, absum


def conv_bwd_points(geom: Geom, a, b, weight: bool, idx):
    """Selected backward elements and their S.  weight=False: a = dy, b = w, idx rows of
    (n, d, h, w, g, c); weight=True: a = x, b = dy, idx rows of (g, k, z, y, x, c)."""
    lib = _load()
    if weight:
        a = _f32(a).reshape(geom.x_shape())
        b = _f32(b).reshape(geom.y_shape())
    else:
        a = _f32(a).reshape(geom.y_shape())
        b = _f32(b).reshape(geom.w_shape())
    idx = np.ascontiguousarray(idx, dtype=np.int64).reshape(-1, 6)
    out = np.empty(len(idx), dtype=np.float64)
    absum = np.empty(len(idx), dtype=np.float64)
    p = geom.params()
    rc = lib.oracle_conv_bwd_points(p.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), a.ctypes.data,
                                    b.ctypes.data, int(bool(weight)), idx.ctypes.data, len(idx), out.ctypes.data,
                                    absum.ctypes.data)
    if rc != 0:
        raise ValueError("bad problem or index")
    return out, absum
