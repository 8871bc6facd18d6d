"""ctypes binding of ``libconvfwd.so`` (declared in include/conv.h).

The functions carry the C-ABI names and only marshal arguments: device pointers are
passed as integers (``tensor.data_ptr()``), streams as ``cudaStream_t`` integers
(``torch.cuda.current_stream().cuda_stream``).  A non-OK status raises ``ConvError``.
``ConvPlan`` wraps one plan and uses PyTorch only to allocate the packed weights and
the workspace; the arithmetic of every step runs in the library's kernels.

There is no fallback: if the library is missing or cannot be loaded, the first call
raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "ConvError", "CONV_OK", "CONV_ERR_INVALID_ARG", "CONV_ERR_UNSUPPORTED", "CONV_ERR_ALIGNMENT",
    "CONV_ERR_WORKSPACE", "CONV_ERR_CUDA", "CONV_ERR_TIMEOUT", "CONV_F32", "CONV_BF16", "CONV_EPI_NONE",
    "CONV_EPI_BIAS", "CONV_EPI_BIAS_GELU", "CONV_EPI_GELU", "library_path", "load_library",
    "conv_plan_create", "conv_plan_output_shape", "conv_prepacked_weight_bytes", "conv_workspace_bytes",
    "conv_plan_set_workspace", "conv_prepack_weights", "conv_fwd", "conv_plan_check", "conv_plan_destroy",
    "conv_status_string", "conv_plan_describe", "conv_plan_flops", "ConvPlan", "EXPORTED",
    "conv_fwd_static_scratch", "conv_static_scratch_bytes", "conv_plan_set_overlap",
]

CONV_OK, CONV_ERR_INVALID_ARG, CONV_ERR_UNSUPPORTED, CONV_ERR_ALIGNMENT = 0, 1, 2, 3
CONV_ERR_WORKSPACE, CONV_ERR_CUDA, CONV_ERR_TIMEOUT = 4, 5, 6
CONV_F32, CONV_BF16 = 0, 1
CONV_EPI_NONE, CONV_EPI_BIAS, CONV_EPI_BIAS_GELU, CONV_EPI_GELU = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None

_I64P = ctypes.POINTER(ctypes.c_int64)
_VP = ctypes.c_void_p
_SIGS = {
    "conv_plan_create": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, _I64P, _I64P, _I64P, _I64P, _I64P,
                                        ctypes.c_int, ctypes.c_int]),
    "conv_plan_output_shape": (ctypes.c_int, [_VP, _I64P]),
    "conv_prepacked_weight_bytes": (ctypes.c_size_t, [_VP]),
    "conv_workspace_bytes": (ctypes.c_size_t, [_VP]),
    "conv_plan_set_workspace": (ctypes.c_int, [_VP, _VP, ctypes.c_size_t]),
    "conv_prepack_weights": (ctypes.c_int, [_VP, _VP, _VP, _VP]),
    "conv_fwd": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP]),
    "conv_plan_check": (ctypes.c_int, [_VP, _VP]),
    "conv_plan_destroy": (ctypes.c_int, [_VP]),
    "conv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "conv_plan_describe": (ctypes.c_char_p, [_VP]),
    "conv_plan_flops": (ctypes.c_double, [_VP]),
    "conv_fwd_static_scratch": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP]),
    "conv_static_scratch_bytes": (ctypes.c_size_t, []),
    "conv_plan_set_overlap": (ctypes.c_int, [_VP, ctypes.c_int]),
    "conv_bwd_data_plan_create": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.c_int64, ctypes.c_int64, _I64P, _I64P, _I64P, _I64P, _I64P,
                                                 ctypes.c_int]),
    "conv_bwd_data": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP]),
    "conv_bwd_weight_plan_create": (ctypes.c_int, [ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_int64,
                                                   ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _I64P, _I64P,
                                                   _I64P, _I64P, _I64P, ctypes.c_int]),
    "conv_bwd_weight": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP]),
    "conv_tune_scratch_bytes": (ctypes.c_size_t, [_VP]),
    "conv_plan_tune": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, ctypes.c_int, _VP]),
    "conv_tune_table_save": (ctypes.c_int, [ctypes.c_char_p]),
    "conv_tune_table_load": (ctypes.c_int, [ctypes.c_char_p]),
    "conv_tune_table_clear": (ctypes.c_int, []),
}
EXPORTED = tuple(_SIGS)


class ConvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {conv_status_string(status)}")


def library_path() -> str:
    return os.environ.get("CONVFWD_LIBRARY", os.path.join(_HERE, "libconvfwd.so"))


def load_library():
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"libconvfwd.so not built ({path}); run __graft_entry__.build() "
                                   "or python -m convolution_forward_implicit_gb300.build")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(st: int, what: str):
    if st != CONV_OK:
        raise ConvError(st, what)


def _arr(v):
    v = [int(a) for a in v]
    return (ctypes.c_int64 * len(v))(*v)


def conv_status_string(status: int) -> str:
    return load_library().conv_status_string(int(status)).decode()


def conv_plan_create(ndim, N, G, C, K, spatial, filter, stride, pad, dilation, dtype, epilogue) -> int:
    h = _VP()
    st = load_library().conv_plan_create(ctypes.byref(h), int(ndim), int(N), int(G), int(C), int(K),
                                         _arr(spatial), _arr(filter), _arr(stride), _arr(pad), _arr(dilation),
                                         int(dtype), int(epilogue))
    _check(st, "conv_plan_create")
    return h.value


def conv_bwd_data_plan_create(ndim, N, G, C, K, spatial, filter, stride, pad, dilation, dtype) -> int:
    h = _VP()
    st = load_library().conv_bwd_data_plan_create(ctypes.byref(h), int(ndim), int(N), int(G), int(C), int(K),
                                                  _arr(spatial), _arr(filter), _arr(stride), _arr(pad),
                                                  _arr(dilation), int(dtype))
    _check(st, "conv_bwd_data_plan_create")
    return h.value


def conv_bwd_weight_plan_create(ndim, N, G, C, K, spatial, filter, stride, pad, dilation, dtype) -> int:
    h = _VP()
    st = load_library().conv_bwd_weight_plan_create(ctypes.byref(h), int(ndim), int(N), int(G), int(C), int(K),
                                                    _arr(spatial), _arr(filter), _arr(stride), _arr(pad),
                                                    _arr(dilation), int(dtype))
    _check(st, "conv_bwd_weight_plan_create")
    return h.value


def conv_bwd_data(plan: int, dy_ptr: int, w_packed_ptr: int, dx_ptr: int, stream: int = 0):
    _check(load_library().conv_bwd_data(plan, dy_ptr, w_packed_ptr, dx_ptr, stream or None), "conv_bwd_data")


def conv_bwd_weight(plan: int, x_ptr: int, dy_ptr: int, dw_ptr: int, stream: int = 0):
    _check(load_library().conv_bwd_weight(plan, x_ptr, dy_ptr, dw_ptr, stream or None), "conv_bwd_weight")


def conv_plan_output_shape(plan: int, ndim: int):
    out = (ctypes.c_int64 * ndim)()
    _check(load_library().conv_plan_output_shape(plan, out), "conv_plan_output_shape")
    return tuple(int(v) for v in out)


def conv_prepacked_weight_bytes(plan: int) -> int:
    return int(load_library().conv_prepacked_weight_bytes(plan))


def conv_workspace_bytes(plan: int) -> int:
    return int(load_library().conv_workspace_bytes(plan))


def conv_plan_set_workspace(plan: int, ptr: int, nbytes: int):
    _check(load_library().conv_plan_set_workspace(plan, ptr or None, int(nbytes)), "conv_plan_set_workspace")


def conv_prepack_weights(plan: int, w_ptr: int, w_packed_ptr: int, stream: int = 0):
    _check(load_library().conv_prepack_weights(plan, w_ptr, w_packed_ptr, stream or None), "conv_prepack_weights")


def conv_fwd(plan: int, x_ptr: int, w_packed_ptr: int, bias_ptr: int, y_ptr: int, stream: int = 0):
    _check(load_library().conv_fwd(plan, x_ptr, w_packed_ptr, bias_ptr or None, y_ptr, stream or None),
           "conv_fwd")


def conv_fwd_static_scratch(plan: int, x_ptr: int, w_packed_ptr: int, bias_ptr: int, y_ptr: int, stream: int = 0):
    """conv_fwd for callers that cannot allocate: split-K scratch lives in the library's
    own device array (conv_static_scratch_bytes() of them); see include/conv.h."""
    _check(load_library().conv_fwd_static_scratch(plan, x_ptr, w_packed_ptr, bias_ptr or None, y_ptr,
                                                  stream or None), "conv_fwd_static_scratch")


def conv_static_scratch_bytes() -> int:
    """Size in bytes of the library's own device array that conv_fwd_static_scratch uses."""
    return int(load_library().conv_static_scratch_bytes())


def conv_plan_check(plan: int, stream: int = 0):
    _check(load_library().conv_plan_check(plan, stream or None), "conv_plan_check")


def conv_plan_destroy(plan: int):
    _check(load_library().conv_plan_destroy(plan), "conv_plan_destroy")


def conv_plan_set_overlap(plan: int, enable: bool = True):
    """Launch this plan's kernels as programmatic dependents of the previous kernel on the
    stream (see include/conv.h): set-up and packed-weight loads overlap the previous layer."""
    _check(load_library().conv_plan_set_overlap(plan, 1 if enable else 0), "conv_plan_set_overlap")


def conv_tune_scratch_bytes(plan: int) -> int:
    return int(load_library().conv_tune_scratch_bytes(plan))


def conv_plan_tune(plan: int, x_ptr: int, w_ptr: int, bias_ptr: int, y_ptr: int, scratch_ptr: int,
                   scratch_bytes: int, iters: int = 10, stream: int = 0):
    """Time the candidate plans of this problem and switch the plan to the fastest (see
    include/conv.h); afterwards the packed weight and workspace must be re-made."""
    _check(load_library().conv_plan_tune(plan, x_ptr, w_ptr, bias_ptr or None, y_ptr, scratch_ptr,
                                         int(scratch_bytes), int(iters), stream or None), "conv_plan_tune")


def conv_tune_table_save(path: str):
    _check(load_library().conv_tune_table_save(os.fsencode(path)), "conv_tune_table_save")


def conv_tune_table_load(path: str):
    _check(load_library().conv_tune_table_load(os.fsencode(path)), "conv_tune_table_load")


def conv_tune_table_clear():
    _check(load_library().conv_tune_table_clear(), "conv_tune_table_clear")


def conv_plan_describe(plan: int) -> str:
    return load_library().conv_plan_describe(plan).decode()


def conv_plan_flops(plan: int) -> float:
    return float(load_library().conv_plan_flops(plan))


class ConvPlan:
    """One plan plus the device buffers it needs (packed weights, workspace), allocated
    with PyTorch on the current device.  Tensors are channels-last, dtype float32 or
    bfloat16 matching the plan.  direction: "fwd" (conv_fwd), "bwd_data" (conv_bwd_data)
    or "bwd_weight" (conv_bwd_weight); the backward plans take the forward problem's
    description and ignore the epilogue."""

    def __init__(self, ndim, N, G, C, K, spatial, filter, stride, pad, dilation, dtype, epilogue,
                 direction="fwd"):
        self.ndim, self.N, self.G, self.C, self.K = int(ndim), int(N), int(G), int(C), int(K)
        self.dtype, self.epilogue, self.direction = int(dtype), int(epilogue), direction
        if direction == "fwd":
            self.handle = conv_plan_create(ndim, N, G, C, K, spatial, filter, stride, pad, dilation, dtype, epilogue)
        elif direction == "bwd_data":
            self.handle = conv_bwd_data_plan_create(ndim, N, G, C, K, spatial, filter, stride, pad, dilation, dtype)
        elif direction == "bwd_weight":
            self.handle = conv_bwd_weight_plan_create(ndim, N, G, C, K, spatial, filter, stride, pad, dilation,
                                                      dtype)
        else:
            raise ValueError(f"unknown direction {direction!r}")
        self.spatial = tuple(int(v) for v in spatial)
        self.filter = tuple(int(v) for v in filter)
        self.out_spatial = conv_plan_output_shape(self.handle, self.ndim)
        self.workspace = None
        self.w_packed = None

    # shapes in the caller's ndim form
    def x_shape(self):
        return (self.N, *self.spatial, self.G, self.C)

    def w_shape(self):
        return (self.G, self.K, *self.filter, self.C)

    def y_shape(self):
        return (self.N, *self.out_spatial, self.G, self.K)

    @property
    def flops(self) -> float:
        return conv_plan_flops(self.handle)

    def describe(self) -> str:
        return conv_plan_describe(self.handle)

    def torch_dtype(self):
        import torch
        return torch.bfloat16 if self.dtype == CONV_BF16 else torch.float32

    def allocate(self, device=None):
        """Allocate the packed-weight buffer and (if needed) the workspace."""
        import torch
        dev = device or torch.device("cuda", torch.cuda.current_device())
        self.w_packed = torch.empty(max(conv_prepacked_weight_bytes(self.handle), 16), dtype=torch.uint8,
                                    device=dev)
        nws = conv_workspace_bytes(self.handle)
        if nws:
            self.workspace = torch.empty(nws, dtype=torch.uint8, device=dev)
            conv_plan_set_workspace(self.handle, self.workspace.data_ptr(), nws)
        return self

    def prepack(self, w, stream=None):
        import torch
        if self.w_packed is None:
            self.allocate(w.device)
        s = stream if stream is not None else torch.cuda.current_stream(w.device).cuda_stream
        conv_prepack_weights(self.handle, w.data_ptr(), self.w_packed.data_ptr(), s)
        return self.w_packed

    def forward(self, x, bias, y, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        conv_fwd(self.handle, x.data_ptr(), self.w_packed.data_ptr(), 0 if bias is None else bias.data_ptr(),
                 y.data_ptr(), s)
        return y

    def backward_data(self, dy, dx, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(dy.device).cuda_stream
        conv_bwd_data(self.handle, dy.data_ptr(), self.w_packed.data_ptr(), dx.data_ptr(), s)
        return dx

    def backward_weight(self, x, dy, dw, stream=None):
        import torch
        if self.workspace is None and conv_workspace_bytes(self.handle):
            self.allocate(x.device)
        s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        conv_bwd_weight(self.handle, x.data_ptr(), dy.data_ptr(), dw.data_ptr(), s)
        return dw

    def set_overlap(self, enable: bool = True):
        conv_plan_set_overlap(self.handle, enable)

    def tune(self, x, w, bias, y, iters: int = 10, stream=None):
        """Measure the candidate plans on these tensors, keep the fastest, and re-make the
        packed weight and workspace for it.  y is overwritten."""
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
        nbytes = conv_tune_scratch_bytes(self.handle)
        scratch = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
        conv_plan_tune(self.handle, x.data_ptr(), w.data_ptr(), 0 if bias is None else bias.data_ptr(),
                       y.data_ptr(), scratch.data_ptr(), nbytes, iters, s)
        del scratch
        self.workspace = None
        self.w_packed = None
        self.allocate(x.device)
        self.prepack(w, stream)
        return self.describe()

    def check(self, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
        conv_plan_check(self.handle, s)

    def close(self):
        if self.handle:
            conv_plan_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
