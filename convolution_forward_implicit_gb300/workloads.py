"""The convolution workloads this library is measured and checked on, with their input
recipe.  Shapes and distributions only; no convolution arithmetic.

Sources (all synthetic, seeded; no dataset or trained weights is involved):
  * Whisper-tiny conv frontend and its single-layer form: page "[ET-VK] conv1d runs at
    ~3% of the GPU's matmul throughput ...", section "Measurements" (80 -> 384, k=3,
    L=3000; 384 -> 384, k=3, stride 2, output 1500) and section "The conv2d path already
    solves this" (two convs plus GELU).
  * A wider conv1d frontend sweep (128 -> 1280 -> 1280) at batch 1, 8 and 32.
  * Grouped 2D / 3D forward NHWGC x GKYXC -> NHWGK with dilation: page
    "composable_kernel dispatcher/heuristics/LEARNINGS_GROUPED_CONV.md", introduction
    and section 2 (3D shapes and dilation_d/h/w).
Distributions: x ~ N(0,1); w ~ U(+-1/sqrt(C_in * taps)); bias ~ U(+-0.05) where a
layer has one.  Layer l of workload i draws its weights from stream
BASE_SEED + 1000*i + 10*l + 1 and its bias from ... + 2; the input from BASE_SEED + 1000*i.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional, Tuple

import numpy as np

from . import synthetic as syn
from .binding import CONV_BF16, CONV_EPI_BIAS, CONV_EPI_BIAS_GELU, CONV_EPI_NONE, CONV_F32


@dataclass(frozen=True)
class Layer:
    ndim: int
    N: int
    G: int
    C: int
    K: int
    spatial: Tuple[int, ...]
    filter: Tuple[int, ...]
    stride: Tuple[int, ...]
    pad: Tuple[int, ...]
    dilation: Tuple[int, ...]
    epilogue: int
    bias_bound: Optional[float]     # None: no bias

    @property
    def taps(self) -> int:
        return int(np.prod(self.filter))

    @property
    def w_bound(self) -> float:
        return 1.0 / math.sqrt(self.C * self.taps)

    def x_shape(self):
        return (self.N, *self.spatial, self.G, self.C)

    def w_shape(self):
        return (self.G, self.K, *self.filter, self.C)

    def plan_args(self, dtype_code: int):
        return (self.ndim, self.N, self.G, self.C, self.K, self.spatial, self.filter, self.stride, self.pad,
                self.dilation, dtype_code, self.epilogue)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                  # seed index
    dtype: str                  # 'f32' or 'bf16'
    layers: Tuple[Layer, ...]   # layer l+1 reads layer l's output
    note: str = ""

    @property
    def dtype_code(self) -> int:
        return CONV_BF16 if self.dtype == "bf16" else CONV_F32


def _conv1d(N, C, K, L, stride, epi, bias=0.05):
    return Layer(1, N, 1, C, K, (L,), (3,), (stride,), (1,), (1,), epi, bias)


def whisper_layers(N=1, L=3000):
    return (_conv1d(N, 80, 384, L, 1, CONV_EPI_BIAS_GELU), _conv1d(N, 384, 384, L, 2, CONV_EPI_BIAS_GELU))


def sweep_layers(N, L=3000):
    return (_conv1d(N, 128, 1280, L, 1, CONV_EPI_BIAS_GELU), _conv1d(N, 1280, 1280, L, 2, CONV_EPI_BIAS_GELU))


def grouped2d(G, C, d, N=16, HW=56):
    return Layer(2, N, G, C, C, (HW, HW), (3, 3), (1, 1), (1, 1), (d, d), CONV_EPI_NONE, None)


def grouped3d(d, N=4, D=16, HW=56, G=4, C=64):
    return Layer(3, N, G, C, C, (D, HW, HW), (3, 3, 3), (1, 1, 1), (1, 1, 1), (d, d, d), CONV_EPI_BIAS, 0.05)


def whisper_mlp_layers():
    """The encoder's feed-forward block as 1x1 convolutions over the 1500 frame positions
    (page "[ET-VK] conv1d ...", "Measurements": the linear dispatches M=1500, N=1536, K=384
    and M=1500, N=384, K=1536): 384 -> 1536 with bias and GELU, then 1536 -> 384 with bias."""
    return (Layer(1, 1, 1, 384, 1536, (1500,), (1,), (1,), (0,), (1,), CONV_EPI_BIAS_GELU, 0.05),
            Layer(1, 1, 1, 1536, 384, (1500,), (1,), (1,), (0,), (1,), CONV_EPI_BIAS, 0.05))


WORKLOADS = {
    "conv1d_f32_80to384_L3000": Workload(
        "conv1d_f32_80to384_L3000", 0, "f32", (_conv1d(1, 80, 384, 3000, 1, CONV_EPI_BIAS),),
        "conv1d fp32 N=1 80->384 k3 s1 p1 L=3000, bias, no activation"),
    "whisper_frontend_f32": Workload("whisper_frontend_f32", 1, "f32", whisper_layers(),
                                     "Whisper-tiny conv frontend fp32, N=1"),
    "whisper_frontend_bf16": Workload("whisper_frontend_bf16", 1, "bf16", whisper_layers(),
                                      "Whisper-tiny conv frontend bf16, N=1"),
    "sweep_bf16_n1": Workload("sweep_bf16_n1", 2, "bf16", sweep_layers(1), "conv1d frontend sweep, N=1"),
    "sweep_bf16_n8": Workload("sweep_bf16_n8", 2, "bf16", sweep_layers(8), "conv1d frontend sweep, N=8"),
    "sweep_bf16_n32": Workload("sweep_bf16_n32", 2, "bf16", sweep_layers(32), "conv1d frontend sweep, N=32"),
    "grouped2d_g8_c64_d1": Workload("grouped2d_g8_c64_d1", 3, "bf16", (grouped2d(8, 64, 1),)),
    "grouped2d_g8_c64_d2": Workload("grouped2d_g8_c64_d2", 3, "bf16", (grouped2d(8, 64, 2),)),
    "grouped2d_g32_c8_d1": Workload("grouped2d_g32_c8_d1", 4, "bf16", (grouped2d(32, 8, 1),)),
    "grouped2d_g32_c8_d2": Workload("grouped2d_g32_c8_d2", 4, "bf16", (grouped2d(32, 8, 2),)),
    "grouped3d_g4_c64_d1": Workload("grouped3d_g4_c64_d1", 5, "bf16", (grouped3d(1),)),
    "grouped3d_g4_c64_d2": Workload("grouped3d_g4_c64_d2", 5, "bf16", (grouped3d(2),)),
    "whisper_mlp_f32": Workload("whisper_mlp_f32", 6, "f32", whisper_mlp_layers(),
                                "Whisper-tiny encoder MLP as 1x1 convs fp32, 1500 positions"),
    "whisper_mlp_bf16": Workload("whisper_mlp_bf16", 6, "bf16", whisper_mlp_layers(),
                                 "Whisper-tiny encoder MLP as 1x1 convs bf16, 1500 positions"),
}


def layer_seed(index: int, layer: int, tensor: int) -> int:
    return syn.BASE_SEED + 1000 * index + 10 * layer + tensor


def gen_inputs(wl: Workload):
    """Storage arrays (float32, or bf16 bits as uint16): x, and per layer (w, bias or None)."""
    l0 = wl.layers[0]
    x = syn.gen_normal(layer_seed(wl.index, 0, syn.TENSOR_X), l0.x_shape(), wl.dtype)
    params = []
    for li, L in enumerate(wl.layers):
        w = syn.gen_uniform_pm(layer_seed(wl.index, li, syn.TENSOR_W), L.w_shape(), L.w_bound, wl.dtype)
        b = None
        if L.bias_bound is not None:
            b = syn.gen_uniform_pm(layer_seed(wl.index, li, syn.TENSOR_BIAS), (L.G * L.K,), L.bias_bound, wl.dtype)
        params.append((w, b))
    return x, params


def shrink(wl: Workload, **changes) -> Workload:
    """The same workload with some layer fields changed on every layer (e.g. N, spatial)."""
    return replace(wl, layers=tuple(replace(L, **changes) for L in wl.layers))
