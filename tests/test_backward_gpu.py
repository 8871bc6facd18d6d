"""GPU parity of the backward passes (backward data, backward weight) through the C-ABI
against the CPU oracle, element by element, on seeded inputs; integer inputs bit-exact."""
import dataclasses
import os
import zlib

import numpy as np
import pytest

import oracle
from convolution_forward_implicit_gb300 import synthetic as syn
from convolution_forward_implicit_gb300.binding import CONV_BF16, CONV_EPI_NONE, CONV_F32, ConvPlan
from convolution_forward_implicit_gb300.workloads import WORKLOADS
from tests.helpers import SENTINEL, assert_within, from_device, geom_of, to_device
from tests.test_parity_gpu import L

pytestmark = pytest.mark.gpu


def make_bwd_inputs(layer, dtype, seed, kind="normal"):
    g = geom_of(layer)
    if kind == "int":
        x = syn.gen_int(seed, layer.x_shape(), -3, 3, dtype)
        w = syn.gen_int(seed + 1, layer.w_shape(), -3, 3, dtype)
        dy = syn.gen_int(seed + 2, g.y_shape(), -3, 3, dtype)
    else:
        x = syn.gen_normal(seed, layer.x_shape(), dtype)
        w = syn.gen_uniform_pm(seed + 1, layer.w_shape(), layer.w_bound, dtype)
        dy = syn.gen_normal(seed + 2, g.y_shape(), dtype)
    return x, w, dy


def _guarded(n, tdt, guard=64):
    import torch
    buf = torch.full((n + 2 * guard,), SENTINEL, dtype=tdt, device="cuda")
    return buf, buf[guard:guard + n]


def _check_guard(buf, n, guard=64):
    import torch
    sent = torch.cat([buf[:guard], buf[guard + n:]]).float()
    assert bool((sent == SENTINEL).all()), "kernel wrote outside its output"


def run_bwd_data(layer, dtype, dy, w, env=None):
    import torch
    code = CONV_BF16 if dtype == "bf16" else CONV_F32
    plan = _plan_with_env(layer, code, "bwd_data", env)
    plan.allocate()
    plan.prepack(to_device(w, dtype))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    n = int(np.prod(layer.x_shape()))
    buf, dx = _guarded(n, tdt)
    plan.backward_data(to_device(dy, dtype), dx)
    plan.check()
    torch.cuda.synchronize()
    _check_guard(buf, n)
    desc = plan.describe()
    plan.close()
    return from_device(dx, dtype), desc


def _plan_with_env(layer, code, direction, env):
    old = {}
    for k, v in (env or {}).items():
        old[k] = os.environ.get(k)
        os.environ[k] = str(v)
    try:
        return ConvPlan(*layer.plan_args(code), direction=direction)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def run_bwd_weight(layer, dtype, x, dy, env=None):
    import torch
    code = CONV_BF16 if dtype == "bf16" else CONV_F32
    plan = _plan_with_env(layer, code, "bwd_weight", env)
    plan.allocate()
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    n = int(np.prod(layer.w_shape()))
    buf, dw = _guarded(n, tdt)
    plan.backward_weight(to_device(x, dtype), to_device(dy, dtype), dw)
    plan.check()
    torch.cuda.synchronize()
    _check_guard(buf, n)
    desc = plan.describe()
    plan.close()
    return from_device(dw, dtype), desc


def B_(ndim, N, G, C, K, spatial, filt, stride, pad, dil):
    return L(ndim, N, G, C, K, spatial, filt, stride, pad, dil, CONV_EPI_NONE)


CASES = [
    # unit stride: backward data runs the forward kernels on the transposed problem
    ("1d_s1", "bf16", B_(1, 2, 1, 64, 72, (301,), (3,), (1,), (1,), (1,))),
    ("1d_s1_whisper_l1_shape", "bf16", B_(1, 1, 1, 80, 384, (517,), (3,), (1,), (1,), (1,))),
    ("2d_s1_groups", "bf16", B_(2, 2, 4, 32, 40, (19, 23), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("2d_s1_dil2_g8", "bf16", B_(2, 1, 8, 64, 64, (20, 18), (3, 3), (1, 1), (2, 2), (2, 2))),
    ("3d_s1_g4", "bf16", B_(3, 1, 4, 64, 64, (5, 9, 10), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1))),
    ("2d_s1_g32_c8", "bf16", B_(2, 2, 32, 8, 8, (17, 15), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("2d_s1_no_pad", "bf16", B_(2, 1, 1, 16, 24, (9, 12), (3, 2), (1, 1), (0, 0), (1, 1))),
    ("1d_s1_f32", "f32", B_(1, 1, 1, 80, 96, (300,), (3,), (1,), (1,), (1,))),
    ("2d_s1_f32_groups", "f32", B_(2, 2, 3, 40, 24, (11, 13), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("3d_s1_f32_odd", "f32", B_(3, 1, 2, 5, 7, (4, 6, 5), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1))),
    # stride > 1 or padding beyond the filter's reach: the gather kernel
    ("1d_s2", "bf16", B_(1, 1, 1, 64, 96, (301,), (3,), (2,), (1,), (1,))),
    ("1d_s2_whisper_l2_shape", "f32", B_(1, 1, 1, 96, 64, (400,), (3,), (2,), (1,), (1,))),
    ("2d_s2_dil", "bf16", B_(2, 2, 2, 24, 16, (17, 15), (5, 3), (2, 3), (3, 2), (1, 2))),
    ("3d_s2", "f32", B_(3, 1, 2, 8, 12, (7, 9, 8), (3, 3, 3), (2, 1, 2), (1, 1, 1), (1, 1, 1))),
    ("2d_big_pad", "bf16", B_(2, 1, 1, 16, 16, (6, 6), (3, 3), (1, 1), (3, 3), (1, 1))),
    ("1d_1x1_s2", "f32", B_(1, 2, 2, 12, 20, (33,), (1,), (2,), (0,), (1,))),
    # stride phases on the tensor cores: outputs on a lattice of dx
    ("1d_s2_c128", "bf16", B_(1, 2, 1, 128, 128, (1001,), (3,), (2,), (1,), (1,))),
    ("2d_s2_3x3_c64", "bf16", B_(2, 2, 1, 64, 64, (29, 31), (3, 3), (2, 2), (1, 1), (1, 1))),
    ("2d_1x1_s2_zero_fill", "bf16", B_(2, 1, 2, 64, 64, (15, 14), (1, 1), (2, 2), (0, 0), (1, 1))),
    ("3d_s2_c64", "bf16", B_(3, 1, 1, 64, 64, (7, 9, 10), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1))),
    ("1d_s2_tf32", "f32", B_(1, 1, 1, 64, 96, (777,), (3,), (2,), (1,), (1,))),
    ("2d_s2_dil2_pad3", "bf16", B_(2, 1, 2, 32, 48, (21, 19), (3, 3), (2, 2), (3, 3), (2, 2))),
    ("1d_s3_k5", "bf16", B_(1, 1, 1, 64, 64, (500,), (5,), (3,), (2,), (1,))),
    ("2d_s2_groups_c8", "bf16", B_(2, 1, 16, 8, 8, (20, 22), (3, 3), (2, 2), (1, 1), (1, 1))),
]


@pytest.mark.parametrize("name,dtype,layer", CASES, ids=[c[0] for c in CASES])
def test_backward_data_matches_oracle(name, dtype, layer):
    x, w, dy = make_bwd_inputs(layer, dtype, 7000 + zlib.crc32(name.encode()) % 1000)
    got, desc = run_bwd_data(layer, dtype, dy, w)
    ref, S = oracle.conv_bwd_data(geom_of(layer), syn.as_f32(dy, dtype), syn.as_f32(w, dtype))
    assert_within(dtype, CONV_EPI_NONE, got, ref.reshape(-1), S.reshape(-1), f"{name} [{desc}]")


@pytest.mark.parametrize("name,dtype,layer", CASES, ids=[c[0] for c in CASES])
def test_backward_weight_matches_oracle(name, dtype, layer):
    x, w, dy = make_bwd_inputs(layer, dtype, 8000 + zlib.crc32(name.encode()) % 1000)
    got, desc = run_bwd_weight(layer, dtype, x, dy)
    ref, S = oracle.conv_bwd_weight(geom_of(layer), syn.as_f32(x, dtype), syn.as_f32(dy, dtype))
    assert_within(dtype, CONV_EPI_NONE, got, ref.reshape(-1), S.reshape(-1), f"{name} [{desc}]")


@pytest.mark.parametrize("name", ["2d_s1_groups", "2d_s2_dil", "3d_s1_g4", "1d_s1_f32", "3d_s2"])
def test_backward_integer_inputs_bit_exact(name):
    """Small integers: every product and partial sum is exact in fp32, so fp32 results equal
    the oracle exactly and bf16 results equal its round-to-nearest-even."""
    dtype, layer = {c[0]: (c[1], c[2]) for c in CASES}[name]
    x, w, dy = make_bwd_inputs(layer, dtype, 9000, kind="int")
    g = geom_of(layer)
    for kind in ("data", "weight"):
        if kind == "data":
            got, desc = run_bwd_data(layer, dtype, dy, w)
            ref, _ = oracle.conv_bwd_data(g, syn.as_f32(dy, dtype), syn.as_f32(w, dtype))
        else:
            got, desc = run_bwd_weight(layer, dtype, x, dy)
            ref, _ = oracle.conv_bwd_weight(g, syn.as_f32(x, dtype), syn.as_f32(dy, dtype))
        if dtype == "f32":
            assert np.array_equal(got.reshape(-1).astype(np.float64), ref.reshape(-1)), f"{name} {kind} [{desc}]"
        else:
            want = syn.f32_to_bf16_bits(ref.reshape(-1).astype(np.float32))
            assert np.array_equal(got.reshape(-1), want), f"{name} {kind} [{desc}]"


FULL = ["grouped2d_g8_c64_d1", "grouped2d_g32_c8_d2", "grouped3d_g4_c64_d2", "whisper_frontend_bf16",
        "whisper_frontend_f32"]


@pytest.mark.parametrize("wl_name", FULL)
def test_backward_full_size_every_element(wl_name):
    """The workloads at full size: every element of dx and dw against the oracle."""
    wl = WORKLOADS[wl_name]
    for li, layer in enumerate(wl.layers):
        layer = dataclasses.replace(layer, epilogue=CONV_EPI_NONE, bias_bound=None)
        x, w, dy = make_bwd_inputs(layer, wl.dtype, 9500 + 10 * wl.index + li)
        g = geom_of(layer)
        dx, ddesc = run_bwd_data(layer, wl.dtype, dy, w)
        ref, S = oracle.conv_bwd_data(g, syn.as_f32(dy, wl.dtype), syn.as_f32(w, wl.dtype))
        assert_within(wl.dtype, CONV_EPI_NONE, dx, ref.reshape(-1), S.reshape(-1), f"{wl_name} L{li + 1} dx [{ddesc}]")
        dw, wdesc = run_bwd_weight(layer, wl.dtype, x, dy)
        ref, S = oracle.conv_bwd_weight(g, syn.as_f32(x, wl.dtype), syn.as_f32(dy, wl.dtype))
        assert_within(wl.dtype, CONV_EPI_NONE, dw, ref.reshape(-1), S.reshape(-1), f"{wl_name} L{li + 1} dw [{wdesc}]")


VARIANT_LAYERS = ["2d_s1_groups", "1d_s2", "2d_s1_g32_c8", "3d_s1_g4", "2d_s2_dil"]


@pytest.mark.parametrize("env", [{"CONV_FORCE_SIMT": 1}, {"CONV_FORCE_BN": 64, "CONV_FORCE_SPLITK": 3},
                                 {"CONV_FORCE_BN": 128, "CONV_FORCE_SPLITK": 1},
                                 {"CONV_FORCE_BN": 256, "CONV_FORCE_SPLITK": 7}],
                         ids=["ffma", "tc_bn64_split3", "tc_bn128_whole", "tc_bn256_split7"])
@pytest.mark.parametrize("name", VARIANT_LAYERS)
def test_backward_weight_variants(name, env):
    """Both backward-weight kernels, every tensor-core N tile, whole and split reductions."""
    dtype, layer = {c[0]: (c[1], c[2]) for c in CASES}[name]
    x, w, dy = make_bwd_inputs(layer, dtype, 8500 + len(name))
    got, desc = run_bwd_weight(layer, dtype, x, dy, env=env)
    if "CONV_FORCE_SIMT" in env:
        assert desc.startswith("variant=simt"), desc
    else:
        packed = "pack=1" not in desc          # packed small groups always use 64-wide tiles
        assert "operands=mn-major" in desc and f"tile=128x{64 if packed else env['CONV_FORCE_BN']}" in desc, desc
    ref, S = oracle.conv_bwd_weight(geom_of(layer), syn.as_f32(x, dtype), syn.as_f32(dy, dtype))
    assert_within(dtype, CONV_EPI_NONE, got, ref.reshape(-1), S.reshape(-1), f"{name} [{desc}]")


@pytest.mark.parametrize("splits", [1, 2, 3])
@pytest.mark.parametrize("name", ["1d_s2_c128", "2d_s2_3x3_c64", "1d_s2_tf32"])
def test_backward_data_phases_with_split_reductions(name, splits):
    """Stride phases with whole reductions, cluster-summed splits (2) and the reduction kernel (3),
    whose outputs land on the lattice too."""
    dtype, layer = {c[0]: (c[1], c[2]) for c in CASES}[name]
    x, w, dy = make_bwd_inputs(layer, dtype, 7700 + splits)
    got, desc = run_bwd_data(layer, dtype, dy, w, env={"CONV_FORCE_SPLITK": splits})
    assert "bwd_data(phases)" in desc, desc
    ref, S = oracle.conv_bwd_data(geom_of(layer), syn.as_f32(dy, dtype), syn.as_f32(w, dtype))
    assert_within(dtype, CONV_EPI_NONE, got, ref.reshape(-1), S.reshape(-1), f"{name} [{desc}]")


PACKED = [
    ("g32_c8_k8", B_(2, 2, 32, 8, 8, (17, 15), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("g16_c8_k16", B_(2, 1, 16, 8, 16, (13, 20), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("g8_c16_k8_s2", B_(2, 1, 8, 16, 8, (19, 23), (3, 3), (2, 2), (1, 1), (1, 1))),
    ("g6_c16_k16_ragged_pack", B_(1, 2, 6, 16, 16, (200,), (3,), (1,), (1,), (1,))),
    ("g12_c32_k32_3d", B_(3, 1, 12, 32, 32, (4, 7, 9), (3, 3, 3), (1, 1, 1), (1, 1, 1), (2, 1, 1))),
]


@pytest.mark.parametrize("no_pack", [0, 1])
@pytest.mark.parametrize("name,layer", PACKED, ids=[c[0] for c in PACKED])
def test_backward_weight_packed_small_groups(name, layer, no_pack):
    """Groups narrower than half a 64-channel box share one tile (only the diagonal blocks are
    stored), including a last pack with fewer groups; CONV_NO_PACK=1 runs them one per tile."""
    x, w, dy = make_bwd_inputs(layer, "bf16", 8800 + len(name))
    got, desc = run_bwd_weight(layer, "bf16", x, dy, env={"CONV_NO_PACK": no_pack} if no_pack else None)
    assert ("pack=1" in desc) == bool(no_pack), desc
    ref, S = oracle.conv_bwd_weight(geom_of(layer), syn.as_f32(x, "bf16"), syn.as_f32(dy, "bf16"))
    assert_within("bf16", CONV_EPI_NONE, got, ref.reshape(-1), S.reshape(-1), f"{name} [{desc}]")


@pytest.mark.parametrize("name", ["1d_s1_f32", "2d_s1_f32_groups", "1d_s2_whisper_l2_shape", "1d_s2_tf32"])
def test_fp32_backward_weight_on_tensor_cores_meets_the_fp32_bound(name):
    """fp32 x and dy split into three bf16 planes, six plane products per tile: the fp32 bound
    (1e-5 of the sum of |x dy|) holds, and the plan is the tensor-core one."""
    dtype, layer = {c[0]: (c[1], c[2]) for c in CASES}[name]
    x, w, dy = make_bwd_inputs(layer, dtype, 8900 + len(name))
    got, desc = run_bwd_weight(layer, dtype, x, dy)
    assert desc.startswith("variant=tc_bf16x3"), desc
    ref, S = oracle.conv_bwd_weight(geom_of(layer), syn.as_f32(x, dtype), syn.as_f32(dy, dtype))
    ratio, _ = assert_within(dtype, CONV_EPI_NONE, got, ref.reshape(-1), S.reshape(-1), f"{name} [{desc}]")
    assert ratio < 0.1, ratio      # two orders of magnitude inside the bound


SLAB_W = [
    ("2d_3x3_c64_g2_wide", B_(2, 2, 2, 64, 64, (20, 70), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("2d_3x3_c64_dil2", B_(2, 1, 1, 64, 64, (18, 33), (3, 3), (1, 1), (2, 2), (2, 2))),
    ("3d_3x3x3_c64", B_(3, 1, 2, 64, 64, (5, 9, 70), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1))),
    ("1d_k5_c128", B_(1, 2, 1, 128, 64, (300,), (5,), (1,), (2,), (1,))),
    ("2d_g16_c8_packed", B_(2, 1, 16, 8, 8, (20, 22), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("2d_s2_rows_only", B_(2, 1, 1, 64, 64, (21, 40), (3, 3), (2, 1), (1, 1), (1, 1))),
]


@pytest.mark.parametrize("per_tap", [0, 1])
@pytest.mark.parametrize("name,layer", SLAB_W, ids=[c[0] for c in SLAB_W])
def test_backward_weight_slab_windows(name, layer, per_tap):
    """Unit stride along W: one x box per filter row serves every tap of that row as shifted
    MN-major windows (slab mode); CONV_FORCE_GATHER=tma runs the per-tap boxes instead."""
    x, w, dy = make_bwd_inputs(layer, "bf16", 9100 + len(name))
    got, desc = run_bwd_weight(layer, "bf16", x, dy, env={"CONV_FORCE_GATHER": "tma"} if per_tap else None)
    assert ("operands=mn-major-slab" in desc) == (not per_tap), desc
    ref, S = oracle.conv_bwd_weight(geom_of(layer), syn.as_f32(x, "bf16"), syn.as_f32(dy, "bf16"))
    assert_within("bf16", CONV_EPI_NONE, got, ref.reshape(-1), S.reshape(-1), f"{name} [{desc}]")
