"""GPU parity: the CUDA path through the C-ABI against the CPU oracle, element by element,
on the same seeded inputs.  Every test here needs a GB300 and the built library."""
import os
import zlib

import numpy as np
import pytest

from convolution_forward_implicit_gb300 import synthetic as syn
from convolution_forward_implicit_gb300.binding import (CONV_BF16, CONV_EPI_BIAS, CONV_EPI_BIAS_GELU,
                                                        CONV_EPI_GELU, CONV_EPI_NONE, CONV_ERR_ALIGNMENT,
                                                        CONV_ERR_WORKSPACE, CONV_F32, ConvError, ConvPlan)
from convolution_forward_implicit_gb300.workloads import WORKLOADS, Layer, gen_inputs
from tests.helpers import assert_within, has_bias, oracle_full, run_gpu, to_device

pytestmark = pytest.mark.gpu

def make_inputs(layer, dtype, seed, kind="normal"):
    if kind == "int":
        x = syn.gen_int(seed, layer.x_shape(), -3, 3, dtype)
        w = syn.gen_int(seed + 1, layer.w_shape(), -3, 3, dtype)
        b = syn.gen_int(seed + 2, (layer.G * layer.K,), -2, 2, dtype)
    else:
        x = syn.gen_normal(seed, layer.x_shape(), dtype)
        w = syn.gen_uniform_pm(seed + 1, layer.w_shape(), layer.w_bound, dtype)
        b = syn.gen_uniform_pm(seed + 2, (layer.G * layer.K,), 0.05, dtype)
    return x, w, b


def L(ndim, N, G, C, K, spatial, filt, stride, pad, dil, epi=CONV_EPI_BIAS_GELU):
    return Layer(ndim, N, G, C, K, tuple(spatial), tuple(filt), tuple(stride), tuple(pad), tuple(dil), epi,
                 0.05 if has_bias(epi) else None)


# Small problems spanning several tiles with ragged tails, every ndim, groups, stride,
# padding, dilation and epilogue; bf16 cases with C, K multiples of 8 take the tensor-core
# path, the others the FFMA path.
SMALL = [
    ("1d_tc_ragged", "bf16", L(1, 2, 1, 64, 72, (301,), (3,), (1,), (1,), (1,))),
    ("1d_tc_s2", "bf16", L(1, 1, 1, 80, 384, (517,), (3,), (2,), (1,), (1,))),
    ("1d_tc_dil_pad", "bf16", L(1, 3, 2, 16, 24, (97,), (5,), (2,), (4,), (3,), CONV_EPI_BIAS)),
    ("2d_tc_group", "bf16", L(2, 2, 4, 32, 40, (19, 23), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_NONE)),
    ("2d_tc_dil2", "bf16", L(2, 1, 2, 64, 64, (30, 27), (3, 3), (1, 1), (1, 1), (2, 2), CONV_EPI_GELU)),
    ("2d_tc_stride2_big_pad", "bf16", L(2, 2, 1, 24, 200, (17, 15), (5, 3), (2, 3), (3, 2), (1, 2))),
    ("3d_tc", "bf16", L(3, 2, 2, 8, 16, (6, 9, 11), (3, 3, 3), (1, 1, 1), (1, 1, 1), (2, 1, 2), CONV_EPI_BIAS)),
    ("3d_tc_k8", "bf16", L(3, 1, 3, 8, 8, (5, 7, 6), (3, 2, 3), (1, 2, 1), (1, 0, 1), (1, 1, 2))),
    ("1d_tc_k264", "bf16", L(1, 1, 1, 40, 264, (260,), (3,), (1,), (1,), (1,))),
    ("2d_tc_k512", "bf16", L(2, 1, 1, 16, 512, (12, 13), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("1d_bf16_simt_oddC", "bf16", L(1, 2, 1, 5, 7, (203,), (3,), (1,), (1,), (1,))),
    ("2d_bf16_simt_c12", "bf16", L(2, 1, 3, 12, 20, (11, 14), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("1d_f32", "f32", L(1, 1, 1, 80, 384, (300,), (3,), (1,), (1,), (1,), CONV_EPI_BIAS)),
    ("1d_f32_s2", "f32", L(1, 2, 1, 48, 96, (257,), (3,), (2,), (1,), (1,))),
    ("2d_f32_group_dil", "f32", L(2, 2, 4, 8, 12, (21, 17), (3, 3), (1, 1), (2, 2), (2, 2), CONV_EPI_NONE)),
    ("3d_f32", "f32", L(3, 1, 2, 16, 20, (5, 9, 10), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), CONV_EPI_BIAS)),
    ("2d_f32_odd", "f32", L(2, 3, 1, 3, 5, (13, 11), (2, 3), (1, 2), (0, 1), (1, 1))),
    ("1d_f32_1x1", "f32", L(1, 4, 2, 20, 36, (77,), (1,), (1,), (0,), (1,))),
    ("2d_bf16_1x1", "bf16", L(2, 2, 2, 32, 48, (9, 10), (1, 1), (1, 1), (0, 0), (1, 1))),
    ("2d_tc_taps_in_padding", "bf16", L(2, 1, 1, 16, 16, (4, 4), (3, 3), (3, 3), (5, 5), (4, 4))),
    ("1d_tc_tiny_M", "bf16", L(1, 1, 1, 8, 16, (1,), (1,), (1,), (0,), (1,))),
    # TMA gather: both tensor-map layouts, strides, dilation, ragged tiles
    ("2d_tma_map1_c72", "bf16", L(2, 2, 2, 72, 40, (13, 21), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("1d_tma_s2_dil", "bf16", L(1, 2, 1, 64, 64, (400,), (5,), (2,), (4,), (2,))),
    ("2d_tma_stride2", "bf16", L(2, 1, 1, 128, 64, (30, 35), (3, 3), (2, 2), (1, 1), (1, 1))),
    ("3d_tma_c64_dil", "bf16", L(3, 1, 2, 64, 64, (5, 9, 10), (3, 3, 3), (1, 1, 1), (2, 2, 2), (2, 2, 2),
                                 CONV_EPI_BIAS)),
    ("3d_g2_c96_cpasync", "bf16", L(3, 1, 2, 96, 32, (4, 6, 7), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1))),
    ("2d_tma_wide_w", "bf16", L(2, 1, 1, 64, 48, (3, 300), (3, 3), (1, 3), (1, 1), (1, 1))),
    # fp32 I/O on the tensor cores (3xTF32)
    ("1d_tf32_s2_k384", "f32", L(1, 1, 1, 384, 384, (301,), (3,), (2,), (1,), (1,))),
    ("2d_tf32_group_map1", "f32", L(2, 2, 3, 40, 24, (11, 13), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_BIAS)),
    ("2d_tf32_g2_c32_dil", "f32", L(2, 1, 2, 32, 36, (17, 19), (3, 3), (1, 1), (2, 2), (2, 2), CONV_EPI_NONE)),
    ("3d_tf32_c64", "f32", L(3, 1, 2, 64, 40, (4, 7, 9), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), CONV_EPI_BIAS)),
    ("1d_tf32_k4", "f32", L(1, 3, 1, 32, 4, (129,), (3,), (1,), (1,), (1,))),
]


@pytest.mark.parametrize("name,dtype,layer", SMALL, ids=[s[0] for s in SMALL])
def test_small_problems_full_parity(name, dtype, layer):
    x, w, b = make_inputs(layer, dtype, 1000 + zlib.crc32(name.encode()) % 1000)
    got, desc = run_gpu(layer, dtype, x, w, b, guard=64)
    ref, S = oracle_full(layer, dtype, x, w, b)
    assert_within(dtype, layer.epilogue, got, ref, S, f"{name} [{desc}]")


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_split_k_matches_oracle_and_is_deterministic(splits, dtype):
    layer = L(1, 1, 1, 128, 128, (700,), (3,), (2,), (1,), (1,))
    x, w, b = make_inputs(layer, dtype, 77)
    env = {"CONV_FORCE_SPLITK": splits}
    got, desc = run_gpu(layer, dtype, x, w, b, env=env, guard=64)
    assert f"splits={splits}" in desc or splits > 1
    ref, S = oracle_full(layer, dtype, x, w, b)
    assert_within(dtype, layer.epilogue, got, ref, S, desc)
    again, _ = run_gpu(layer, dtype, x, w, b, env=env)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("bn", [16, 32, 64, 128, 256])
def test_every_tensor_core_tile_width(bn):
    layer = L(2, 1, 2, 24, 136, (13, 37), (3, 3), (1, 1), (1, 1), (1, 1))
    x, w, b = make_inputs(layer, "bf16", 500 + bn)
    got, desc = run_gpu(layer, "bf16", x, w, b, env={"CONV_FORCE_BN": bn}, guard=64)
    assert f"tile=128x{bn}" in desc
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, got, ref, S, desc)


@pytest.mark.parametrize("bn", [64, 128, 256])
def test_every_tile_width_with_tma_gather(bn):
    layer = L(2, 2, 1, 64, 200, (9, 37), (3, 3), (1, 1), (1, 1), (1, 1))
    x, w, b = make_inputs(layer, "bf16", 600 + bn)
    got, desc = run_gpu(layer, "bf16", x, w, b, env={"CONV_FORCE_BN": bn}, guard=64)
    assert f"tile=128x{bn}" in desc and "gather=tma" in desc
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, got, ref, S, desc)


@pytest.mark.parametrize("case", [0, 1, 2])
def test_tma_and_cp_async_gathers_agree(case):
    layer = [L(1, 1, 1, 80, 384, (517,), (3,), (2,), (1,), (1,)),
             L(2, 2, 4, 64, 64, (14, 14), (3, 3), (1, 1), (2, 2), (2, 2), CONV_EPI_NONE),
             L(3, 1, 2, 64, 64, (4, 8, 8), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), CONV_EPI_BIAS)][case]
    x, w, b = make_inputs(layer, "bf16", 700 + case)
    ref, S = oracle_full(layer, "bf16", x, w, b)
    a, da = run_gpu(layer, "bf16", x, w, b)
    c, dc = run_gpu(layer, "bf16", x, w, b, env={"CONV_FORCE_GATHER": "cpasync"})
    assert "gather=tma" in da and "gather=cp.async" in dc
    assert_within("bf16", layer.epilogue, a, ref, S, da)
    assert_within("bf16", layer.epilogue, c, ref, S, dc)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_integer_inputs_bit_exact(dtype):
    """Integer x, w in [-3, 3], bias in [-2, 2]: every partial sum is an integer below 2^24,
    so fp32 accumulation is exact in any order; fp32 output equals the oracle exactly and
    bf16 output equals the oracle rounded to nearest even."""
    layers = [L(1, 2, 1, 128, 80, (150,), (3,), (2,), (1,), (1,), CONV_EPI_BIAS),
              L(2, 1, 4, 16, 24, (14, 12), (3, 3), (1, 1), (2, 1), (2, 1), CONV_EPI_BIAS),
              L(3, 1, 2, 24, 16, (5, 6, 7), (3, 3, 3), (1, 1, 2), (1, 1, 1), (1, 1, 1), CONV_EPI_BIAS)]
    for li, layer in enumerate(layers):
        for splits in (1, 3):
            x, w, b = make_inputs(layer, dtype, 900 + li, kind="int")
            got, desc = run_gpu(layer, dtype, x, w, b, env={"CONV_FORCE_SPLITK": splits})
            ref, _ = oracle_full(layer, dtype, x, w, b)
            if dtype == "f32":
                assert np.array_equal(got.reshape(-1).astype(np.float64), ref), desc
            else:
                assert np.array_equal(got.reshape(-1), syn.f32_to_bf16_bits(ref.astype(np.float32))), desc


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_delta_kernel_identity_and_shift_exact(dtype):
    G, C = 2, 16
    for t0 in [(1, 1), (0, 2), (2, 0)]:
        layer = L(2, 2, G, C, C, (9, 20), (3, 3), (1, 1), (2, 2), (2, 2), CONV_EPI_NONE)
        x = syn.gen_normal(31, layer.x_shape(), dtype)
        w = np.zeros(layer.w_shape(), np.float32)
        for gi in range(G):
            for k in range(C):
                w[gi, k, t0[0], t0[1], k] = 1.0
        w = syn.to_storage(w.astype(np.float64), dtype)
        got, desc = run_gpu(layer, dtype, x, w, None)
        xs = syn.as_f32(x, dtype).reshape(layer.x_shape())
        ref = np.zeros_like(xs)
        sh = [(t - 1) * 2 for t in t0]
        for oh in range(9):
            for ow in range(20):
                ih, iw = oh + sh[0], ow + sh[1]
                if 0 <= ih < 9 and 0 <= iw < 20:
                    ref[:, oh, ow] = xs[:, ih, iw]
        assert np.array_equal(syn.as_f32(got, dtype).reshape(ref.shape), ref), desc


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_conv1d_is_bit_identical_to_conv2d_with_h1(dtype):
    l1 = L(1, 2, 1, 64, 96, (301,), (3,), (2,), (1,), (2,))
    l2 = L(2, 2, 1, 64, 96, (1, 301), (1, 3), (1, 2), (0, 1), (1, 2))
    x, w, b = make_inputs(l1, dtype, 5)
    a, _ = run_gpu(l1, dtype, x, w, b)
    c, _ = run_gpu(l2, dtype, x.reshape(l2.x_shape()), w.reshape(l2.w_shape()), b)
    assert np.array_equal(a.reshape(-1), c.reshape(-1))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_grouped_equals_independent_convs(dtype):
    G = 3
    lg = L(2, 2, G, 16, 24, (11, 13), (3, 3), (1, 1), (1, 1), (1, 2), CONV_EPI_BIAS)
    l1 = L(2, 2, 1, 16, 24, (11, 13), (3, 3), (1, 1), (1, 1), (1, 2), CONV_EPI_BIAS)
    x, w, b = make_inputs(lg, dtype, 6)
    one_split = {"CONV_FORCE_SPLITK": 1}     # same reduction order in both runs
    got, _ = run_gpu(lg, dtype, x, w, b, env=one_split)
    got = syn.as_f32(got, dtype).reshape(2, *layer_out_spatial(lg), G, 24)
    xs, ws, bs = x.reshape(lg.x_shape()), w.reshape(lg.w_shape()), b.reshape(G, 24)
    for gi in range(G):
        one, _ = run_gpu(l1, dtype, np.ascontiguousarray(xs[..., gi:gi + 1, :]), np.ascontiguousarray(ws[gi:gi + 1]),
                         np.ascontiguousarray(bs[gi]), env=one_split)
        assert np.array_equal(syn.as_f32(one, dtype).reshape(got[..., gi, :].shape), got[..., gi, :])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_linearity_power_of_two_exact(dtype):
    layer = L(2, 1, 2, 32, 32, (15, 16), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_NONE)
    x, w, _ = make_inputs(layer, dtype, 8)
    x2 = syn.to_storage(2.0 * syn.as_f32(x, dtype).astype(np.float64), dtype)
    a, _ = run_gpu(layer, dtype, x, w, None)
    c, _ = run_gpu(layer, dtype, x2, w, None)
    assert np.array_equal(2.0 * syn.as_f32(a, dtype), syn.as_f32(c, dtype))


def test_error_paths_workspace_and_alignment():
    import torch
    layer = L(1, 1, 1, 64, 128, (700,), (3,), (2,), (1,), (1,))
    os.environ["CONV_FORCE_SPLITK"] = "3"
    try:
        plan = ConvPlan(*layer.plan_args(CONV_BF16))
    finally:
        os.environ.pop("CONV_FORCE_SPLITK")
    x = torch.zeros(layer.x_shape(), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(plan.y_shape(), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(128, dtype=torch.bfloat16, device="cuda")
    plan.w_packed = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ConvError) as e:
        plan.forward(x, b, y)
    assert e.value.status == CONV_ERR_WORKSPACE
    plan.allocate()
    xflat = x.view(-1)
    with pytest.raises(ConvError) as e:
        from convolution_forward_implicit_gb300.binding import conv_fwd
        conv_fwd(plan.handle, xflat[1:].data_ptr(), plan.w_packed.data_ptr(), b.data_ptr(), y.data_ptr(), 0)
    assert e.value.status == CONV_ERR_ALIGNMENT
    plan.check()
    plan.close()


def _sample_chunks(layer, max_macs=1.2e10):
    """Batch ranges [n0, n1) of at most max_macs multiply-adds each (at least one sample)."""
    per = layer.C * layer.taps * layer.G * layer.K * int(np.prod(layer_out_spatial(layer)))
    step = max(1, int(max_macs // max(per, 1)))
    return [(n0, min(layer.N, n0 + step)) for n0 in range(0, layer.N, step)]


def _workload_parity(name):
    """Every output of every layer against the oracle, a batch chunk at a time (outputs of
    sample n depend on sample n's input alone, so the oracle runs each chunk as its own
    problem with the same arithmetic)."""
    from dataclasses import replace
    wl = WORKLOADS[name]
    x, params = gen_inputs(wl)
    cur = x
    report = []
    for li, layer in enumerate(wl.layers):
        w, b = params[li]
        got, desc = run_gpu(layer, wl.dtype, cur, w, b)
        out_sp = layer_out_spatial(layer)
        got = got.reshape(layer.N, -1)
        cur_b = cur.reshape(layer.N, -1)
        worst, worst_bare, cos_min, n_el = 0.0, 0.0, 1.0, 0
        for n0, n1 in _sample_chunks(layer):
            sub = replace(layer, N=n1 - n0)
            ref, S = oracle_full(sub, wl.dtype, cur_b[n0:n1].reshape(sub.x_shape()), w, b)
            st = {}
            ratio, cos = assert_within(wl.dtype, layer.epilogue, got[n0:n1], ref, S,
                                       f"{name} layer {li} samples {n0}..{n1 - 1} [{desc}]", stats=st)
            worst, worst_bare = max(worst, ratio), max(worst_bare, st["bare_ratio"])
            cos_min, n_el = min(cos_min, cos), n_el + st["elements"]
        assert n_el == got.size
        print(f"{name} layer {li}: {n_el} outputs, every one checked; max err/bound {worst:.3f}, "
              f"max err/(rel*S) {worst_bare:.3f}, min cosine per chunk {cos_min:.8f} [{desc}]")
        report.append((li, desc, worst, cos_min))
        cur = got.reshape(layer.N, *out_sp, layer.G * layer.K)   # next layer's input (GPU bits)
    return report


def layer_out_spatial(layer):
    import oracle
    return tuple(oracle.out_len(i, f, s, p, d) for i, f, s, p, d in
                 zip(layer.spatial, layer.filter, layer.stride, layer.pad, layer.dilation))


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_every_output(name):
    """Every workload at its full size, in the configuration the benchmark times, with every
    output compared to the oracle.  Chained layers: layer l+1's oracle reads the GPU's
    layer-l output bits, so each layer meets the bound on its own."""
    _workload_parity(name)


def test_plan_made_before_any_cuda_context_still_uses_tma():
    """A plan created in a fresh process before any CUDA call picks the TMA gather."""
    import subprocess
    import sys
    code = ("from convolution_forward_implicit_gb300 import binding as B\n"
            "h = B.conv_plan_create(1, 1, 1, 128, 128, (500,), (3,), (1,), (1,), (1,), B.CONV_BF16, 0)\n"
            "print(B.conv_plan_describe(h))\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert "gather=tma" in out.stdout, out.stdout


@pytest.mark.parametrize("case", [0, 1])
def test_tf32x3_and_ffma_both_meet_the_fp32_bound(case):
    """fp32 I/O: the 3xTF32 tensor-core kernel and the FFMA kernel on the same inputs."""
    layer = [L(1, 1, 1, 80, 384, (3000,), (3,), (1,), (1,), (1,), CONV_EPI_BIAS_GELU),
             L(1, 1, 1, 384, 384, (3000,), (3,), (2,), (1,), (1,), CONV_EPI_BIAS_GELU)][case]
    x, w, b = make_inputs(layer, "f32", 800 + case)
    ref, S = oracle_full(layer, "f32", x, w, b)
    a, da = run_gpu(layer, "f32", x, w, b)
    c, dc = run_gpu(layer, "f32", x, w, b, env={"CONV_FORCE_SIMT": 1})
    assert "tc_tf32x3" in da and "simt" in dc
    ra, _ = assert_within("f32", layer.epilogue, a, ref, S, da)
    rc, _ = assert_within("f32", layer.epilogue, c, ref, S, dc)
    assert ra < 0.5, f"3xTF32 uses {ra:.2f} of the fp32 bound"


def test_gelu_epilogue_on_every_bf16_value_in_range():
    """Identity 1x1 conv with a GELU epilogue over every bf16 value in [-8, 8]: the output
    must be the exact (erf) GELU rounded to bf16, give or take one bf16 unit in the last
    place where the value sits next to a rounding boundary.  In the far negative tail, where
    GELU(v) is below 1e-3 |v|, an erf evaluated to a fixed absolute accuracy cannot give
    the tiny value to a few ulps; there the bound is the absolute one, 1e-6 |v|, plus the
    output's own bf16 rounding."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = syn.bf16_bits_to_f32(bits)
    keep = np.isfinite(vals) & (np.abs(vals) <= 8.0)
    vals = np.unique(vals[keep])
    C = 16
    n = (len(vals) + C - 1) // C
    xs = np.zeros(n * C, np.float32)
    xs[:len(vals)] = vals
    layer = L(1, 1, 1, C, C, (n,), (1,), (1,), (0,), (1,), CONV_EPI_GELU)
    x = syn.f32_to_bf16_bits(xs).reshape(layer.x_shape())
    w = syn.f32_to_bf16_bits(np.eye(C, dtype=np.float32)).reshape(layer.w_shape())
    got, desc = run_gpu(layer, "bf16", x, w, None)
    ref, _ = oracle_full(layer, "bf16", x, w, None)
    ref_bits = syn.f32_to_bf16_bits(ref.astype(np.float32))
    gi = got.reshape(-1).astype(np.int64)
    ri = ref_bits.astype(np.int64)
    # bf16 bit patterns of same-sign values differ by the ulp count
    same_sign = (gi >> 15) == (ri >> 15)
    ulps = np.where(same_sign, np.abs(gi - ri), np.abs(gi & 0x7FFF) + np.abs(ri & 0x7FFF))
    v = xs.astype(np.float64)
    tail = np.abs(ref) < 1e-3 * np.abs(v)
    assert ulps[~tail].max() <= 1, desc
    assert (ulps[~tail] == 0).mean() > 0.99, desc
    gotf = syn.bf16_bits_to_f32(got.reshape(-1)).astype(np.float64)
    rt = np.abs(ref[tail])
    ulp = np.where(rt > 0, 2.0 ** (np.floor(np.log2(np.maximum(rt, 1e-300))) - 7), 0.0)   # bf16 ulp at |ref|
    assert np.all(np.abs(gotf[tail] - ref[tail]) <= 1e-6 * np.abs(v[tail]) + ulp + 1e-30), desc


PACKED = [
    ("2d_g32_c8", L(2, 2, 32, 8, 8, (13, 15), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_NONE)),
    ("2d_g16_c8_k16_d2", L(2, 1, 16, 8, 16, (12, 17), (3, 3), (1, 1), (2, 2), (2, 2))),
    ("2d_g8_c16_k8_s2", L(2, 2, 8, 16, 8, (15, 13), (3, 3), (2, 2), (1, 1), (1, 1), CONV_EPI_BIAS)),
    ("1d_g4_c32_k40", L(1, 3, 4, 32, 40, (97,), (3,), (1,), (1,), (1,))),
    ("3d_g16_c8", L(3, 1, 16, 8, 8, (4, 7, 9), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), CONV_EPI_BIAS)),
]


@pytest.mark.parametrize("name,layer", PACKED, ids=[p[0] for p in PACKED])
def test_packed_small_groups_match_oracle_and_unpacked(name, layer):
    """Groups narrower than 64 channels run packed into block-diagonal super-groups; the
    same problem with packing disabled takes the cp.async path.  Both meet the bound, and
    on integer inputs both are exact."""
    x, w, b = make_inputs(layer, "bf16", 1200 + zlib.crc32(name.encode()) % 500)
    ref, S = oracle_full(layer, "bf16", x, w, b)
    a, da = run_gpu(layer, "bf16", x, w, b, guard=64)
    c, dc = run_gpu(layer, "bf16", x, w, b, env={"CONV_NO_PACK": 1})
    assert "pack=" in da and "pack=" not in dc
    assert_within("bf16", layer.epilogue, a, ref, S, da)
    assert_within("bf16", layer.epilogue, c, ref, S, dc)
    from dataclasses import replace
    li = replace(layer, epilogue=CONV_EPI_BIAS, bias_bound=0.05)     # integer sums are exact; GELU is not
    xi, wi, bi = make_inputs(li, "bf16", 1300, kind="int")
    refi, _ = oracle_full(li, "bf16", xi, wi, bi)
    ai, _ = run_gpu(li, "bf16", xi, wi, bi)
    assert np.array_equal(ai.reshape(-1), syn.f32_to_bf16_bits(refi.astype(np.float32))), da


SLAB = [
    ("2d_d1", "bf16", L(2, 2, 2, 64, 64, (14, 14), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_BIAS)),
    ("2d_d2_nopad", "bf16", L(2, 1, 2, 64, 48, (19, 17), (3, 3), (1, 1), (0, 0), (2, 2))),
    ("2d_wide_w", "bf16", L(2, 1, 1, 64, 64, (5, 300), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_NONE)),
    ("2d_5x3_c128", "bf16", L(2, 1, 1, 128, 96, (11, 23), (5, 3), (1, 1), (2, 1), (1, 1))),
    ("3d_d1", "bf16", L(3, 1, 2, 64, 64, (5, 9, 10), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), CONV_EPI_BIAS)),
    ("3d_d2", "bf16", L(3, 1, 1, 64, 32, (6, 11, 13), (3, 3, 3), (1, 1, 1), (1, 1, 1), (2, 2, 2), CONV_EPI_BIAS)),
    ("1d_k3_c80", "bf16", L(1, 2, 1, 80, 136, (517,), (3,), (1,), (1,), (1,))),
    ("1d_k5_d2", "bf16", L(1, 1, 1, 64, 64, (300,), (5,), (1,), (4,), (2,))),
    ("1d_k3_d8_aligned_windows", "bf16", L(1, 1, 1, 64, 64, (400,), (3,), (1,), (8,), (8,), CONV_EPI_NONE)),
    ("2d_aligned_windows", "bf16", L(2, 1, 1, 64, 64, (6, 16), (3, 3), (1, 1), (1, 8), (1, 8), CONV_EPI_NONE)),
    ("2d_map1_g2_c72", "bf16", L(2, 2, 2, 72, 40, (13, 21), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("2d_weight_reload_g3", "bf16", L(2, 8, 3, 64, 64, (30, 60), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_BIAS)),
    ("packed_g32_c8", "bf16", L(2, 1, 32, 8, 8, (13, 15), (3, 3), (1, 1), (1, 1), (2, 2), CONV_EPI_NONE)),
    ("1d_tf32_c80", "f32", L(1, 1, 1, 80, 384, (300,), (3,), (1,), (1,), (1,))),
    ("2d_tf32_g2_c32", "f32", L(2, 1, 2, 32, 36, (17, 19), (3, 3), (1, 1), (2, 2), (2, 2), CONV_EPI_BIAS)),
    ("3d_tf32_c64", "f32", L(3, 1, 1, 64, 40, (4, 7, 9), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), CONV_EPI_BIAS)),
]


@pytest.mark.parametrize("name,dtype,layer", SLAB, ids=[s[0] for s in SLAB])
def test_slab_mode_matches_oracle_and_per_tap(name, dtype, layer):
    """Stride-1 problems take the slab gather (one box per tile and input plane, taps as
    shifted windows); the same problem with per-tap boxes must meet the same bound."""
    x, w, b = make_inputs(layer, dtype, 1500 + zlib.crc32(name.encode()) % 500)
    ref, S = oracle_full(layer, dtype, x, w, b)
    # small problems would split K (which slab mode does not do): keep whole reductions
    a, da = run_gpu(layer, dtype, x, w, b, env={"CONV_FORCE_SPLITK": 1}, guard=64)
    c, dc = run_gpu(layer, dtype, x, w, b, env={"CONV_FORCE_GATHER": "tma"})
    assert "gather=tma-slab" in da and "gather=tma " in dc + " ", (da, dc)
    assert_within(dtype, layer.epilogue, a, ref, S, da)
    assert_within(dtype, layer.epilogue, c, ref, S, dc)


@pytest.mark.parametrize("bn", [32, 64, 128])
def test_slab_mode_every_tile_width(bn):
    layer = L(2, 1, 1, 64, 200, (9, 37), (3, 3), (1, 1), (1, 1), (1, 1))
    x, w, b = make_inputs(layer, "bf16", 1700 + bn)
    got, desc = run_gpu(layer, "bf16", x, w, b, env={"CONV_FORCE_BN": bn, "CONV_FORCE_SPLITK": 1},
                        guard=64)
    assert f"tile=128x{bn}" in desc and "tma-slab" in desc, desc
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, got, ref, S, desc)


@pytest.mark.parametrize("name", ["2d_d1", "3d_d2", "1d_tf32_c80", "2d_weight_reload_g3"])
def test_slab_mode_streamed_weights(name):
    """Slab mode with the weights streamed through a ring of stages instead of held resident."""
    dtype, layer = next((d, l) for n, d, l in SLAB if n == name)
    x, w, b = make_inputs(layer, dtype, 1800 + zlib.crc32(name.encode()) % 500)
    got, desc = run_gpu(layer, dtype, x, w, b, env={"CONV_FORCE_SPLITK": 1, "CONV_FORCE_SLAB_STREAM": 1}, guard=64)
    assert "tma-slab" in desc and "w " not in desc, desc
    ref, S = oracle_full(layer, dtype, x, w, b)
    assert_within(dtype, layer.epilogue, got, ref, S, desc)


@pytest.mark.parametrize("epi_warps", [8, 16])
@pytest.mark.parametrize("bn", [128, 256])
def test_per_tap_epilogue_widths(epi_warps, bn):
    """The per-tap kernel with 8 or 16 epilogue warps (2 or 4 per TMEM lane quarter), bias and
    GELU, several tiles per CTA and a ragged last tile."""
    layer = L(1, 3, 1, 128, 640, (1000,), (3,), (1,), (1,), (1,), CONV_EPI_BIAS_GELU)
    x, w, b = make_inputs(layer, "bf16", 1900 + epi_warps + bn)
    got, desc = run_gpu(layer, "bf16", x, w, b, env={"CONV_FORCE_EPI_WARPS": epi_warps, "CONV_FORCE_BN": bn,
                                                    "CONV_FORCE_SPLITK": 1, "CONV_FORCE_GATHER": "tma"}, guard=64)
    assert f"tile=128x{bn}" in desc and f"epi_warps={epi_warps}" in desc, desc
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, got, ref, S, desc)


PAIR_CASES = ["2d_d1", "2d_d2_nopad", "2d_5x3_c128", "3d_d2", "2d_map1_g2_c72", "packed_g32_c8",
              "2d_weight_reload_g3"]


@pytest.mark.parametrize("stream", [0, 1])
@pytest.mark.parametrize("name", PAIR_CASES)
def test_slab_tile_pairs(name, stream):
    """Slab units of two tiles stacked along H (two accumulators sharing one slab and one
    weight pass), with the last unit's second tile partly or wholly outside the output."""
    dtype, layer = next((d, l) for n, d, l in SLAB if n == name)
    x, w, b = make_inputs(layer, dtype, 2100 + zlib.crc32(name.encode()) % 500 + stream)
    env = {"CONV_FORCE_SPLITK": 1, "CONV_FORCE_SLAB_PAIR": 1, "CONV_FORCE_SLAB_STREAM": stream}
    got, desc = run_gpu(layer, dtype, x, w, b, env=env, guard=64)
    assert "tma-slab" in desc and "acc=2" in desc, desc
    ref, S = oracle_full(layer, dtype, x, w, b)
    assert_within(dtype, layer.epilogue, got, ref, S, desc)


@pytest.mark.parametrize("splits", [2, 4, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cluster_split_k_reduction_equals_the_reduction_kernel(splits, dtype):
    """Split-K partials summed inside a thread-block cluster through distributed shared
    memory, in split order, give bit for bit the output of the separate reduction kernel
    (which sums the same partials in the same order), and meet the oracle's bound."""
    layer = L(1, 1, 1, 512, 256, (700,), (3,), (2,), (1,), (1,), CONV_EPI_BIAS_GELU)
    x, w, b = make_inputs(layer, dtype, 2300 + splits)
    env = {"CONV_FORCE_SPLITK": splits, "CONV_FORCE_GATHER": "tma", "CONV_FORCE_BN": 64}
    a, da = run_gpu(layer, dtype, x, w, b, env=dict(env, CONV_FORCE_CLUSTER_RED=1), guard=64)
    c, dc = run_gpu(layer, dtype, x, w, b, env=dict(env, CONV_FORCE_CLUSTER_RED=0), guard=64)
    assert f"splits={splits}" in da and "reduce=cluster" in da, da
    assert "reduce=kernel" in dc, dc
    assert np.array_equal(a, c), "cluster and kernel reductions differ"
    ref, S = oracle_full(layer, dtype, x, w, b)
    assert_within(dtype, layer.epilogue, a, ref, S, da)


MC_CASES = [
    # odd number of M tiles (the last pair's second tile lies past the output), 256-wide N tiles
    ("1d_s2_odd_mt_bn256", L(1, 3, 1, 128, 256, (701,), (3,), (2,), (1,), (1,)),
     {"CONV_FORCE_BN": 256, "CONV_FORCE_SPLITK": 1}),
    # even number of M tiles, 128-wide N tiles, per-tap boxes at unit stride
    ("1d_s1_bn128", L(1, 2, 1, 64, 128, (500,), (3,), (1,), (1,), (1,), CONV_EPI_BIAS),
     {"CONV_FORCE_BN": 128, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_GATHER": "tma"}),
    # 2D tiles of several output rows, groups, a ragged N tile, 8 epilogue warps
    ("2d_s2_groups_bn128_ew8", L(2, 2, 2, 64, 200, (27, 33), (3, 3), (2, 2), (1, 1), (1, 1), CONV_EPI_GELU),
     {"CONV_FORCE_BN": 128, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_EPI_WARPS": 8}),
    # a long reduction (60 K blocks) as in the wide conv1d layer, batch 1
    ("1d_s2_c1280", L(1, 1, 1, 1280, 1280, (3000,), (3,), (2,), (1,), (1,)), {"CONV_FORCE_SPLITK": 1}),
    # no padding, two images, a ragged last tile per image, 8 epilogue warps
    ("1d_s2_pad0_n2", L(1, 2, 1, 384, 256, (1000,), (3,), (2,), (0,), (1,), CONV_EPI_BIAS),
     {"CONV_FORCE_BN": 256, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_EPI_WARPS": 8}),
    # two groups, GELU
    ("1d_s2_groups", L(1, 1, 2, 256, 256, (1200,), (3,), (2,), (1,), (1,), CONV_EPI_GELU),
     {"CONV_FORCE_BN": 256, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_EPI_WARPS": 8}),
    # padding 2, three channel blocks, an odd number of M tiles
    ("1d_s2_pad2_odd_mt", L(1, 1, 1, 192, 256, (640,), (3,), (2,), (2,), (1,), CONV_EPI_NONE),
     {"CONV_FORCE_BN": 256, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_EPI_WARPS": 8}),
    # 2D with a 1x3 filter at stride (1, 2): tiles of one output row on three rows
    ("2d_1x3_s12", L(2, 1, 1, 128, 256, (3, 512), (1, 3), (1, 2), (0, 1), (1, 1), CONV_EPI_BIAS_GELU),
     {"CONV_FORCE_BN": 256, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_EPI_WARPS": 8}),
]


@pytest.mark.parametrize("name,layer,env", MC_CASES, ids=[c[0] for c in MC_CASES])
def test_weight_multicast_pairs_are_bit_identical(name, layer, env):
    """CTA pairs that share each weight tile by multicast issue the same MMAs on the same data
    as single CTAs: the outputs are bit-identical, and within the bound of the oracle."""
    x, w, b = make_inputs(layer, "bf16", 900 + len(name))
    on, don = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_MC": 1}, guard=64)
    off, doff = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_MC": 0, "CONV_FORCE_PAIR": 0})
    assert "weights=multicast2" in don and "weights=" not in doff, (don, doff)
    assert np.array_equal(on, off), f"{name}: multicast result differs [{don}]"
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, on, ref, S, don)


@pytest.mark.parametrize("name,layer,env", MC_CASES, ids=[c[0] for c in MC_CASES])
def test_cta_pair_tiles_are_bit_identical(name, layer, env):
    """M = 256 tiles over a CTA pair (.cta_group::2 MMAs: each CTA holds its 128 rows of the
    activations and half of every weight tile) give the same bits as 128-row tiles on single
    CTAs, and meet the bound against the oracle."""
    x, w, b = make_inputs(layer, "bf16", 950 + len(name))
    on, don = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_PAIR": 1}, guard=64)
    off, doff = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_PAIR": 0})
    assert "cta_pair=m256" in don and "cta_pair" not in doff, (don, doff)
    assert np.array_equal(on, off), f"{name}: CTA-pair result differs [{don}]"
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, on, ref, S, don)


YSTORE_CASES = [
    # ragged last tile (Wo = 351: the last box is clipped at the end of the row), 16 epilogue warps
    ("1d_s2_ragged_bn256", L(1, 3, 1, 128, 256, (701,), (3,), (2,), (1,), (1,)),
     {"CONV_FORCE_BN": 256, "CONV_FORCE_SPLITK": 1}),
    # groups with K % 64 == 0, 8 epilogue warps (two 64-column chunks per warp)
    ("1d_groups_k128_ew8", L(1, 2, 2, 64, 128, (517,), (3,), (1,), (1,), (1,), CONV_EPI_BIAS),
     {"CONV_FORCE_BN": 128, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_GATHER": "tma", "CONV_FORCE_EPI_WARPS": 8}),
    # CTA pairs and weight multicast with tensor-map stores
    ("1d_pair_bn256", L(1, 3, 1, 128, 256, (701,), (3,), (2,), (1,), (1,), CONV_EPI_NONE),
     {"CONV_FORCE_BN": 256, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_EPI_WARPS": 8, "CONV_FORCE_PAIR": 1}),
    ("1d_mc_bn256", L(1, 3, 1, 128, 256, (701,), (3,), (2,), (1,), (1,)),
     {"CONV_FORCE_BN": 256, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_MC": 1}),
    # 2D problem with one-row tiles (Wo >= 128)
    ("2d_one_row_tiles", L(2, 1, 1, 64, 256, (3, 512), (3, 3), (1, 2), (1, 1), (1, 1)),
     {"CONV_FORCE_BN": 256, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_GATHER": "tma"}),
    # 32-column chunks (64-byte swizzle): 128-wide tiles with 16 epilogue warps, 64-wide tiles
    # with 8, and 128-wide CTA pairs with 16; K not a multiple of the tile width
    ("1d_bn128_ew16", L(1, 2, 1, 128, 320, (650,), (3,), (1,), (1,), (1,)),
     {"CONV_FORCE_BN": 128, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_GATHER": "tma", "CONV_FORCE_EPI_WARPS": 16}),
    ("1d_bn64_ew8", L(1, 2, 1, 128, 192, (650,), (3,), (1,), (1,), (1,), CONV_EPI_BIAS),
     {"CONV_FORCE_BN": 64, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_GATHER": "tma", "CONV_FORCE_EPI_WARPS": 8}),
    ("1d_pair_bn128_ew16", L(1, 3, 1, 128, 256, (701,), (3,), (2,), (1,), (1,)),
     {"CONV_FORCE_BN": 128, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_EPI_WARPS": 16, "CONV_FORCE_PAIR": 1}),
]


@pytest.mark.parametrize("name,layer,env", YSTORE_CASES, ids=[c[0] for c in YSTORE_CASES])
def test_tensor_map_stores_are_bit_identical(name, layer, env):
    """Epilogues that store y through a tensor map (one TMA box of 64 or 32 channels x 32 pixels
    per warp and chunk) write the same bits as per-lane stores, nothing outside y, and meet the
    bound against the oracle."""
    x, w, b = make_inputs(layer, "bf16", 970 + len(name))
    on, don = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_YSTORE": 1}, guard=4096)
    off, doff = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_YSTORE": 0})
    assert "store=tma" in don and "store=tma" not in doff, (don, doff)
    assert np.array_equal(on, off), f"{name}: tensor-map stores differ [{don}]"
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, on, ref, S, don)


SLAB_PAIR_CASES = [
    # resident weights, groups, bias + GELU
    ("2d_g2_c64_resident", L(2, 2, 2, 64, 64, (13, 21), (3, 3), (1, 1), (1, 1), (1, 1)), {}),
    # packed small groups (8 groups of 8 channels per 64-channel tile), dilation 2
    ("2d_g8_c8_packed_dil2", L(2, 2, 8, 8, 8, (15, 17), (3, 3), (1, 1), (2, 2), (2, 2), CONV_EPI_NONE), {}),
    # streamed weights over three input planes (3D)
    ("3d_streamed", L(3, 1, 2, 64, 64, (4, 20, 10), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), CONV_EPI_BIAS),
     {"CONV_FORCE_SLAB_STREAM": 1}),
    # an odd number of slab units (the last pair's second unit lies past the output), 32-wide N tiles
    ("2d_k32_odd_units", L(2, 1, 1, 64, 32, (15, 40), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_GELU), {}),
    # dilation 2 in 3D with a short weight ring
    ("3d_dil2_streamed", L(3, 1, 2, 64, 64, (6, 24, 56), (3, 3, 3), (1, 1, 1), (2, 2, 2), (2, 2, 2),
                           CONV_EPI_BIAS), {"CONV_FORCE_SLAB_STREAM": 1}),
    # dilation 2 in 3D on tiles of half the output width (27 of 54 columns, slab rows of 31
    # pixels), the plan the rules choose for the full-size 3D d2 layer
    ("3d_dil2_narrow", L(3, 1, 2, 64, 64, (6, 24, 56), (3, 3, 3), (1, 1, 1), (1, 1, 1), (2, 2, 2),
                         CONV_EPI_BIAS), {"CONV_FORCE_SLAB_BW": 27}),
    # 2D dilation 2, narrow tiles that do not divide the output width (20 + 20 + 10 of 50
    # columns), GELU, streamed weights
    ("2d_dil2_narrow_ragged", L(2, 2, 1, 64, 64, (33, 54), (3, 3), (1, 1), (1, 1), (2, 2), CONV_EPI_BIAS_GELU),
     {"CONV_FORCE_SLAB_BW": 20, "CONV_FORCE_SLAB_STREAM": 1}),
]


@pytest.mark.parametrize("name,layer,env", SLAB_PAIR_CASES, ids=[c[0] for c in SLAB_PAIR_CASES])
def test_slab_cta_pairs_are_bit_identical(name, layer, env):
    """Slab units on CTA pairs (each CTA its own slab and half of every weight tile, M = 256
    MMAs) give the same bits as the single-CTA slab kernel and meet the bound against the
    oracle."""
    env = {"CONV_FORCE_SLAB_PAIR": 1, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_BN": 64 if layer.K * (64 // max(layer.C, 1)
                                                                                           if layer.C < 64 else 1) >= 64
                                                                              else 32, **env}
    x, w, b = make_inputs(layer, "bf16", 990 + len(name))
    on, don = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_PAIR": 1}, guard=64)
    off, doff = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_PAIR": 0})
    assert "cta_pair=m256" in don and "gather=tma-slab" in don and "acc=2" in don, don
    assert "cta_pair" not in doff and "gather=tma-slab" in doff, doff
    assert np.array_equal(on, off), f"{name}: slab CTA-pair result differs [{don}]"
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, on, ref, S, don)


ONE_ACC_PAIR_CASES = [
    # 3D dilation 2 (the rules' plan for the 3D G=4 C=K=64 d2 shape, at a smaller size)
    ("3d_dil2", L(3, 1, 2, 64, 64, (6, 20, 56), (3, 3, 3), (1, 1, 1), (1, 1, 1), (2, 2, 2), CONV_EPI_BIAS), {}),
    # 2D, an odd number of slab units (the last pair's second unit lies past the output), GELU,
    # streamed weights
    ("2d_odd_units_gelu", L(2, 1, 1, 64, 64, (13, 40), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_GELU),
     {"CONV_FORCE_SLAB_STREAM": 1}),
    # 32-wide N tiles, two groups, resident weights
    ("2d_g2_k32", L(2, 2, 2, 64, 32, (20, 30), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_BIAS), {}),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,layer,env", ONE_ACC_PAIR_CASES, ids=[c[0] for c in ONE_ACC_PAIR_CASES])
def test_slab_cta_pairs_with_one_accumulator_are_bit_identical(name, layer, env):
    """Slab units of one accumulator per CTA on CTA pairs (M = 256 MMAs, one issuing warp) give
    the same bits as the single-CTA slab kernel with one accumulator, and meet the bound
    against the oracle."""
    env = {"CONV_FORCE_SLAB_PAIR": 0, "CONV_FORCE_SPLITK": 1, "CONV_FORCE_BN": 64 if layer.K >= 64 else 32, **env}
    x, w, b = make_inputs(layer, "bf16", 1990 + len(name))
    on, don = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_PAIR": 1}, guard=64)
    off, doff = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_PAIR": 0})
    assert "cta_pair=m256" in don and "gather=tma-slab" in don and "acc=1" in don, don
    assert "cta_pair" not in doff and "gather=tma-slab" in doff and "acc=1" in doff, doff
    assert np.array_equal(on, off), f"{name}: one-accumulator CTA-pair result differs [{don}]"
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, on, ref, S, don)
