"""Pins that tie the CPU oracle to something other than itself (no GPU needed).

Each test names the fact it checks.  Together they are chosen so that a plausible
slip in the oracle (a wrong sign or index, swapped stride and dilation, a
transposed weight, a dropped bias, the tanh form of GELU, a wrong output-size
formula) fails at least one of them; ``test_pins_catch_planted_mistakes`` checks
exactly that on mutated copies of the oracle source.
"""
import ctypes
import json
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest
import scipy.signal
import scipy.special
import torch

import oracle
from convolution_forward_implicit_gb300 import synthetic as syn

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- helpers (test side)
def rand_problem(rng, ndim):
    G = int(rng.integers(1, 4))
    C = int(rng.integers(1, 6))
    K = int(rng.integers(1, 6))
    N = int(rng.integers(1, 3))
    spatial, filt, stride, pad, dil = [], [], [], [], []
    for _ in range(ndim):
        f = int(rng.integers(1, 4))
        d = int(rng.integers(1, 3))
        s = int(rng.integers(1, 3))
        p = int(rng.integers(0, 3))
        need = d * (f - 1) + 1 - 2 * p
        i = int(rng.integers(max(need, 1), max(need, 1) + (9 if ndim == 1 else 5)))
        spatial.append(i); filt.append(f); stride.append(s); pad.append(p); dil.append(d)
    return oracle.Geom(N, G, C, K, spatial, filt, stride, pad, dil)


def torch_conv_f64(g: oracle.Geom, x, w, bias):
    """torch.nn.functional.conv{1,2,3}d in float64 on the CPU, layouts permuted."""
    nd = g.ndim
    xs = np.asarray(x, np.float64).reshape(g.x_shape())           # N D H W G C
    ws = np.asarray(w, np.float64).reshape(g.w_shape())           # G K Z Y X C
    xs = xs.reshape(g.N, *g.spatial[3 - nd:], g.G * g.C)
    xt = torch.from_numpy(np.moveaxis(xs, -1, 1).copy())
    wt = ws.reshape(g.G * g.K, *g.filt[3 - nd:], g.C)
    wt = torch.from_numpy(np.moveaxis(wt, -1, 1).copy())
    bt = None if bias is None else torch.from_numpy(np.asarray(bias, np.float64).reshape(-1))
    fn = {1: torch.nn.functional.conv1d, 2: torch.nn.functional.conv2d, 3: torch.nn.functional.conv3d}[nd]
    yt = fn(xt, wt, bt, stride=g.stride[3 - nd:], padding=g.pad[3 - nd:], dilation=g.dilation[3 - nd:],
            groups=g.G)
    y = np.moveaxis(yt.numpy(), 1, -1)
    return y.reshape(g.y_shape())


def gen_case(g, seed, with_bias=True, dtype="f32"):
    x = syn.as_f32(syn.gen_normal(seed, g.x_shape(), dtype), dtype)
    w = syn.as_f32(syn.gen_uniform_pm(seed + 1, g.w_shape(), 0.7, dtype), dtype)
    b = syn.as_f32(syn.gen_uniform_pm(seed + 2, (g.G * g.K,), 0.5, dtype), dtype) if with_bias else None
    return x, w, b


# ---------------------------------------------------------------- pins
@pytest.mark.parametrize("ndim", [1, 2, 3])
def test_matches_torch_conv_f64(ndim):
    """Library routine: torch's fp64 CPU convolution (groups, stride, pad, dilation, bias)."""
    rng = np.random.default_rng(100 + ndim)
    for case in range(25 if ndim < 3 else 12):
        g = rand_problem(rng, ndim)
        x, w, b = gen_case(g, 1000 * ndim + case, with_bias=bool(case % 2))
        out, S = oracle.conv_fwd(g, x, w, b, gelu=False, nthreads=3)
        ref = torch_conv_f64(g, x, w, b)
        assert out.shape == ref.shape
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12 * (1.0 + S.max()))


@pytest.mark.parametrize("ndim", [1, 2, 3])
def test_gelu_epilogue_matches_torch_gelu(ndim):
    """Library routine: torch.nn.functional.gelu (exact erf form) applied to torch's conv."""
    rng = np.random.default_rng(200 + ndim)
    for case in range(8):
        g = rand_problem(rng, ndim)
        x, w, b = gen_case(g, 2000 * ndim + case)
        out, _ = oracle.conv_fwd(g, x, w, b, gelu=True)
        pre = torch.from_numpy(torch_conv_f64(g, x, w, b))
        ref = torch.nn.functional.gelu(pre, approximate="none").numpy()
        np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_absum_is_conv_of_magnitudes():
    """S = sum |x*w| equals the convolution of |x| with |w| (no bias), by torch."""
    rng = np.random.default_rng(7)
    for ndim in (1, 2, 3):
        for case in range(6):
            g = rand_problem(rng, ndim)
            x, w, b = gen_case(g, 300 * ndim + case)
            _, S = oracle.conv_fwd(g, x, w, b)
            ref = torch_conv_f64(g, np.abs(x), np.abs(w), None)
            np.testing.assert_allclose(S, ref, rtol=1e-13, atol=1e-13)


def test_pointwise_conv_is_matmul():
    """A 1x1 kernel with stride 1 and no padding is Y = X W^T per group (numpy matmul)."""
    g = oracle.Geom(2, 3, 5, 4, (3, 4, 5), (1, 1, 1), (1, 1, 1), (0, 0, 0), (1, 1, 1))
    x, w, b = gen_case(g, 42)
    out, _ = oracle.conv_fwd(g, x, w, b)
    X = x.reshape(-1, g.G, g.C).astype(np.float64)
    W = w.reshape(g.G, g.K, g.C).astype(np.float64)
    ref = np.einsum("mgc,gkc->mgk", X, W) + b.reshape(g.G, g.K)
    np.testing.assert_allclose(out.reshape(-1, g.G, g.K), ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("ndim", [1, 2, 3])
def test_single_channel_vs_scipy_correlate(ndim):
    """Textbook routine: scipy.signal.correlate on the zero-padded input, with the
    dilated kernel spread out with zeros and the result subsampled by the stride."""
    rng = np.random.default_rng(50 + ndim)
    for case in range(6):
        g0 = rand_problem(rng, ndim)
        g = oracle.Geom(1, 1, 1, 1, g0.spatial[3 - ndim:], g0.filt[3 - ndim:], g0.stride[3 - ndim:],
                        g0.pad[3 - ndim:], g0.dilation[3 - ndim:])
        x, w, _ = gen_case(g, 60 * ndim + case, with_bias=False)
        out, _ = oracle.conv_fwd(g, x, w, None)
        xi = x.reshape(g.spatial[3 - ndim:]).astype(np.float64)
        wi = w.reshape(g.filt[3 - ndim:]).astype(np.float64)
        xp = np.pad(xi, [(p, p) for p in g.pad[3 - ndim:]])
        wd = np.zeros([d * (f - 1) + 1 for f, d in zip(g.filt[3 - ndim:], g.dilation[3 - ndim:])])
        wd[tuple(slice(None, None, d) for d in g.dilation[3 - ndim:])] = wi
        full = scipy.signal.correlate(xp, wd, mode="valid", method="direct")
        ref = full[tuple(slice(None, None, s) for s in g.stride[3 - ndim:])]
        np.testing.assert_allclose(out.reshape(ref.shape), ref, rtol=1e-13, atol=1e-13)


def test_delta_kernel_identity_and_shift():
    """w[g,k,t,c] = [c == k][t == t0]: the centre tap gives the identity (pad keeps the
    size), an off-centre tap gives an exact shift with zeros at the border."""
    G, C = 2, 3
    g = oracle.Geom(1, G, C, C, (4, 5, 6), (3, 3, 3), (1, 1, 1), (2, 2, 2), (2, 2, 2))
    x, _, _ = gen_case(g, 9, with_bias=False)
    xs = x.reshape(g.x_shape())
    for t0 in [(1, 1, 1), (0, 2, 1), (2, 0, 0)]:
        w = np.zeros(g.w_shape(), np.float32)
        for gi in range(G):
            for k in range(C):
                w[gi, k, t0[0], t0[1], t0[2], k] = 1.0
        out, _ = oracle.conv_fwd(g, x, w, None)
        assert g.out_spatial == g.spatial
        shift = [(t - 1) * 2 for t in t0]              # tap offset relative to the centre, times dilation
        ref = np.zeros(g.y_shape())
        for od in range(4):
            for oh in range(5):
                for ow in range(6):
                    i = (od + shift[0], oh + shift[1], ow + shift[2])
                    if all(0 <= a < b for a, b in zip(i, g.spatial)):
                        ref[0, od, oh, ow] = xs[0, i[0], i[1], i[2]]
        assert np.array_equal(out, ref)


def test_integer_inputs_exact_against_brute_force():
    """Brute force on a tiny integer problem: python loops with exact integers."""
    g = oracle.Geom(2, 2, 3, 2, (3, 4), (2, 3), (2, 1), (1, 2), (1, 2))
    x = syn.gen_int(11, g.x_shape(), -3, 3, "f32")
    w = syn.gen_int(12, g.w_shape(), -3, 3, "f32")
    b = syn.gen_int(13, (g.G * g.K,), -2, 2, "f32")
    out, S = oracle.conv_fwd(g, x, w, b)
    xi = x.reshape(g.x_shape()).astype(np.int64)
    wi = w.reshape(g.w_shape()).astype(np.int64)
    bi = b.astype(np.int64).reshape(g.G, g.K)
    _, _, Ho, Wo = g.out_spatial[0], None, g.out_spatial[1], g.out_spatial[2]
    for n in range(g.N):
        for oh in range(Ho):
            for ow in range(Wo):
                for gi in range(g.G):
                    for k in range(g.K):
                        acc, s = int(bi[gi, k]), 0
                        for yy in range(g.filt[1]):
                            for xx in range(g.filt[2]):
                                ih = oh * g.stride[1] - g.pad[1] + yy * g.dilation[1]
                                iw = ow * g.stride[2] - g.pad[2] + xx * g.dilation[2]
                                if 0 <= ih < g.spatial[1] and 0 <= iw < g.spatial[2]:
                                    for c in range(g.C):
                                        p = int(xi[n, 0, ih, iw, gi, c]) * int(wi[gi, k, 0, yy, xx, c])
                                        acc += p
                                        s += abs(p)
                        assert out[n, 0, oh, ow, gi, k] == acc
                        assert S[n, 0, oh, ow, gi, k] == s


def test_gelu_closed_form_values():
    """GELU(v) = v * Phi(v): Phi(0) = 1/2, Phi(1) and Phi(-1) from the normal CDF table,
    limits v and 0, and scipy's ndtr everywhere else."""
    v = np.array([0.0, 1.0, -1.0, 2.0, -3.0, 12.0, -12.0, 0.5])
    got = oracle.gelu(v)
    assert got[0] == 0.0
    assert abs(got[1] - 0.8413447460685429) < 1e-15
    assert abs(got[2] + 0.15865525393145707) < 1e-15
    assert got[5] == 12.0 and abs(got[6]) < 1e-30
    np.testing.assert_allclose(got, v * scipy.special.ndtr(v), rtol=1e-14, atol=1e-16)
    tanh_form = 0.5 * v * (1 + np.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))
    assert np.max(np.abs(got - tanh_form)) > 1e-5        # the exact form, not the tanh approximation


def test_page_facts_whisper_frontend():
    """Values printed on the page: output lengths 3000 and 1500 (so pad = 1), 576k
    outputs and 664 M MACs for layer 2, and GFLOP/s that equal 2*MACs over the printed
    times within their rounding."""
    with open(os.path.join(HERE, "golden", "whisper_frontend_page_facts.json")) as f:
        facts = json.load(f)["facts"]
    for fct in facts:
        g = oracle.Geom(1, 1, fct["C_in"], fct["C_out"], (fct["L_in"],), (fct["kernel"],),
                        (fct["stride"],), (1,), (1,))
        assert g.out_spatial[2] == fct["L_out"]
        # pad 0 would not give the printed length
        g0 = oracle.Geom(1, 1, fct["C_in"], fct["C_out"], (fct["L_in"],), (fct["kernel"],),
                         (fct["stride"],), (0,), (1,))
        assert g0.out_spatial[2] != fct["L_out"]
        gflops = 2 * g.macs() / (fct["ms_printed"] * 1e-3) / 1e9
        assert abs(gflops - fct["gflops_printed"]) / fct["gflops_printed"] < 0.02
    l2 = facts[1]
    g = oracle.Geom(1, 1, 384, 384, (3000,), (3,), (2,), (1,), (1,))
    assert g.out_spatial[2] * 384 == l2["invocations"]
    assert 3 * 384 == l2["iterations_per_invocation_printed"]
    assert abs(g.macs() - l2["macs_printed_value"]) < 0.5e6


def test_invariants_linearity_zero_input_channel_permutation():
    rng = np.random.default_rng(3)
    g = rand_problem(rng, 2)
    x, w, b = gen_case(g, 77)
    out, _ = oracle.conv_fwd(g, x, w, b)
    out2, _ = oracle.conv_fwd(g, 2 * x, w, b)
    bb = b.reshape(g.G, g.K).astype(np.float64)
    assert np.array_equal(out2 - bb, 2 * (out - bb))          # power-of-two scaling is exact
    out0, _ = oracle.conv_fwd(g, np.zeros_like(x), w, b, gelu=True)
    assert np.array_equal(out0, np.broadcast_to(oracle.gelu(bb), out0.shape))
    perm = rng.permutation(g.K)
    wp = w.reshape(g.w_shape())[:, perm]
    outp, _ = oracle.conv_fwd(g, x, wp, b.reshape(g.G, g.K)[:, perm])
    assert np.array_equal(outp, out[..., perm])


def test_grouped_equals_independent_groups_and_conv1d_equals_h1():
    rng = np.random.default_rng(5)
    g = oracle.Geom(2, 3, 4, 2, (5, 7), (3, 2), (1, 2), (1, 0), (2, 1))
    x, w, b = gen_case(g, 5)
    out, _ = oracle.conv_fwd(g, x, w, b)
    xs, ws, bs = x.reshape(g.x_shape()), w.reshape(g.w_shape()), b.reshape(g.G, g.K)
    for gi in range(g.G):
        g1 = oracle.Geom(2, 1, 4, 2, (5, 7), (3, 2), (1, 2), (1, 0), (2, 1))
        o1, _ = oracle.conv_fwd(g1, xs[..., gi:gi + 1, :], ws[gi:gi + 1], bs[gi])
        assert np.array_equal(o1[..., 0, :], out[..., gi, :])
    g1d = oracle.Geom(1, 1, 3, 4, (11,), (3,), (2,), (1,), (2,))
    g2d = oracle.Geom(1, 1, 3, 4, (1, 11), (1, 3), (1, 2), (0, 1), (1, 2))
    x, w, b = gen_case(g1d, 6)
    a, _ = oracle.conv_fwd(g1d, x, w, b)
    c, _ = oracle.conv_fwd(g2d, x, w, b)
    assert np.array_equal(a, c)
    _ = rng


def test_points_match_full_output():
    rng = np.random.default_rng(8)
    g = rand_problem(rng, 3)
    x, w, b = gen_case(g, 8)
    out, S = oracle.conv_fwd(g, x, w, b, gelu=True)
    idx = np.array(np.unravel_index(np.arange(out.size), out.shape)).T
    pts, ps = oracle.conv_fwd_points(g, x, w, b, True, idx[:, [0, 1, 2, 3, 4, 5]])
    assert np.array_equal(pts, out.reshape(-1))
    assert np.array_equal(ps, S.reshape(-1))


# ---------------------------------------------------------------- the pins have teeth
MUTANTS = {
    "stride_for_dilation": ("int64_t iw = ow * g->sw - g->pw + xx * g->dw;\n                if",
                            "int64_t iw = ow * g->sw - g->pw + xx * g->sw;\n                if"),
    "pad_sign": ("int64_t ih = oh * g->sh - g->ph + y * g->dh;\n            if",
                 "int64_t ih = oh * g->sh + g->ph + y * g->dh;\n            if"),
    "transposed_weight_groups": ("const float* wp = w + ((((gi * g->K + k) * g->Z",
                                 "const float* wp = w + ((((k * g->G + gi) * g->Z"),
    "dropped_bias": ("if (bias) acc += (double)bias[gi * g->K + k];", "if (bias) acc += 0.0;"),
    "tanh_gelu": ("0.5 * v * (1.0 + erf(v / sqrt(2.0)))",
                  "0.5 * v * (1.0 + tanh(sqrt(2.0 / 3.141592653589793) * (v + 0.044715 * v * v * v)))"),
    "signed_absum": ("s += fabs(prod);\n                }\n            }\n        }\n    }\n    if (bias)",
                     "s += prod;\n                }\n            }\n        }\n    }\n    if (bias)"),
    "out_len": ("in + 2 * pad - dil * (filt - 1) - 1", "in + 2 * pad - dil * filt"),
    "flipped_kernel": ("const float* wp = w + ((((gi * g->K + k) * g->Z + z) * g->Y + y) * g->X + xx) * g->C;",
                       "const float* wp = w + ((((gi * g->K + k) * g->Z + z) * g->Y + y) * g->X + (g->X - 1 - xx)) * g->C;"),
}


def _check_all_pins(lib_path):
    """Re-run the library-routine pins against a given oracle build; True if all pass."""
    saved = oracle._lib
    try:
        oracle._lib = None
        lib = ctypes.CDLL(lib_path)
        orig_build = oracle.build
        oracle.build = lambda force=False: lib_path
        try:
            oracle._lib = None
            for fn in (lambda: test_matches_torch_conv_f64(1), lambda: test_matches_torch_conv_f64(2),
                       lambda: test_matches_torch_conv_f64(3), lambda: test_gelu_epilogue_matches_torch_gelu(1),
                       test_absum_is_conv_of_magnitudes, test_gelu_closed_form_values,
                       test_page_facts_whisper_frontend):
                fn()
            return True
        except Exception:        # an assertion, a shape mismatch or a rejected problem
            return False
        finally:
            oracle.build = orig_build
            del lib
    finally:
        oracle._lib = saved


def test_pins_catch_planted_mistakes():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "conv_oracle.c")).read()
    with tempfile.TemporaryDirectory() as td:
        for name, (old, new) in MUTANTS.items():
            assert src.count(old) == 1, name
            path = os.path.join(td, f"{name}.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = os.path.join(td, f"lib{name}.so")
            subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-shared", "-fPIC", "-o", so, path,
                                   "-lm", "-lpthread"])
            assert not _check_all_pins(so), f"mutant {name} passed every pin"


# ---------------------------------------------------------------- backward passes
def torch_conv_grads_f64(g: oracle.Geom, x, w, dy):
    """dx and dw of sum(conv(x, w) * dy) by torch autograd in float64 on the CPU (the
    library's own convolution backward), layouts permuted back to channels-last."""
    nd = g.ndim
    xs = np.asarray(x, np.float64).reshape(g.N, *g.spatial[3 - nd:], g.G * g.C)
    xt = torch.from_numpy(np.moveaxis(xs, -1, 1).copy()).requires_grad_(True)
    ws = np.asarray(w, np.float64).reshape(g.G * g.K, *g.filt[3 - nd:], g.C)
    wt = torch.from_numpy(np.moveaxis(ws, -1, 1).copy()).requires_grad_(True)
    fn = {1: torch.nn.functional.conv1d, 2: torch.nn.functional.conv2d, 3: torch.nn.functional.conv3d}[nd]
    yt = fn(xt, wt, None, stride=g.stride[3 - nd:], padding=g.pad[3 - nd:], dilation=g.dilation[3 - nd:],
            groups=g.G)
    dys = np.asarray(dy, np.float64).reshape(g.N, *g.out_spatial[3 - nd:], g.G * g.K)
    (yt * torch.from_numpy(np.moveaxis(dys, -1, 1).copy())).sum().backward()
    dx = np.moveaxis(xt.grad.numpy(), 1, -1).reshape(g.x_shape())
    dw = np.moveaxis(wt.grad.numpy(), 1, -1).reshape(g.w_shape())
    return dx, dw


def gen_dy(g, seed, dtype="f32"):
    return syn.as_f32(syn.gen_normal(seed, g.y_shape(), dtype), dtype)


def gen_int_case(g, seed):
    rng = np.random.default_rng(seed)
    x = rng.integers(-3, 4, g.x_shape()).astype(np.float32)
    w = rng.integers(-3, 4, g.w_shape()).astype(np.float32)
    dy = rng.integers(-3, 4, g.y_shape()).astype(np.float32)
    return x, w, dy


@pytest.mark.parametrize("ndim", [1, 2, 3])
def test_backward_matches_torch_autograd_f64(ndim):
    """Library routine: torch's fp64 convolution backward (groups, stride, pad, dilation)."""
    rng = np.random.default_rng(500 + ndim)
    for case in range(20 if ndim < 3 else 10):
        g = rand_problem(rng, ndim)
        x, w, _ = gen_case(g, 5000 * ndim + case, with_bias=False)
        dy = gen_dy(g, 5000 * ndim + case + 7)
        dx, Sx = oracle.conv_bwd_data(g, dy, w, nthreads=2)
        dw, Sw = oracle.conv_bwd_weight(g, x, dy, nthreads=3)
        rdx, rdw = torch_conv_grads_f64(g, x, w, dy)
        np.testing.assert_allclose(dx, rdx, rtol=0, atol=1e-12 * (1.0 + Sx.max()))
        np.testing.assert_allclose(dw, rdw, rtol=0, atol=1e-12 * (1.0 + Sw.max()))


def test_backward_absum_is_backward_of_magnitudes():
    """S of each backward element equals the same backward applied to |dy| and |w| (|x|), by torch."""
    rng = np.random.default_rng(510)
    for ndim in (1, 2, 3):
        for case in range(5):
            g = rand_problem(rng, ndim)
            x, w, _ = gen_case(g, 5100 + 10 * ndim + case, with_bias=False)
            dy = gen_dy(g, 5200 + 10 * ndim + case)
            _, Sx = oracle.conv_bwd_data(g, dy, w)
            _, Sw = oracle.conv_bwd_weight(g, x, dy)
            rdx, rdw = torch_conv_grads_f64(g, np.abs(x), np.abs(w), np.abs(dy))
            np.testing.assert_allclose(Sx, rdx, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(Sw, rdw, rtol=1e-13, atol=1e-13)


def test_backward_brute_force_impulse_responses():
    """On tiny integer problems, every dx element is <conv(e_i, w), dy> and every dw element
    is <conv(x, e_j), dy>, with the forward oracle run on unit impulses: exact."""
    rng = np.random.default_rng(520)
    for ndim in (1, 2, 3):
        for case in range(3):
            g = rand_problem(rng, ndim)
            x, w, dy = gen_int_case(g, 5300 + 10 * ndim + case)
            dx, _ = oracle.conv_bwd_data(g, dy, w)
            dw, _ = oracle.conv_bwd_weight(g, x, dy)
            bdx = np.empty(x.size)
            for i in range(x.size):
                e = np.zeros(x.size, np.float32)
                e[i] = 1.0
                bdx[i] = float((oracle.conv_fwd(g, e, w)[0] * dy).sum())
            bdw = np.empty(w.size)
            for j in range(w.size):
                e = np.zeros(w.size, np.float32)
                e[j] = 1.0
                bdw[j] = float((oracle.conv_fwd(g, x, e)[0] * dy).sum())
            assert np.array_equal(dx.reshape(-1), bdx), (ndim, case)
            assert np.array_equal(dw.reshape(-1), bdw), (ndim, case)


def test_backward_adjoint_identity_exact_on_integers():
    """<conv(x, w), dy> = <x, dx(dy, w)> = <w, dw(x, dy)>, exactly on integer inputs."""
    rng = np.random.default_rng(530)
    for ndim in (1, 2, 3):
        for case in range(10):
            g = rand_problem(rng, ndim)
            x, w, dy = gen_int_case(g, 5400 + 10 * ndim + case)
            y, _ = oracle.conv_fwd(g, x, w)
            lhs = float((y * dy).sum())
            assert lhs == float((oracle.conv_bwd_data(g, dy, w)[0] * x).sum())
            assert lhs == float((oracle.conv_bwd_weight(g, x, dy)[0] * w).sum())


def test_backward_pointwise_is_matmul():
    """1x1 kernel, stride 1, no padding: dx = dY W and dw = dY^T X per group (numpy)."""
    g = oracle.Geom(2, 3, 5, 4, (3, 4, 5), (1, 1, 1), (1, 1, 1), (0, 0, 0), (1, 1, 1))
    x, w, _ = gen_case(g, 43, with_bias=False)
    dy = gen_dy(g, 44)
    X = x.reshape(-1, g.G, g.C).astype(np.float64)
    W = w.reshape(g.G, g.K, g.C).astype(np.float64)
    DY = dy.reshape(-1, g.G, g.K).astype(np.float64)
    dx, _ = oracle.conv_bwd_data(g, dy, w)
    dw, _ = oracle.conv_bwd_weight(g, x, dy)
    np.testing.assert_allclose(dx.reshape(-1, g.G, g.C), np.einsum("mgk,gkc->mgc", DY, W), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dw.reshape(g.G, g.K, g.C), np.einsum("mgk,mgc->gkc", DY, X), rtol=1e-13,
                               atol=1e-13)


def test_stride1_backward_data_is_a_forward_conv_with_flipped_transposed_weights():
    """Textbook: at stride 1, dx = conv(dy, w') with w'[g,c,t,k] = w[g,k,F-1-t,c] and padding
    dil*(F-1) - pad (the transposed convolution)."""
    rng = np.random.default_rng(540)
    for ndim in (1, 2, 3):
        for case in range(4):
            g = rand_problem(rng, ndim)
            fl = g.filt[3 - ndim:]
            dl = g.dilation[3 - ndim:]
            pd = g.pad[3 - ndim:]
            if any(d * (f - 1) - p < 0 for f, d, p in zip(fl, dl, pd)):
                continue
            g = oracle.Geom(g.N, g.G, g.C, g.K, g.spatial[3 - ndim:], fl, (1,) * ndim, pd, dl)
            _, w, _ = gen_case(g, 5500 + 10 * ndim + case, with_bias=False)
            dy = gen_dy(g, 5600 + 10 * ndim + case)
            dx, _ = oracle.conv_bwd_data(g, dy, w)
            wf = w.reshape(g.w_shape())[:, :, ::-1, ::-1, ::-1, :]             # flip every tap axis
            wt = np.ascontiguousarray(np.moveaxis(wf, (1, 5), (5, 1)))          # G C Z Y X K
            gt = oracle.Geom(g.N, g.G, g.K, g.C, g.out_spatial[3 - ndim:], fl, (1,) * ndim,
                             [d * (f - 1) - p for f, d, p in zip(fl, dl, pd)], dl)
            assert gt.out_spatial == g.spatial
            ref, _ = oracle.conv_fwd(gt, dy, wt)
            np.testing.assert_allclose(dx, ref, rtol=1e-13, atol=1e-13)


def test_backward_points_match_full_output():
    rng = np.random.default_rng(550)
    g = rand_problem(rng, 3)
    x, w, _ = gen_case(g, 55, with_bias=False)
    dy = gen_dy(g, 56)
    for weight, (full, S) in ((False, oracle.conv_bwd_data(g, dy, w)), (True, oracle.conv_bwd_weight(g, x, dy))):
        idx = np.array(np.unravel_index(np.arange(full.size), full.shape)).T
        pts, ps = oracle.conv_bwd_points(g, x if weight else dy, dy if weight else w, weight, idx)
        assert np.array_equal(pts, full.reshape(-1)) and np.array_equal(ps, S.reshape(-1))


BWD_MUTANTS = {
    "dx_no_divisibility": ("if (num < 0 || num % s != 0) return -1;", "if (num < 0) return -1;"),
    "dx_pad_sign": ("int64_t num = i + p - t * d;", "int64_t num = i - p - t * d;"),
    "dx_flipped_tap": ("int64_t ow = source_pos(iw, xx, g->sw, g->pw, g->dw, g->Wo);",
                       "int64_t ow = source_pos(iw, g->X - 1 - xx, g->sw, g->pw, g->dw, g->Wo);"),
    "dx_weight_k_c_swapped": ("(double)w[((((gi * g->K + k) * g->Z + z) * g->Y + y) * g->X + xx) * g->C + c];",
                              "(double)w[((((gi * g->K + (k % g->C) % g->K) * g->Z + z) * g->Y + y) * g->X + xx) * g->C + (c % g->K) % g->C];"),
    "dw_dilation_for_stride": ("int64_t iw = ow * g->sw - g->pw + xx * g->dw;\n                    if (iw < 0",
                               "int64_t iw = ow * g->dw - g->pw + xx * g->sw;\n                    if (iw < 0"),
    "dw_skips_batch": ("for (int64_t n = 0; n < g->N; ++n)\n        for (int64_t od",
                       "for (int64_t n = 0; n < 1; ++n)\n        for (int64_t od"),
}


def _check_bwd_pins(lib_path):
    saved, orig_build = oracle._lib, oracle.build
    try:
        oracle._lib = None
        oracle.build = lambda force=False: lib_path
        for fn in (lambda: test_backward_matches_torch_autograd_f64(1),
                   lambda: test_backward_matches_torch_autograd_f64(2),
                   lambda: test_backward_matches_torch_autograd_f64(3)):
            fn()
        return True
    except Exception:
        return False
    finally:
        oracle.build = orig_build
        oracle._lib = saved


def test_backward_pins_catch_planted_mistakes():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "conv_oracle.c")).read()
    with tempfile.TemporaryDirectory() as td:
        for name, (old, new) in BWD_MUTANTS.items():
            assert src.count(old) == 1, name
            path = os.path.join(td, f"{name}.c")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = os.path.join(td, f"lib{name}.so")
            subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-shared", "-fPIC", "-o", so, path,
                                   "-lm", "-lpthread"])
            assert not _check_bwd_pins(so), f"mutant {name} passed every backward pin"
