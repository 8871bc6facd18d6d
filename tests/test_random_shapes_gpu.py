"""Seeded random problems through all three passes on the GPU against the oracle: ndim 1-3,
groups, channel counts on and off the tensor-core multiples, stride, padding (also beyond
the filter's reach), dilation, every epilogue, fp32 and bf16.  Each case prints its plan on
failure, so a miss names the kernel that produced it."""
import dataclasses

import numpy as np
import pytest

import oracle
from convolution_forward_implicit_gb300 import synthetic as syn
from convolution_forward_implicit_gb300.binding import (CONV_EPI_BIAS, CONV_EPI_BIAS_GELU, CONV_EPI_GELU,
                                                        CONV_EPI_NONE)
from tests.helpers import assert_within, geom_of, oracle_full, run_gpu
from tests.test_backward_gpu import make_bwd_inputs, run_bwd_data, run_bwd_weight
from tests.test_parity_gpu import L, make_inputs

pytestmark = pytest.mark.gpu

EPIS = [CONV_EPI_NONE, CONV_EPI_BIAS, CONV_EPI_BIAS_GELU, CONV_EPI_GELU]


def random_layer(rng):
    ndim = int(rng.integers(1, 4))
    G = int(rng.choice([1, 1, 2, 3, 4, 8]))
    if rng.random() < 0.7:
        C = int(rng.choice([8, 16, 24, 32, 64, 72, 128]))
        K = int(rng.choice([8, 16, 32, 40, 64, 96, 136]))
    else:
        C = int(rng.integers(1, 20))
        K = int(rng.integers(1, 20))
    N = int(rng.integers(1, 3))
    spatial, filt, stride, pad, dil = [], [], [], [], []
    for a in range(ndim):
        f = int(rng.integers(1, 4 if ndim == 3 else 6))
        d = int(rng.integers(1, 3))
        s = int(rng.integers(1, 4))
        p = int(rng.integers(0, d * (f - 1) + 3))
        lo, hi = (6, 14) if ndim == 3 else ((8, 24) if ndim == 2 else (40, 400))
        i = int(rng.integers(max(lo, d * (f - 1) + 1 - 2 * p), hi))
        spatial.append(i); filt.append(f); stride.append(s); pad.append(p); dil.append(d)
    epi = int(rng.choice(EPIS))
    return L(ndim, N, G, C, K, spatial, filt, stride, pad, dil, epi)


CASES = [(seed, "bf16" if seed % 2 else "f32") for seed in range(120)]


@pytest.mark.parametrize("seed,dtype", CASES, ids=[f"{s}_{d}" for s, d in CASES])
def test_random_problem_all_passes(seed, dtype):
    rng = np.random.default_rng(70000 + seed)
    layer = random_layer(rng)
    g = geom_of(layer)
    what = f"seed {seed} {dtype} {layer}"
    # forward
    x, w, b = make_inputs(layer, dtype, 71000 + 10 * seed)
    got, desc = run_gpu(layer, dtype, x, w, b, guard=64)
    ref, S = oracle_full(layer, dtype, x, w, b)
    assert_within(dtype, layer.epilogue, got, ref, S, f"fwd {what} [{desc}]")
    # backward data and backward weight of the linear part
    lb = dataclasses.replace(layer, epilogue=CONV_EPI_NONE, bias_bound=None)
    x, w, dy = make_bwd_inputs(lb, dtype, 72000 + 10 * seed)
    got, desc = run_bwd_data(lb, dtype, dy, w)
    ref, S = oracle.conv_bwd_data(g, syn.as_f32(dy, dtype), syn.as_f32(w, dtype))
    assert_within(dtype, CONV_EPI_NONE, got, ref.reshape(-1), S.reshape(-1), f"dx {what} [{desc}]")
    got, desc = run_bwd_weight(lb, dtype, x, dy)
    ref, S = oracle.conv_bwd_weight(g, syn.as_f32(x, dtype), syn.as_f32(dy, dtype))
    assert_within(dtype, CONV_EPI_NONE, got, ref.reshape(-1), S.reshape(-1), f"dw {what} [{desc}]")
