"""Seeded random bf16 problems run on CTA pairs (.cta_group::2: per-tap M = 256 tiles, and slab
units with tile pairs or one accumulator, at the rules' slab width or a narrower one) and on
single CTAs with the same tiles: the two must give the same bits (every output is one sum in the
same order, whichever CTA holds its accumulator), and the pair's result meets the bound against
the oracle.  Shapes span several tiles with ragged edges, groups, padding and dilation."""
import numpy as np
import pytest

from convolution_forward_implicit_gb300.binding import (CONV_EPI_BIAS, CONV_EPI_BIAS_GELU, CONV_EPI_GELU,
                                                        CONV_EPI_NONE)
from tests.helpers import assert_within, oracle_full, run_gpu
from tests.test_parity_gpu import L, make_inputs

pytestmark = pytest.mark.gpu

EPIS = [CONV_EPI_NONE, CONV_EPI_BIAS, CONV_EPI_BIAS_GELU, CONV_EPI_GELU]


def random_pair_case(rng):
    """A layer and the variables that plan it as a slab (stride 1) or per-tap pair."""
    ndim = int(rng.integers(2, 4))
    slab = rng.random() < 0.6
    G = int(rng.choice([1, 2, 4]))
    C = int(rng.choice([64, 128])) if not slab else 64
    K = int(rng.choice([32, 64])) if slab else int(rng.choice([128, 256, 200]))
    N = int(rng.integers(1, 3))
    spatial, filt, stride, pad, dil = [], [], [], [], []
    for a in range(ndim):
        f = 3
        d = int(rng.integers(1, 3))
        s = 1 if slab else int(rng.integers(1, 3))
        p = int(rng.integers(0, d + 1))
        lo, hi = ((4, 8) if a == 0 else (14, 30)) if ndim == 3 else (12, 40)
        i = int(rng.integers(max(lo, d * (f - 1) + 1), hi))
        spatial.append(i); filt.append(f); stride.append(s); pad.append(p); dil.append(d)
    epi = int(rng.choice(EPIS))
    layer = L(ndim, N, G, C, K, spatial, filt, stride, pad, dil, epi)
    env = {"CONV_FORCE_SPLITK": 1}
    if slab:
        env["CONV_FORCE_BN"] = K
        env["CONV_FORCE_SLAB_PAIR"] = int(rng.integers(0, 2))
        if rng.random() < 0.5:
            env["CONV_FORCE_SLAB_STREAM"] = 1
        if rng.random() < 0.4:
            env["CONV_FORCE_SLAB_BW"] = int(rng.integers(8, 40))
    else:
        env["CONV_FORCE_BN"] = 256 if K > 128 else 128
        env["CONV_FORCE_GATHER"] = "tma"
        env["CONV_FORCE_EPI_WARPS"] = int(rng.choice([8, 16]))
    return layer, env, slab


CASES = list(range(40))


@pytest.mark.parametrize("seed", CASES)
def test_random_cta_pair_problem_is_bit_identical(seed):
    rng = np.random.default_rng(91000 + seed)
    layer, env, slab = random_pair_case(rng)
    x, w, b = make_inputs(layer, "bf16", 92000 + 10 * seed)
    on, don = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_PAIR": 1}, guard=64)
    off, doff = run_gpu(layer, "bf16", x, w, b, env={**env, "CONV_FORCE_PAIR": 0})
    what = f"seed {seed} {layer} {env}"
    assert "cta_pair=m256" in don and "cta_pair" not in doff, (what, don, doff)
    assert ("gather=tma-slab" in don) == slab, (what, don)
    assert np.array_equal(on, off), f"{what}: CTA-pair result differs [{don}] vs [{doff}]"
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, on, ref, S, f"{what} [{don}]")
