"""Planner invariants over random geometries, for all three plan kinds (forward, backward
data, backward weight), on the host only: no call here launches a kernel.

Every plan the library accepts must agree with the size formula of the oracle, credit the
forward problem's 2*MACs, describe itself as key=value pairs, and size its buffers
consistently with the reduction it chose: a split reduction either sums its partials in a
thread-block cluster (every unit resident at once, no workspace) or through the reduction
kernel (one fp32 partial per split and output).  Geometries with an empty output are
rejected."""
import numpy as np
import pytest

import oracle
from convolution_forward_implicit_gb300 import binding as B

CREATE = {
    "fwd": lambda nd, N, G, C, K, sp, f, s, p, d, dt: B.conv_plan_create(nd, N, G, C, K, sp, f, s, p, d, dt,
                                                                         B.CONV_EPI_BIAS_GELU),
    "bwd_data": lambda *a: B.conv_bwd_data_plan_create(*a),
    "bwd_weight": lambda *a: B.conv_bwd_weight_plan_create(*a),
}


@pytest.fixture(scope="module")
def lib():
    from convolution_forward_implicit_gb300.build import build_library
    build_library()
    return B.load_library()


def _sm_count():
    """The SM count the library plans for: the device's, or 152 (one GB300) without a GPU."""
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152


def _geometry(rng):
    nd = int(rng.integers(1, 4))
    sp = [int(rng.integers(1, 3001))] if nd == 1 else [int(rng.integers(1, 33)) for _ in range(nd)]
    f = [int(rng.integers(1, 6)) for _ in range(nd)]
    s = [int(rng.integers(1, 5)) for _ in range(nd)]
    p = [int(rng.integers(0, 4)) for _ in range(nd)]
    d = [int(rng.integers(1, 4)) for _ in range(nd)]
    N = int(rng.choice([1, 2, 3, 8]))
    G = int(rng.choice([1, 1, 2, 3, 4, 8, 32]))
    C = int(rng.choice([1, 3, 8, 16, 24, 64, 80, 96, 128, 200, 384]))
    K = int(rng.choice([1, 5, 8, 16, 32, 64, 100, 384, 1280]))
    dt = B.CONV_BF16 if rng.integers(0, 2) else B.CONV_F32
    return nd, N, G, C, K, sp, f, s, p, d, dt


@pytest.mark.parametrize("kind", sorted(CREATE))
def test_random_plans_are_consistent(lib, kind):
    rng = np.random.default_rng({"fwd": 11, "bwd_data": 12, "bwd_weight": 13}[kind])
    accepted = 0
    sm_count = _sm_count()
    for _ in range(1500):
        nd, N, G, C, K, sp, f, s, p, d, dt = _geometry(rng)
        g = oracle.Geom(N, G, C, K, sp, f, s, p, d)
        if min(g.out_spatial) <= 0:
            with pytest.raises(B.ConvError) as e:
                CREATE[kind](nd, N, G, C, K, sp, f, s, p, d, dt)
            assert e.value.status == B.CONV_ERR_INVALID_ARG
            continue
        h = CREATE[kind](nd, N, G, C, K, sp, f, s, p, d, dt)
        accepted += 1
        try:
            where = f"{kind} nd={nd} N={N} G={G} C={C} K={K} in={sp} f={f} s={s} p={p} d={d} dtype={dt}"
            assert B.conv_plan_output_shape(h, nd) == g.out_spatial[3 - nd:], where
            assert B.conv_plan_flops(h) == 2.0 * g.macs(), where
            desc = B.conv_plan_describe(h)
            kv = dict(tok.split("=", 1) for tok in desc.split())
            assert all(kv.values()) and "variant" in kv, (where, desc)
            ws = B.conv_workspace_bytes(h)
            wb = B.conv_prepacked_weight_bytes(h)
            if kind == "bwd_weight":
                assert wb == 0, (where, desc)   # the weight is this pass's output: nothing to prepack
                continue
            assert wb > 0, (where, desc)
            if kv["variant"].startswith("tc"):
                assert wb % 16 == 0, (where, desc)
            if kind == "fwd" and kv["variant"].startswith("tc"):
                splits = int(kv["splits"])
                m_outputs = N * int(np.prod(g.out_spatial)) * G * K
                if splits == 1:
                    assert ws == 0, (where, desc)
                elif ws == 0:
                    # cluster sum: one unit per CTA, all resident at once
                    assert kv.get("reduce", "cluster") == "cluster", (where, desc)
                    assert int(kv["units"]) == int(kv["grid"]) <= sm_count, (where, desc)
                    assert splits <= 8 and 128 % splits == 0, (where, desc)
                else:
                    assert kv.get("reduce", "kernel") == "kernel", (where, desc)
                    assert ws == splits * m_outputs * 4, (where, desc)
        finally:
            B.conv_plan_destroy(h)
    assert accepted > 1000


FORCINGS = [
    {}, {"CONV_FORCE_PAIR": "1"}, {"CONV_FORCE_PAIR": "0"}, {"CONV_FORCE_GATHER": "tma"},
    {"CONV_FORCE_GATHER": "cp.async"}, {"CONV_FORCE_SLAB_PAIR": "1"}, {"CONV_FORCE_SLAB_STREAM": "1"},
    {"CONV_FORCE_MC": "1"}, {"CONV_FORCE_BN": "64"}, {"CONV_FORCE_BN": "256"}, {"CONV_FORCE_SPLITK": "3"},
    {"CONV_FORCE_EPI_WARPS": "16"}, {"CONV_NO_PACK": "1"}, {"CONV_FORCE_SLAB_BW": "20"},
    {"CONV_FORCE_PAIR": "1", "CONV_FORCE_BN": "128", "CONV_FORCE_GATHER": "tma"},
    {"CONV_FORCE_SLAB_PAIR": "1", "CONV_FORCE_PAIR": "1"},
]


def _expected_units(g, kv):
    """Work units a tensor-core forward plan implies: output tiles (BH x BW pixels of one output
    plane per unit where the plan names its pixels, else 128 GEMM rows), times the groups (packed
    groups counting once) and N tiles, halved along M (rounded up) on CTA pairs or weight-sharing
    clusters, times the K splits."""
    pack = int(kv.get("pack", "1"))
    bn = int(kv["tile"].split("x")[1])
    N = g.N
    do, ho, wo = (1,) * (3 - len(g.out_spatial)) + tuple(g.out_spatial)
    if "pixels" in kv:
        bh, bw = (int(v) for v in kv["pixels"].split("x"))
        num_mt = N * do * -(-ho // bh) * -(-wo // bw)
    else:
        num_mt = -(-(N * do * ho * wo) // 128)
    if kv.get("cta_pair") == "m256" or kv.get("weights") == "multicast2":
        num_mt = -(-num_mt // 2)
    return num_mt * (g.G // pack) * -(-(pack * g.K) // bn) * int(kv["splits"])


def test_tensor_core_plan_units_match_their_tiles(lib, monkeypatch):
    """Every tensor-core forward plan, under each of the planner's forcing variables, holds the
    unit count its tile shape implies and a grid that fits it: at most one CTA per SM and per
    unit, in whole clusters of two on CTA pairs.  (A plan whose rules tried a shape on the way
    and kept a stale count would give kernels units past the output, or leave some out.)"""
    rng = np.random.default_rng(14)
    sm_count = _sm_count()
    checked = 0
    for i in range(1200):
        nd, N, G, C, K, sp, f, s, p, d, dt = _geometry(rng)
        if nd > 1 and rng.random() < 0.5:
            # grouped layers of the slab and CTA-pair sizes: unit stride, 3-tap filters, C = K = 64
            sp = [int(rng.integers(4, 12))] + [int(rng.integers(14, 60)) for _ in range(nd - 1)]
            f, s, C, K, G = [3] * nd, [1] * nd, 64, int(rng.choice([32, 64])), int(rng.choice([1, 2, 4, 8]))
            dt = B.CONV_BF16
        g = oracle.Geom(N, G, C, K, sp, f, s, p, d)
        if min(g.out_spatial) <= 0:
            continue
        env = FORCINGS[i % len(FORCINGS)]
        with monkeypatch.context() as m:
            for k, v in env.items():
                m.setenv(k, v)
            try:
                h = CREATE["fwd"](nd, N, G, C, K, sp, f, s, p, d, dt)
            except B.ConvError:
                continue        # a forced choice the problem cannot take
        try:
            kv = dict(tok.split("=", 1) for tok in B.conv_plan_describe(h).split())
        finally:
            B.conv_plan_destroy(h)
        if not kv["variant"].startswith("tc"):
            continue
        where = f"nd={nd} N={N} G={G} C={C} K={K} in={sp} f={f} s={s} p={p} d={d} dtype={dt} env={env} {kv}"
        units, grid = int(kv["units"]), int(kv["grid"])
        assert units == _expected_units(g, kv), where
        assert 1 <= grid <= sm_count, where
        if kv.get("cta_pair") == "m256" or kv.get("weights") == "multicast2":
            assert grid % 2 == 0 and grid // 2 <= units, where
        else:
            assert grid <= units, where
        checked += 1
    assert checked > 600
