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
