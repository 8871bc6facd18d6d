"""GPU: the measured selector times every candidate plan of a problem on this device and
switches the plan to the fastest; the switched plan still matches the oracle element by
element, and the selector's table, saved and loaded again, gives new plans of the same
problem the same choice.  Every choice the selector may make is also checked against the
oracle directly (N tile x split factor x gather mode)."""
import numpy as np
import pytest

from convolution_forward_implicit_gb300 import binding as B
from convolution_forward_implicit_gb300.binding import CONV_BF16, CONV_EPI_BIAS, CONV_F32, ConvPlan
from convolution_forward_implicit_gb300.workloads import WORKLOADS
from tests.helpers import assert_within, from_device, has_bias, oracle_full, run_gpu, to_device
from tests.test_parity_gpu import L, make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    ("whisper_l1_bf16", "bf16", WORKLOADS["whisper_frontend_bf16"].layers[0]),
    ("whisper_l2_f32", "f32", WORKLOADS["whisper_frontend_f32"].layers[1]),
    ("2d_g8_c64", "bf16", L(2, 1, 8, 64, 64, (20, 24), (3, 3), (1, 1), (1, 1), (1, 1))),
    ("3d_g4_c64_d2", "bf16", L(3, 1, 4, 64, 64, (6, 10, 12), (3, 3, 3), (1, 1, 1), (2, 2, 2), (2, 2, 2),
                               CONV_EPI_BIAS)),
    ("2d_g32_c8", "bf16", L(2, 2, 32, 8, 8, (24, 20), (3, 3), (1, 1), (1, 1), (1, 1))),
]


@pytest.mark.parametrize("name,dtype,layer", CASES, ids=[c[0] for c in CASES])
def test_tuned_plan_matches_oracle_and_table_round_trips(name, dtype, layer, tmp_path):
    import torch
    code = CONV_BF16 if dtype == "bf16" else CONV_F32
    x, w, b = make_inputs(layer, dtype, 4100 + len(name))
    xd, wd = to_device(x, dtype), to_device(w, dtype)
    bd = to_device(b, dtype) if has_bias(layer.epilogue) else None
    B.conv_tune_table_clear()
    try:
        plan = ConvPlan(*layer.plan_args(code))
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        y = torch.empty(plan.y_shape(), dtype=tdt, device="cuda")
        desc = plan.tune(xd, wd, bd, y, iters=3)
        y.fill_(float("nan"))
        plan.forward(xd, bd, y)
        plan.check()
        torch.cuda.synchronize()
        ref, S = oracle_full(layer, dtype, x, w, b)
        assert_within(dtype, layer.epilogue, from_device(y.contiguous(), dtype).reshape(-1), ref, S,
                      f"{name} [{desc}]")
        plan.close()

        def new_desc():
            h = B.conv_plan_create(*layer.plan_args(code))
            d = B.conv_plan_describe(h)
            B.conv_plan_destroy(h)
            return d

        assert new_desc() == desc                  # later plans of the problem take the choice
        f = tmp_path / "table.txt"
        B.conv_tune_table_save(str(f))
        lines = f.read_text().splitlines()
        rows = [ln for ln in lines if not ln.startswith("#")]
        log = [ln.split("\t") for ln in lines if ln.startswith("#")]
        assert len(rows) == 1 and len(log) >= 2
        # the row records the fastest candidate's time, and that candidate is the plan taken
        us = {entry[2]: float(entry[1][3:]) for entry in log}
        assert desc in us and us[desc] == min(us.values())
        assert abs(float(rows[0].rsplit("us=", 1)[1]) - us[desc]) < 1e-3
        B.conv_tune_table_clear()
        B.conv_tune_table_load(str(f))
        assert new_desc() == desc
    finally:
        B.conv_tune_table_clear()


def test_tune_rejects_a_scratch_buffer_too_small_for_every_candidate():
    import torch
    layer = CASES[0][2]
    x, w, b = make_inputs(layer, "bf16", 4242)
    xd, wd, bd = to_device(x, "bf16"), to_device(w, "bf16"), to_device(b, "bf16")
    plan = ConvPlan(*layer.plan_args(CONV_BF16))
    before = plan.describe()
    y = torch.empty(plan.y_shape(), dtype=torch.bfloat16, device="cuda")
    scratch = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.ConvError) as e:
        B.conv_plan_tune(plan.handle, xd.data_ptr(), wd.data_ptr(), bd.data_ptr(), y.data_ptr(),
                         scratch.data_ptr(), 256, 2, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == B.CONV_ERR_WORKSPACE
    assert plan.describe() == before
    plan.close()


COMBO_LAYERS = {
    "bf16": L(2, 1, 2, 64, 136, (13, 37), (3, 3), (1, 1), (1, 1), (1, 1)),
    "f32": L(2, 1, 2, 32, 72, (11, 29), (3, 3), (1, 1), (1, 1), (1, 1)),
}


@pytest.mark.parametrize("gather", ["", "tma"])
@pytest.mark.parametrize("splits", [1, 2, 4])
@pytest.mark.parametrize("bn", [32, 64, 128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_every_selector_candidate_matches_oracle(dtype, bn, splits, gather):
    layer = COMBO_LAYERS[dtype]
    x, w, b = make_inputs(layer, dtype, 4300 + bn + splits)
    env = {"CONV_FORCE_BN": bn, "CONV_FORCE_SPLITK": splits}
    if gather:
        env["CONV_FORCE_GATHER"] = gather
    got, desc = run_gpu(layer, dtype, x, w, b, env=env, guard=64)
    assert f"x{bn} " in desc, desc
    ref, S = oracle_full(layer, dtype, x, w, b)
    assert_within(dtype, layer.epilogue, got, ref, S, desc)


def test_selector_tunes_a_unit_stride_backward_data_plan():
    """Backward data at unit stride runs the forward kernels on the transposed problem, so the
    selector can time its candidates too; the tuned plan still matches the oracle."""
    import torch
    import oracle
    from convolution_forward_implicit_gb300 import synthetic as syn
    from convolution_forward_implicit_gb300.binding import CONV_EPI_NONE
    from tests.helpers import geom_of
    layer = L(2, 1, 8, 64, 64, (20, 24), (3, 3), (1, 1), (1, 1), (1, 1), CONV_EPI_NONE)
    g = geom_of(layer)
    w = syn.gen_uniform_pm(4601, layer.w_shape(), layer.w_bound, "bf16")
    dy = syn.gen_normal(4602, g.y_shape(), "bf16")
    B.conv_tune_table_clear()
    try:
        plan = ConvPlan(*layer.plan_args(CONV_BF16), direction="bwd_data")
        assert "transposed_forward" in plan.describe()
        wd, dyd = to_device(w, "bf16"), to_device(dy, "bf16")
        dx = torch.empty(layer.x_shape(), dtype=torch.bfloat16, device="cuda")
        desc = plan.tune(dyd, wd, None, dx, iters=3)
        assert "transposed_forward" in desc
        dx.fill_(float("nan"))
        plan.backward_data(dyd, dx)
        plan.check()
        torch.cuda.synchronize()
        ref, S = oracle.conv_bwd_data(g, syn.as_f32(dy, "bf16"), syn.as_f32(w, "bf16"))
        assert_within("bf16", CONV_EPI_NONE, from_device(dx, "bf16").reshape(-1), ref.reshape(-1), S.reshape(-1),
                      desc)
        plan.close()
    finally:
        B.conv_tune_table_clear()
