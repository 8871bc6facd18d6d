"""conv_fwd_static_scratch: the forward pass for callers that cannot allocate device memory
(a plugin or custom operator given only its input and output buffers, or a loop that must
not allocate after start-up).  Its split-K scratch is the library's own device array, so
the caller provides no workspace.  This file is collected last on purpose: if it fails, a
run that stops at the first failure has already run every other test."""
import os

import numpy as np
import pytest

from convolution_forward_implicit_gb300 import binding as B
from convolution_forward_implicit_gb300.workloads import WORKLOADS, Layer
from tests.helpers import assert_within, from_device, oracle_full, to_device

pytestmark = pytest.mark.gpu


def _plan(layer, dtype_code, env=None):
    old = {k: os.environ.get(k) for k in (env or {})}
    os.environ.update({k: str(v) for k, v in (env or {}).items()})
    try:
        return B.ConvPlan(*layer.plan_args(dtype_code))
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


SPLIT = Layer(1, 1, 1, 128, 128, (700,), (3,), (2,), (1,), (1,), B.CONV_EPI_BIAS_GELU, 0.05)
# (name, dtype, layer, plan overrides, whether the plan must use the array)
CASES = [
    ("whisper_l2_bf16", "bf16", WORKLOADS["whisper_frontend_bf16"].layers[1], None, False),
    ("whisper_l2_f32_cluster", "f32", WORKLOADS["whisper_frontend_f32"].layers[1], None, False),
    ("split2_bf16_cluster", "bf16", SPLIT, {"CONV_FORCE_SPLITK": 2}, False),
    ("unsplit_2d_bf16", "bf16", Layer(2, 1, 2, 32, 40, (19, 23), (3, 3), (1, 1), (1, 1), (1, 1), B.CONV_EPI_BIAS,
                                      0.05), {"CONV_FORCE_SPLITK": 1}, False),
    # split-K partial sums through the reduction kernel: these write and read the array
    ("split3_bf16", "bf16", SPLIT, {"CONV_FORCE_SPLITK": 3}, True),   # 3 splits cannot share out 128 rows
    ("split2_bf16_reduce_kernel", "bf16", SPLIT, {"CONV_FORCE_SPLITK": 2, "CONV_FORCE_CLUSTER_RED": 0}, True),
    ("whisper_l2_f32_reduce_kernel", "f32", WORKLOADS["whisper_frontend_f32"].layers[1],
     {"CONV_FORCE_CLUSTER_RED": 0}, True),
    ("simt_split4_f32", "f32", Layer(2, 1, 3, 12, 20, (11, 14), (3, 3), (1, 1), (1, 1), (1, 1), B.CONV_EPI_BIAS_GELU,
                                     0.05), {"CONV_FORCE_SIMT": 1, "CONV_FORCE_SPLITK": 4}, True),
]

# Run between the two calls of each case: a problem of another shape whose split-K partial
# sums overwrite the array, so the second call finds another problem's data there.
STALE = Layer(1, 2, 1, 64, 96, (900,), (3,), (1,), (1,), (1,), B.CONV_EPI_BIAS, 0.05)


def _stale_call():
    import torch
    from convolution_forward_implicit_gb300 import synthetic as syn
    plan = _plan(STALE, B.CONV_BF16, {"CONV_FORCE_SPLITK": 5, "CONV_FORCE_CLUSTER_RED": 0})
    assert 0 < B.conv_workspace_bytes(plan.handle) <= B.conv_static_scratch_bytes()
    x = to_device(syn.gen_normal(91, STALE.x_shape(), "bf16"), "bf16")
    w = to_device(syn.gen_uniform_pm(92, STALE.w_shape(), STALE.w_bound, "bf16"), "bf16")
    b = to_device(syn.gen_uniform_pm(93, (STALE.K,), 0.05, "bf16"), "bf16")
    wp = torch.empty(B.conv_prepacked_weight_bytes(plan.handle), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    B.conv_prepack_weights(plan.handle, w.data_ptr(), wp.data_ptr(), s)
    y = torch.empty(plan.y_shape(), dtype=torch.bfloat16, device="cuda")
    B.conv_fwd_static_scratch(plan.handle, x.data_ptr(), wp.data_ptr(), b.data_ptr(), y.data_ptr(), s)
    B.conv_plan_check(plan.handle, s)
    plan.close()


@pytest.mark.parametrize("name,dtype,layer,env,uses_array", CASES, ids=[c[0] for c in CASES])
def test_static_scratch_matches_conv_fwd_on_two_calls(name, dtype, layer, env, uses_array):
    import torch
    from convolution_forward_implicit_gb300 import synthetic as syn
    code = B.CONV_BF16 if dtype == "bf16" else B.CONV_F32
    x = syn.gen_normal(41, layer.x_shape(), dtype)
    w = syn.gen_uniform_pm(42, layer.w_shape(), layer.w_bound, dtype)
    b = syn.gen_uniform_pm(43, (layer.G * layer.K,), 0.05, dtype)
    xd, wd, bd = to_device(x, dtype), to_device(w, dtype), to_device(b, dtype)

    # the existing entry point, with a caller-allocated workspace
    ref_plan = _plan(layer, code, env)
    ref_plan.allocate()
    ref_plan.prepack(wd)
    y_ref = torch.empty(ref_plan.y_shape(), dtype=ref_plan.torch_dtype(), device="cuda")
    ref_plan.forward(xd, bd, y_ref)
    ref_plan.check()

    # the allocation-free entry point: same plan shape, no workspace attached
    plan = _plan(layer, code, env)
    assert plan.describe() == ref_plan.describe()
    need = B.conv_workspace_bytes(plan.handle)
    assert need <= B.conv_static_scratch_bytes()
    assert (need > 0) == uses_array, f"{name}: workspace {need} bytes [{plan.describe()}]"
    plan.w_packed = torch.empty(max(B.conv_prepacked_weight_bytes(plan.handle), 16), dtype=torch.uint8,
                                device="cuda")
    B.conv_prepack_weights(plan.handle, wd.data_ptr(), plan.w_packed.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    s = torch.cuda.current_stream().cuda_stream
    ref_out, S = oracle_full(layer, dtype, x, w, b)
    expected = from_device(y_ref, dtype)
    for call in range(2):
        if call == 1:
            _stale_call()
        y = torch.full(plan.y_shape(), 7.0, dtype=plan.torch_dtype(), device="cuda")
        B.conv_fwd_static_scratch(plan.handle, xd.data_ptr(), plan.w_packed.data_ptr(), bd.data_ptr(),
                                  y.data_ptr(), s)
        B.conv_plan_check(plan.handle, s)
        got = from_device(y, dtype)
        # within the bound of every other parity test, against the existing entry point's output
        assert_within(dtype, layer.epilogue, got, syn.as_f32(expected, dtype).astype(np.float64).reshape(-1),
                      S, f"{name} call {call}")
        assert_within(dtype, layer.epilogue, got, ref_out, S, f"{name} call {call} vs oracle")
    plan.close()
    ref_plan.close()


def test_static_scratch_rejects_plans_beyond_its_size():
    import torch
    layer = Layer(1, 8, 1, 128, 1280, (3000,), (3,), (1,), (1,), (1,), B.CONV_EPI_BIAS, 0.05)
    plan = _plan(layer, B.CONV_BF16, {"CONV_FORCE_SPLITK": 2})
    assert B.conv_workspace_bytes(plan.handle) > B.conv_static_scratch_bytes()
    buf = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.ConvError) as e:
        B.conv_fwd_static_scratch(plan.handle, buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert e.value.status == B.CONV_ERR_WORKSPACE
    plan.close()
