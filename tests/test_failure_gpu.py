"""Failure detection on the GPU without a fault: a test hook makes the tensor-core kernel's MMA
role wait on a barrier that nothing completes.  Its bounded wait runs out (about one second),
the kernel raises the device error word, drains its copies and frees its tensor memory, and
conv_plan_check reports CONV_ERR_TIMEOUT; the context stays usable, so the next call on the
same data matches the oracle."""
import os
import time

import pytest

from convolution_forward_implicit_gb300 import binding as B
from convolution_forward_implicit_gb300.binding import CONV_BF16, ConvPlan
from tests.helpers import assert_within, has_bias, oracle_full, run_gpu, to_device
from tests.test_parity_gpu import L, make_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_is_reported_and_the_context_recovers():
    import torch
    layer = L(1, 1, 1, 64, 64, (300,), (3,), (1,), (1,), (1,))      # 3 CTAs, per-tap TMA kernel
    x, w, b = make_inputs(layer, "bf16", 31337)
    env = {"CONV_FORCE_GATHER": "tma", "CONV_FORCE_SPLITK": "1"}
    old = {k: os.environ.get(k) for k in (*env, "CONV_TEST_STALL")}
    os.environ.update(env)
    os.environ["CONV_TEST_STALL"] = "1"
    try:
        plan = ConvPlan(*layer.plan_args(CONV_BF16))
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    assert "gather=tma " in plan.describe() and "splits=1" in plan.describe(), plan.describe()
    plan.allocate()
    plan.prepack(to_device(w, "bf16"))
    xd, bd = to_device(x, "bf16"), to_device(b, "bf16")
    y = torch.empty(plan.y_shape(), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    t0 = time.time()
    plan.forward(xd, bd if has_bias(layer.epilogue) else None, y)
    with pytest.raises(B.ConvError) as e:
        plan.check()
    assert e.value.status == B.CONV_ERR_TIMEOUT
    assert time.time() - t0 >= 0.9           # it waited out its limit rather than finishing
    plan.check()                             # the error word was read and cleared
    plan.close()
    # the same problem without the hook, on the same context
    got, desc = run_gpu(layer, "bf16", x, w, b, env=env, guard=64)
    ref, S = oracle_full(layer, "bf16", x, w, b)
    assert_within("bf16", layer.epilogue, got, ref, S, desc)
