"""Chained layers launched as programmatic dependents (conv_plan_set_overlap).

Each kernel may start before the previous one on the stream has finished; it must still
read x and write y only after that kernel completes.  The chain below reuses one buffer for
the first layer's output across iterations while the inputs alternate, so a kernel that
read its input too early (a read-after-write race) or overwrote the shared buffer while the
previous iteration's second layer still read it (write-after-read) would change some
iteration's final output.  Every iteration's output must equal, bit for bit, the same
layers run one by one without overlap (the kernels are deterministic), and that result is
checked against the oracle.
"""
import numpy as np
import pytest

from convolution_forward_implicit_gb300 import synthetic as syn
from convolution_forward_implicit_gb300.binding import ConvPlan
from convolution_forward_implicit_gb300.workloads import WORKLOADS, gen_inputs
from helpers import assert_within, from_device, oracle_full, to_device

pytestmark = pytest.mark.gpu

ITERS = 6


def _setup(name, overlap):
    import torch
    wl = WORKLOADS[name]
    x0, params = gen_inputs(wl)
    x1 = syn.gen_normal(4242, wl.layers[0].x_shape(), wl.dtype)
    plans, biases = [], []
    for li, layer in enumerate(wl.layers):
        w, b = params[li]
        p = ConvPlan(*layer.plan_args(wl.dtype_code))
        p.allocate()
        p.prepack(to_device(w, wl.dtype))
        p.set_overlap(overlap)
        plans.append(p)
        biases.append(to_device(b, wl.dtype) if b is not None else None)
    xs = [to_device(x0, wl.dtype), to_device(x1, wl.dtype)]
    tdt = plans[0].torch_dtype()
    mid = torch.empty(plans[0].y_shape(), dtype=tdt, device="cuda")
    outs = [torch.empty(plans[-1].y_shape(), dtype=tdt, device="cuda") for _ in range(ITERS)]
    return wl, (x0, x1), params, plans, biases, xs, mid, outs


def _chain(plans, biases, xs, mid, outs, i):
    plans[0].forward(xs[i % 2], biases[0], mid)
    plans[1].forward(mid, biases[1], outs[i])


@pytest.mark.parametrize("name", ["whisper_frontend_bf16", "whisper_frontend_f32"])
@pytest.mark.parametrize("mode", ["stream", "graph"])
def test_overlapped_chain_is_bit_identical_to_serial_and_meets_the_oracle(name, mode):
    import torch
    assert len(WORKLOADS[name].layers) == 2
    # serial reference: each input through both layers without overlap
    wl, xh, params, plans, biases, xs, mid, outs = _setup(name, overlap=False)
    ref_mid, ref_out = [], []
    for k in range(2):
        _chain(plans, biases, xs, mid, outs, k)
        torch.cuda.synchronize()
        ref_mid.append(from_device(mid.clone(), wl.dtype))
        ref_out.append(from_device(outs[k].clone(), wl.dtype))
    for p in plans:
        p.check()
        p.close()
    # overlapped chain, ITERS iterations back to back on one stream (or one graph)
    wl, xh, params, plans, biases, xs, mid, outs = _setup(name, overlap=True)
    descs = [p.describe() for p in plans]
    if mode == "stream":
        for i in range(ITERS):
            _chain(plans, biases, xs, mid, outs, i)
    else:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            _chain(plans, biases, xs, mid, outs, 0)   # warm-up outside the capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(ITERS):
                _chain(plans, biases, xs, mid, outs, i)
        for o in outs:
            o.zero_()
        g.replay()
    torch.cuda.synchronize()
    for p in plans:
        p.check()
    for i in range(ITERS):
        got = from_device(outs[i], wl.dtype)
        assert np.array_equal(got, ref_out[i % 2]), f"iteration {i} differs from the serial run ({descs})"
    # the serial result itself against the oracle, every output: layer 2 reads layer 1's GPU bits
    layer1, layer2 = wl.layers
    for k in range(2):
        w, b = params[1]
        cur = ref_mid[k].reshape(layer2.x_shape())
        ref, S = oracle_full(layer2, wl.dtype, cur, w, b)
        assert_within(wl.dtype, layer2.epilogue, ref_out[k], ref, S, f"{name} serial layer 2")
    for p in plans:
        p.close()
