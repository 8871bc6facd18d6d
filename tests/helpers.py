"""Shared test helpers: run one layer through the C-ABI on the GPU, run the oracle on the
same inputs, and compare under the per-element bound.

Tolerance (the bound the conv path must meet, per output element):
    |gpu - oracle| <= L * rel * S + u_out * |oracle| + g * B
  rel   = 1e-5 for fp32 I/O, 8e-3 for bf16 I/O (fp32 accumulation);
  S     = sum |x*w| over the receptive field (fp64, from the oracle);
  L     = 1.13 when a GELU follows (a bound on the slope of x*Phi(x)), else 1;
  u_out = unit roundoff of the output type (2^-24 fp32, 2^-8 bf16): the one round-to-
          nearest-even of the stored result, which S does not scale (the bias is outside
          the sum); the fp32 bias add itself costs 2^-24 relative, inside rel * S for
          bf16 and inside the same term for fp32;
  g * B = with a GELU only: the erf-GELU's own evaluation error in fp32 (below 9.5e-7 |v|,
          g = 1e-6) on the bias part of the pre-activation v (B = 0.05, the bound of the test
          biases), which S does not scale either: it is all that is left where every tap of
          an output falls in the padding (S = 0, output GELU(bias)).
"""
from __future__ import annotations

import numpy as np

import oracle
from convolution_forward_implicit_gb300 import synthetic as syn
from convolution_forward_implicit_gb300.binding import (CONV_BF16, CONV_EPI_BIAS_GELU, CONV_EPI_GELU, CONV_F32,
                                                        ConvPlan)

GELU_LIPSCHITZ = 1.13
SENTINEL = -12288.0      # exact in fp32 and bf16; never produced by the test inputs' scale


def rel_for(dtype: str) -> float:
    return 1e-5 if dtype == "f32" else 8e-3


def uout_for(dtype: str) -> float:
    return 2.0 ** -24 if dtype == "f32" else 2.0 ** -8


GELU_EVAL = 1e-6          # erf-GELU evaluation error bound in fp32, relative to |pre-activation|
BIAS_BOUND = 0.05         # |bias| of the test inputs


def tolerance(dtype, epilogue, ref, S):
    gelu = epilogue in (CONV_EPI_BIAS_GELU, CONV_EPI_GELU)
    L = GELU_LIPSCHITZ if gelu else 1.0
    return (L * rel_for(dtype) * S + uout_for(dtype) * np.abs(ref) +
            (GELU_EVAL * BIAS_BOUND if gelu else 0.0) + 1e-30)


def to_device(a: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def from_device(t, dtype: str) -> np.ndarray:
    """Storage array back on the host (float32, or uint16 bf16 bits)."""
    import torch
    if dtype == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.float().cpu().numpy()


def geom_of(layer) -> oracle.Geom:
    return oracle.Geom(layer.N, layer.G, layer.C, layer.K, layer.spatial, layer.filter, layer.stride, layer.pad,
                       layer.dilation)


def has_bias(epilogue) -> bool:
    from convolution_forward_implicit_gb300.binding import CONV_EPI_BIAS
    return epilogue in (CONV_EPI_BIAS, CONV_EPI_BIAS_GELU)


def run_gpu(layer, dtype: str, x, w, b, env=None, stream=None, guard=0):
    """One conv_fwd through the C-ABI.  Returns (storage output, plan description).
    With guard > 0 the output sits inside a buffer with `guard` sentinel elements on each
    side, and the sentinels are checked afterwards."""
    import os
    import torch
    code = CONV_BF16 if dtype == "bf16" else CONV_F32
    old = {}
    for k, v in (env or {}).items():
        old[k] = os.environ.get(k)
        os.environ[k] = str(v)
    try:
        plan = ConvPlan(*layer.plan_args(code))
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    plan.allocate()
    xd, wd = to_device(x, dtype), to_device(w, dtype)
    bd = to_device(b, dtype) if b is not None else None
    plan.prepack(wd)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    n = int(np.prod(plan.y_shape()))
    if guard:
        buf = torch.full((n + 2 * guard,), SENTINEL, dtype=tdt, device="cuda")
        buf = buf.view(-1)
        # keep the 16-byte alignment of the output start
        y = buf[guard:guard + n].view(plan.y_shape())
    else:
        y = torch.empty(plan.y_shape(), dtype=tdt, device="cuda")
    plan.forward(xd, bd if has_bias(layer.epilogue) else None, y)
    plan.check()
    torch.cuda.synchronize()
    if guard:
        sent = torch.cat([buf[:guard], buf[guard + n:]]).float()
        assert bool((sent == SENTINEL).all()), "kernel wrote outside its output"
    desc = plan.describe()
    out = from_device(y.contiguous(), dtype)
    plan.close()
    return out, desc


def oracle_full(layer, dtype, x, w, b):
    g = geom_of(layer)
    gelu = layer.epilogue in (CONV_EPI_BIAS_GELU, CONV_EPI_GELU)
    bb = syn.as_f32(b, dtype) if (b is not None and has_bias(layer.epilogue)) else None
    ref, S = oracle.conv_fwd(g, syn.as_f32(x, dtype), syn.as_f32(w, dtype), bb, gelu=gelu)
    return ref.reshape(-1), S.reshape(-1)


def assert_within(dtype, epilogue, got_storage, ref, S, what="", stats=None):
    """Checks every element against the bound above; returns (max err / bound, cosine).  With
    a dict as stats it also records there the largest ratio against the bare rel * S term
    alone (the stated bound before the output rounding and GELU terms) over the elements with
    S > 0, and how many elements were compared."""
    got = syn.as_f32(got_storage, dtype).astype(np.float64).reshape(-1)
    tol = tolerance(dtype, epilogue, ref, S)
    err = np.abs(got - ref)
    bad = np.nonzero(~(err <= tol))[0]
    if len(bad):
        i = bad[np.argmax(err[bad] / tol[bad])]
        raise AssertionError(f"{what}: {len(bad)}/{len(ref)} outside bound; worst at {i}: gpu={got[i]!r} "
                             f"oracle={ref[i]!r} S={S[i]!r} tol={tol[i]!r}")
    ratio = float(np.max(err / tol)) if len(err) else 0.0
    cos = float(np.dot(got, ref) / (np.linalg.norm(got) * np.linalg.norm(ref) + 1e-300))
    if stats is not None:
        pos = S > 0
        stats["bare_ratio"] = float(np.max(err[pos] / (rel_for(dtype) * S[pos]))) if pos.any() else 0.0
        stats["elements"] = int(len(ref))
    return ratio, cos
