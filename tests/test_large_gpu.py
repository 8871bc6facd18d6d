"""Outputs beyond 2^31 elements: a conv1d of 20 million positions x 128 channels (x and y of
2.56e9 elements, 5.1 GB each in bf16), so every byte offset past the first 2^32 needs 64-bit
arithmetic in the kernels' addressing, TMA coordinates and stores.  The oracle checks sampled
outputs one by one (the first and last positions and random ones), from the receptive-field
windows of x copied back for just those positions; a sentinel band on each side of y shows
that nothing was written outside it."""
import numpy as np
import pytest

from convolution_forward_implicit_gb300 import synthetic as syn
from convolution_forward_implicit_gb300.binding import CONV_BF16, CONV_EPI_BIAS_GELU, ConvPlan
from convolution_forward_implicit_gb300.workloads import Layer
from oracle import Geom, conv_fwd
from tests.helpers import SENTINEL, assert_within, to_device

L_POS, C, K = 20_000_000, 128, 128
LAYER = Layer(1, 1, 1, C, K, (L_POS,), (3,), (1,), (1,), (1,), CONV_EPI_BIAS_GELU, 0.05)

CASES = [
    ("slab", {}),
    ("per_tap_tma_store", {"CONV_FORCE_GATHER": "tma"}),
    ("per_tap_lane_stores", {"CONV_FORCE_GATHER": "tma", "CONV_FORCE_YSTORE": 0}),
    ("per_tap_cta_pairs", {"CONV_FORCE_GATHER": "tma", "CONV_FORCE_PAIR": 1, "CONV_FORCE_BN": 128}),
]


def _sample_positions(rng):
    ends = np.concatenate([np.arange(0, 64), np.arange(L_POS - 64, L_POS)])
    mid = rng.integers(0, L_POS, 4096)
    # around 2^31 / K elements, where 32-bit element offsets would wrap
    wrap = (1 << 31) // K
    near = np.arange(wrap - 32, wrap + 32)
    return np.unique(np.concatenate([ends, mid, near]))


@pytest.mark.gpu
@pytest.mark.parametrize("name,env", CASES, ids=[c[0] for c in CASES])
def test_outputs_beyond_32_bit_element_offsets(name, env):
    import os
    import torch
    assert LAYER.N * L_POS * K > (1 << 31)
    old = {k: os.environ.get(k) for k in env}
    os.environ.update({k: str(v) for k, v in env.items()})
    try:
        plan = ConvPlan(*LAYER.plan_args(CONV_BF16))
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    try:
        plan.allocate()
        w = syn.gen_uniform_pm(4101, LAYER.w_shape(), LAYER.w_bound, "bf16")
        b = syn.gen_uniform_pm(4102, (K,), 0.05, "bf16")
        plan.prepack(to_device(w, "bf16"))
        bd = to_device(b, "bf16")
        gen = torch.Generator(device="cuda")
        gen.manual_seed(4100)
        x = torch.randn((1, L_POS, C), generator=gen, device="cuda", dtype=torch.bfloat16)
        guard = 4096
        n = L_POS * K
        buf = torch.full((n + 2 * guard,), SENTINEL, dtype=torch.bfloat16, device="cuda")
        y = buf[guard:guard + n].view(1, L_POS, K)
        plan.forward(x, bd, y)
        plan.check()
        torch.cuda.synchronize()
        sent = torch.cat([buf[:guard], buf[guard + n:]]).float()
        assert bool((sent == SENTINEL).all()), "kernel wrote outside its output"
        desc = plan.describe()

        pos = _sample_positions(np.random.default_rng(4103))
        # each sampled output's window of x (positions l-1, l, l+1; zeros in the padding) as one
        # sample of a 3-position conv without padding: the oracle gives exactly those outputs
        p = torch.as_tensor(pos, device="cuda")
        rows = torch.stack([p - 1, p, p + 1], dim=1)
        valid = (rows >= 0) & (rows < L_POS)
        win = x[0, rows.clamp(0, L_POS - 1)] * valid.unsqueeze(-1).to(torch.bfloat16)
        win_h = win.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        got = y[0, p].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        g = Geom(len(pos), 1, C, K, (3,), (3,), (1,), (0,), (1,))
        ref, S = conv_fwd(g, syn.as_f32(win_h, "bf16"), syn.as_f32(w, "bf16"), syn.as_f32(b, "bf16"), gelu=True)
        assert_within("bf16", CONV_EPI_BIAS_GELU, got.reshape(-1), ref.reshape(-1), S.reshape(-1),
                      f"{name} [{desc}]")
    finally:
        plan.close()
        torch.cuda.empty_cache()
