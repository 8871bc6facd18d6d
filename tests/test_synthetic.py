"""The seeded input generator: counter-form SplitMix64, Box-Muller, bf16 rounding."""
import numpy as np
import torch

from convolution_forward_implicit_gb300 import synthetic as syn

MASK = (1 << 64) - 1


def _scalar_splitmix(seed, n):
    out, state = [], seed & MASK
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & MASK
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
        out.append(z ^ (z >> 31))
    return out


def test_counter_form_equals_sequential_generator():
    for seed in (0, 1234567, syn.BASE_SEED):
        ref = _scalar_splitmix(seed, 40)
        got = syn.splitmix64(seed, 0, 40)
        assert [int(v) for v in got] == ref
        assert [int(v) for v in syn.splitmix64(seed, 17, 5)] == ref[17:22]


def test_bf16_rounding_matches_torch_rne():
    f = syn.normal(5, 100000).astype(np.float32) * np.float32(37.0)
    f = np.concatenate([f, np.array([1.00390625, 1.01171875, -1.00390625, 0.0, 3.0e38], np.float32)])
    ours = syn.f32_to_bf16_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(syn.bf16_bits_to_f32(ours), torch.from_numpy(f).to(torch.bfloat16).float().numpy())


def test_distributions():
    z = syn.normal(syn.BASE_SEED, 400000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    u = syn.gen_uniform_pm(3, (200000,), 0.25, "f32")
    assert u.min() >= -0.25 and u.max() <= 0.25 and abs(u.mean()) < 0.005
    i = syn.gen_int(4, (10000,), -3, 3, "bf16")
    assert set(np.unique(syn.bf16_bits_to_f32(i)).tolist()) == set(range(-3, 4))


def test_chunked_generation_is_seamless():
    old = syn._CHUNK
    try:
        a = syn.normal(9, 1001)
        syn._CHUNK = 64
        b = syn.normal(9, 1001)
    finally:
        syn._CHUNK = old
    assert np.array_equal(a, b)
