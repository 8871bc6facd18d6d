"""Host logic of the benchmark's JSON line, without a GPU: the kernel-source hash that keys
measured DRAM traffic, the lookup of that traffic in the committed ncu summaries, and the
roofline's choice of bound and fraction."""
import json

import pytest

import bench


def test_source_hash_ignores_comments_but_not_code():
    """Comment text and blank lines drop out; code and string literals stay."""
    a = 'int f(int x) {  // doubles x\n    /* block\n comment */\n    return 2 * x;\n}\nconst char* s = "a // b";\n'
    b = 'int f(int x) {\n    return 2 * x;\n}\n\nconst char* s = "a // b";\n'
    c = 'int f(int x) {\n    return 3 * x;\n}\nconst char* s = "a // b";\n'
    assert bench._strip_comments(a) == bench._strip_comments(b)
    assert bench._strip_comments(a) != bench._strip_comments(c)
    assert '"a // b"' in bench._strip_comments(a)      # string literals are kept whole


def test_traffic_lookup_needs_the_same_sources_and_plan(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k.md").write_text(
        "# summary\n"
        "traffic: 0123456789abcdef 1911424 variant=tc_bf16 gather=tma tile=128x64 splits=1\n"
        "traffic: fedcba9876543210 777 variant=tc_bf16 gather=tma tile=128x32 splits=1\n")
    (tmp_path / "profiles" / "raw.ncu-rep").write_text("traffic: 0123456789abcdef 5 variant=x\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0123456789abcdef")
    assert bench.measured_traffic("variant=tc_bf16 gather=tma tile=128x64 splits=1") == 1911424
    # another plan, the same plan measured on other sources, or a file that is not a summary
    assert bench.measured_traffic("variant=tc_bf16 gather=tma tile=128x64 splits=2") is None
    assert bench.measured_traffic("variant=tc_bf16 gather=tma tile=128x32 splits=1") is None
    assert bench.measured_traffic("variant=x") is None


class _Plan:
    def __init__(self, desc):
        self.desc = desc

    def describe(self):
        return self.desc


class _Layer:
    def __init__(self, flops, nbytes, desc):
        self.flops, self.nbytes, self.plan = flops, nbytes, _Plan(desc)

    def bytes_alg(self):
        return self.nbytes

    def name(self):
        return "L"


@pytest.fixture
def peaks(tmp_path, monkeypatch):
    p = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(p))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    return p


def test_roofline_takes_the_slower_of_pipe_and_hbm(peaks):
    # 1.85 GFLOP over 51.4 MB: 0.9 us on the bf16 pipe, 8.6 us at 6000 GB/s -> HBM-bound
    r = bench.roofline_for(_Layer(1.85e9, 51.4e6, "variant=tc_bf16 pack=8"), 0.025)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6000.0
    assert r["achieved"] == pytest.approx(51.4e6 / 25e-6 / 1e9, rel=1e-4)
    assert r["frac"] == pytest.approx(r["achieved"] / 6000.0, abs=1e-4)
    assert r["peak_source"].endswith("measured") and r["traffic"] is None
    # 177.6 GFLOP over 206 MB: tensor-bound against the measured bf16 peak
    r = bench.roofline_for(_Layer(177.6e9, 206e6, "variant=tc_bf16 gather=tma-slab"), 0.2)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 2000.0
    assert r["achieved"] == pytest.approx(177.6e9 / 0.2e-3 / 1e12, rel=1e-4)
    # 3xTF32: a third of the TF32 peak, itself the bf16 peak scaled by the nominal 1.1 / 2.25
    r = bench.roofline_for(_Layer(1.327e9, 8.68e6, "variant=tc_tf32x3 gather=tma"), 0.0225)
    assert r["peak"] == pytest.approx(2000.0 * 1.1 / 2.25 / 3, abs=0.01)
    # fp32 planes for the backward weight: six bf16 products per useful product
    r = bench.roofline_for(_Layer(1e12, 1e6, "variant=tc_bf16x3 direction=bwd_weight"), 10.0)
    assert r["peak"] == pytest.approx(2000.0 / 6, abs=0.01)
    # the FFMA kernel: plain ALU arithmetic
    r = bench.roofline_for(_Layer(1e11, 1e6, "variant=simt_f32"), 5.0)
    assert r["bound"] == "alu" and r["peak"] == pytest.approx(152 * 128 * 2 * 2070e6 / 1e12, abs=0.01)
