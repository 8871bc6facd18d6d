"""Host-side checks of the C-ABI library that need no GPU: it loads, exports every symbol
include/conv.h declares, and its plan logic (validation, output shape, FLOP count,
variant choice, argument checks of conv_fwd) behaves as documented.  No call here
launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from convolution_forward_implicit_gb300 import binding as B
from convolution_forward_implicit_gb300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from convolution_forward_implicit_gb300.build import build_library
    build_library()
    return B.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "conv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_][a-z_0-9]*\**\s+\**(conv_[a-z_0-9]+)\s*\(", src, re.M)))


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B.EXPORTED)


def test_status_strings(lib):
    for code in range(7):
        s = B.conv_status_string(code)
        assert s.startswith("CONV_") and "UNKNOWN" not in s
    assert B.conv_status_string(99) == "CONV_ERR_UNKNOWN"


def plan(ndim=1, N=1, G=1, C=8, K=8, spatial=(10,), filt=(3,), stride=(1,), pad=(1,), dil=(1,), dtype=B.CONV_BF16,
         epi=B.CONV_EPI_BIAS):
    return B.conv_plan_create(ndim, N, G, C, K, spatial, filt, stride, pad, dil, dtype, epi)


@pytest.mark.parametrize("kw", [dict(ndim=0), dict(ndim=4, spatial=(1, 1, 1, 1), filt=(1,) * 4, stride=(1,) * 4,
                                                     pad=(0,) * 4, dil=(1,) * 4),
                                dict(N=0), dict(G=0), dict(C=0), dict(K=-1), dict(stride=(0,)), dict(pad=(-1,)),
                                dict(dil=(0,)), dict(spatial=(0,)), dict(filt=(0,)),
                                dict(spatial=(2,), filt=(5,), pad=(0,)),           # empty output
                                dict(dtype=7), dict(epi=9)])
def test_plan_rejects_invalid_arguments(lib, kw):
    with pytest.raises(B.ConvError) as e:
        plan(**kw)
    assert e.value.status == B.CONV_ERR_INVALID_ARG


def test_plan_rejects_sizes_beyond_32_bit_indexing(lib):
    with pytest.raises(B.ConvError) as e:
        plan(N=1 << 20, spatial=(1 << 12,))
    assert e.value.status == B.CONV_ERR_UNSUPPORTED


def test_output_shape_and_flops_agree_with_the_oracle(lib):
    rng = np.random.default_rng(0)
    for _ in range(200):
        nd = int(rng.integers(1, 4))
        sp = [int(rng.integers(1, 40)) for _ in range(nd)]
        f = [int(rng.integers(1, 6)) for _ in range(nd)]
        s = [int(rng.integers(1, 4)) for _ in range(nd)]
        p = [int(rng.integers(0, 4)) for _ in range(nd)]
        d = [int(rng.integers(1, 4)) for _ in range(nd)]
        G, C, K, N = (int(rng.integers(1, 5)), int(rng.integers(1, 40)), int(rng.integers(1, 40)),
                      int(rng.integers(1, 4)))
        g = oracle.Geom(N, G, C, K, sp, f, s, p, d)
        empty = min(g.out_spatial) <= 0
        dtype = B.CONV_BF16 if rng.integers(0, 2) else B.CONV_F32
        if empty:
            with pytest.raises(B.ConvError):
                B.conv_plan_create(nd, N, G, C, K, sp, f, s, p, d, dtype, B.CONV_EPI_NONE)
            continue
        h = B.conv_plan_create(nd, N, G, C, K, sp, f, s, p, d, dtype, B.CONV_EPI_NONE)
        try:
            assert B.conv_plan_output_shape(h, nd) == g.out_spatial[3 - nd:]
            assert B.conv_plan_flops(h) == 2.0 * g.macs()
            desc = B.conv_plan_describe(h)
            tf32_ok = (C % 4 == 0 and K % 4 == 0 and C >= 32 and max(s) <= 8 and
                       (C % 32 == 0 or G == 1 or nd <= 2))
            if dtype == B.CONV_BF16 and C % 8 == 0 and K % 8 == 0:
                assert "variant=tc_bf16" in desc
            elif dtype == B.CONV_F32 and tf32_ok:
                assert "variant=tc_tf32x3" in desc
            else:
                assert "variant=simt" in desc
            assert B.conv_prepacked_weight_bytes(h) % 16 == 0 or "simt" in desc
            assert B.conv_prepacked_weight_bytes(h) > 0
        finally:
            B.conv_plan_destroy(h)


def test_workloads_plan_and_report_page_output_lengths(lib):
    """The Whisper layers give 3000 and 1500 outputs, as printed on the page."""
    wl = WORKLOADS["whisper_frontend_bf16"]
    outs = []
    for layer in wl.layers:
        h = B.conv_plan_create(*layer.plan_args(B.CONV_BF16))
        outs.append(B.conv_plan_output_shape(h, 1)[0])
        B.conv_plan_destroy(h)
    assert outs == [3000, 1500]
    for wl in WORKLOADS.values():
        for layer in wl.layers:
            h = B.conv_plan_create(*layer.plan_args(wl.dtype_code))
            assert B.conv_plan_describe(h)
            B.conv_plan_destroy(h)


def test_split_k_plan_needs_a_workspace(lib):
    os.environ["CONV_FORCE_SPLITK"] = "3"
    try:
        h = plan(C=128, K=128, spatial=(700,))
    finally:
        os.environ.pop("CONV_FORCE_SPLITK")
    try:
        need = B.conv_workspace_bytes(h)
        assert need > 0 and "splits=3" in B.conv_plan_describe(h)
        with pytest.raises(B.ConvError) as e:
            B.conv_plan_set_workspace(h, 0, 0)
        assert e.value.status == B.CONV_ERR_WORKSPACE
        with pytest.raises(B.ConvError) as e:
            B.conv_plan_set_workspace(h, 4096, need - 1)
        assert e.value.status == B.CONV_ERR_WORKSPACE
        with pytest.raises(B.ConvError) as e:      # conv_fwd refuses before touching the GPU
            B.conv_fwd(h, 4096, 4096, 4096, 4096, 0)
        assert e.value.status == B.CONV_ERR_WORKSPACE
    finally:
        B.conv_plan_destroy(h)


def test_conv_fwd_argument_checks_precede_any_launch(lib):
    h = plan()
    try:
        for args, status in [((0, 4096, 4096, 4096), B.CONV_ERR_INVALID_ARG),
                             ((4096, 4096, 0, 4096), B.CONV_ERR_INVALID_ARG),      # bias required
                             ((4097, 4096, 4096, 4096), B.CONV_ERR_ALIGNMENT),
                             ((4096, 4104, 4096, 4096), B.CONV_ERR_ALIGNMENT),
                             ((4096, 4096, 4096, 4100), B.CONV_ERR_ALIGNMENT)]:
            with pytest.raises(B.ConvError) as e:
                B.conv_fwd(h, *args, 0)
            assert e.value.status == status
        assert lib.conv_fwd(None, None, None, None, None, None) == B.CONV_ERR_INVALID_ARG
        assert lib.conv_prepack_weights(h, None, None, None) == B.CONV_ERR_INVALID_ARG
        assert lib.conv_plan_output_shape(None, None) == B.CONV_ERR_INVALID_ARG
        assert lib.conv_prepacked_weight_bytes(None) == 0 and lib.conv_workspace_bytes(None) == 0
        assert lib.conv_plan_destroy(None) == B.CONV_OK
    finally:
        B.conv_plan_destroy(h)


def test_tile_and_split_choice_fill_the_gpu(lib):
    """Small problems use narrower tiles (and only then split the reduction) so that the
    work units cover at least three quarters of the SMs in one wave; large ones do not split."""
    def desc_of(layer, code):
        h = B.conv_plan_create(*layer.plan_args(code))
        d = B.conv_plan_describe(h)
        B.conv_plan_destroy(h)
        return dict(kv.split("=") for kv in d.split())
    for code in (B.CONV_BF16, B.CONV_F32):
        for layer in WORKLOADS["whisper_frontend_bf16"].layers:
            d = desc_of(layer, code)
            assert 0.75 * 152 <= int(d["units"]) <= 152, d
    big = WORKLOADS["grouped3d_g4_c64_d1"].layers[0]
    d = desc_of(big, B.CONV_BF16)
    # the 3D layer has thousands of tiles: whole reductions, 64-wide N tiles, paired along H
    assert d["splits"] == "1" and d["tile"] == "256x64" and d["acc"] == "2", d
    d = desc_of(WORKLOADS["sweep_bf16_n32"].layers[1], B.CONV_BF16)
    assert d["tile"] == "128x256"


def _sm_count():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152


def _table_key(layer, code):
    """The selector table's key for one layer (the file format conv_tune_table_save writes)."""
    ndim, N, G, C, K, sp, fl, st, pa, di, dtype, epi = layer.plan_args(code)
    pad3 = lambda v, fill: [fill] * (3 - ndim) + [int(a) for a in v]
    j = lambda v, fill: "x".join(str(a) for a in pad3(v, fill))
    return (f"nd={ndim} N={N} G={G} C={C} K={K} in={j(sp, 1)} f={j(fl, 1)} s={j(st, 1)} p={j(pa, 0)} "
            f"d={j(di, 1)} dtype={dtype} epi={epi} dir=0 sm={_sm_count()}")


def test_selector_table_load_save_and_precedence(lib, tmp_path):
    """A table entry overrides the rules for exactly its problem; saving writes it back;
    a malformed file changes nothing; clearing restores the rules."""
    layer = WORKLOADS["whisper_frontend_bf16"].layers[0]
    other = WORKLOADS["whisper_frontend_bf16"].layers[1]

    def desc_of(l):
        h = B.conv_plan_create(*l.plan_args(B.CONV_BF16))
        d = B.conv_plan_describe(h)
        B.conv_plan_destroy(h)
        return d

    B.conv_tune_table_clear()
    rules, rules_other = desc_of(layer), desc_of(other)
    assert "tile=128x64" in rules and "variant=simt" not in rules
    choice = ("simt=1 no_pack=0 bn=0 bm=0 splits=0 gather=0 slab_stream=0 slab_pair=-1 epi_warps=0 "
              "cluster_red=-1")
    f = tmp_path / "table.txt"
    f.write_text(f"# measured choices\n{_table_key(layer, B.CONV_BF16)} | {choice}\n")
    try:
        B.conv_tune_table_load(str(f))
        assert desc_of(layer).startswith("variant=simt_bf16")
        assert desc_of(other) == rules_other                   # other problems keep the rules
        out = tmp_path / "saved.txt"
        B.conv_tune_table_save(str(out))
        # (a row without the mc field, as older tables wrote it, loads with mc left to the rules)
        assert out.read_text().splitlines() == [f"{_table_key(layer, B.CONV_BF16)} | {choice} mc=-1 pair=-1"]
        B.conv_tune_table_load(str(out))
        assert desc_of(layer).startswith("variant=simt_bf16")
        bad = tmp_path / "bad.txt"
        bad.write_text(f"{_table_key(other, B.CONV_BF16)} | {choice}\nnot a table line\n")
        with pytest.raises(B.ConvError) as e:
            B.conv_tune_table_load(str(bad))
        assert e.value.status == B.CONV_ERR_INVALID_ARG
        assert desc_of(other) == rules_other                   # nothing of the bad file was taken
        with pytest.raises(B.ConvError):
            B.conv_tune_table_load(str(tmp_path / "missing.txt"))
        # the test variables take precedence over the table
        os.environ["CONV_FORCE_BN"] = "32"
        try:
            assert "tile=128x32" in desc_of(layer)
        finally:
            os.environ.pop("CONV_FORCE_BN")
    finally:
        B.conv_tune_table_clear()
    assert desc_of(layer) == rules


def test_weight_multicast_plans(lib):
    """CTA pairs that share each weight tile run only on request (CONV_FORCE_MC or the
    selector): wide unsplit bf16 per-tap plans then take them, with units covering the M tiles
    two at a time and an even grid; the rules never pick them, and plans that cannot (slab,
    3xTF32, narrow or split) ignore the request."""
    for name, li, want in [("sweep_bf16_n32", 0, True), ("sweep_bf16_n32", 1, True), ("sweep_bf16_n8", 1, True),
                           ("grouped3d_g4_c64_d1", 0, False), ("whisper_frontend_f32", 1, False)]:
        wl = WORKLOADS[name]
        h = B.conv_plan_create(*wl.layers[li].plan_args(wl.dtype_code))
        assert "weights=" not in B.conv_plan_describe(h)
        B.conv_plan_destroy(h)
        os.environ["CONV_FORCE_MC"] = "1"
        try:
            h = B.conv_plan_create(*wl.layers[li].plan_args(wl.dtype_code))
        finally:
            os.environ.pop("CONV_FORCE_MC")
        d = dict(kv.split("=", 1) for kv in B.conv_plan_describe(h).split())
        B.conv_plan_destroy(h)
        assert (d.get("weights") == "multicast2") == want, (name, li, d)
        if want:
            assert int(d["grid"]) % 2 == 0 and d["splits"] == "1"
            BW = int(d["pixels"].split("x")[1])
            L = wl.layers[li]
            Wo = oracle.out_len(L.spatial[0], L.filter[0], L.stride[0], L.pad[0], L.dilation[0])
            num_mt = L.N * -(-Wo // BW)
            num_nt = -(-L.K // int(d["tile"].split("x")[1]))
            assert int(d["units"]) == -(-num_mt // 2) * num_nt
    os.environ.update({"CONV_FORCE_MC": "1", "CONV_FORCE_BN": "128"})
    try:
        h = B.conv_plan_create(1, 1, 1, 64, 128, (700,), (3,), (2,), (1,), (1,), B.CONV_BF16, B.CONV_EPI_BIAS)
        d = B.conv_plan_describe(h)
        B.conv_plan_destroy(h)
        assert "weights=multicast2" in d and "tile=128x128" in d and "units=2 " in d, d   # 3 M tiles -> 2 pairs
    finally:
        os.environ.pop("CONV_FORCE_MC")
        os.environ.pop("CONV_FORCE_BN")


def test_cta_pair_plans(lib):
    """bf16 per-tap plans with 128- or 256-wide N tiles, no split and long reductions (8
    epilogue warps) run on CTA pairs (M = 256 tiles) when the pairs' units fill every pair of
    SMs: the 1280 -> 1280 sweep layer at batch 8 and 32; not the 128 -> 1280 layer (16 epilogue
    warps), the batch-1 or Whisper layers, the slab, 3xTF32 or split plans.  Units cover the M
    tiles two at a time and the grid is even."""
    for name, li, want in [("sweep_bf16_n32", 0, False), ("sweep_bf16_n32", 1, True), ("sweep_bf16_n8", 0, False),
                           ("sweep_bf16_n8", 1, True), ("sweep_bf16_n1", 1, False), ("whisper_frontend_bf16", 1, False),
                           ("whisper_frontend_f32", 1, False)]:
        wl = WORKLOADS[name]
        L = wl.layers[li]
        h = B.conv_plan_create(*L.plan_args(wl.dtype_code))
        d = dict(kv.split("=", 1) for kv in B.conv_plan_describe(h).split())
        B.conv_plan_destroy(h)
        assert (d.get("cta_pair") == "m256") == want, (name, li, d)
        if want:
            assert int(d["grid"]) % 2 == 0 and d["splits"] == "1"
            BW = int(d["pixels"].split("x")[1])
            Wo = oracle.out_len(L.spatial[0], L.filter[0], L.stride[0], L.pad[0], L.dilation[0])
            num_mt = L.N * -(-Wo // BW)
            num_nt = -(-L.K // int(d["tile"].split("x")[1]))
            assert int(d["units"]) == -(-num_mt // 2) * num_nt
    os.environ.update({"CONV_FORCE_PAIR": "1", "CONV_FORCE_BN": "128", "CONV_FORCE_SPLITK": "1"})
    try:
        h = B.conv_plan_create(1, 1, 1, 64, 128, (700,), (3,), (2,), (1,), (1,), B.CONV_BF16, B.CONV_EPI_BIAS)
        d = B.conv_plan_describe(h)
        B.conv_plan_destroy(h)
        assert "cta_pair=m256" in d and "units=2 " in d and "grid=4 " in d, d   # 3 M tiles -> 2 pairs
    finally:
        for k in ("CONV_FORCE_PAIR", "CONV_FORCE_BN", "CONV_FORCE_SPLITK"):
            os.environ.pop(k)


def test_slab_cta_pair_plans(lib):
    """Slab plans with tile pairs and N tiles of 32 or 64 run on CTA pairs by rule when three
    slab stages and a ring of at least four weight stages fit (each CTA holds half of every
    weight tile): the 3D dilation-1 configuration, and the 3D dilation-2 one with tiles of half
    the output width (its full-width tile-pair slab of 8 rows leaves room for two weight stages;
    the narrow one has 12 rows of 31 pixels).  Resident weights stay on single CTAs (measured
    no faster as pairs), as do the Whisper layers (too few units); CONV_FORCE_PAIR=1 still
    pairs them."""
    for name, want, stages, acc in [("grouped3d_g4_c64_d1", True, "3+5", "2"), ("grouped3d_g4_c64_d2", True, "3+5", "2"),
                                    ("grouped2d_g8_c64_d1", False, None, "2"), ("grouped2d_g8_c64_d2", False, None, "2"),
                                    ("grouped2d_g32_c8_d1", False, None, "2"), ("whisper_frontend_bf16", False, None, None)]:
        L = WORKLOADS[name].layers[0]
        h = B.conv_plan_create(*L.plan_args(B.CONV_BF16))
        d = dict(kv.split("=", 1) for kv in B.conv_plan_describe(h).split())
        B.conv_plan_destroy(h)
        assert (d.get("cta_pair") == "m256") == want, (name, d)
        if acc:
            assert d["acc"] == acc, (name, d)
        if want:
            assert d["gather"] == "tma-slab" and int(d["grid"]) % 2 == 0
            if stages:
                assert d["stages"] == stages, d
        if name == "grouped3d_g4_c64_d2":
            assert d["pixels"] == "8x27" and d["slab"] == "12x31", d
    os.environ["CONV_FORCE_PAIR"] = "1"
    try:
        h = B.conv_plan_create(*WORKLOADS["grouped2d_g8_c64_d1"].layers[0].plan_args(B.CONV_BF16))
        d = dict(kv.split("=", 1) for kv in B.conv_plan_describe(h).split())
        B.conv_plan_destroy(h)
        # resident weights: the pairs' grid is a multiple of the 8 weight sets, so each keeps its set
        assert d["cta_pair"] == "m256" and d["stages"] == "3+1w" and (int(d["grid"]) // 2) % 8 == 0, d
    finally:
        os.environ.pop("CONV_FORCE_PAIR")


def test_selector_scratch_covers_every_candidate(lib):
    """conv_tune_scratch_bytes is at least this plan's own packed weight plus workspace."""
    for layer in WORKLOADS["whisper_frontend_f32"].layers:
        h = B.conv_plan_create(*layer.plan_args(B.CONV_F32))
        try:
            need = B.conv_tune_scratch_bytes(h)
            own = B.conv_prepacked_weight_bytes(h) + B.conv_workspace_bytes(h)
            assert need >= own > 0
        finally:
            B.conv_plan_destroy(h)
    assert lib.conv_tune_scratch_bytes(None) == 0
    assert lib.conv_plan_tune(None, None, None, None, None, None, 0, 1, None) == B.CONV_ERR_INVALID_ARG


def _bwd_plan(kind, ndim=2, N=1, G=2, C=16, K=24, spatial=(9, 11), filt=(3, 3), stride=(1, 1), pad=(1, 1),
              dil=(1, 1), dtype=B.CONV_BF16):
    create = B.conv_bwd_data_plan_create if kind == "data" else B.conv_bwd_weight_plan_create
    return create(ndim, N, G, C, K, spatial, filt, stride, pad, dil, dtype)


def test_backward_plans_describe_shape_flops_and_variant(lib):
    fwd = plan(ndim=2, G=2, C=16, K=24, spatial=(9, 11), filt=(3, 3), stride=(1, 1), pad=(1, 1), dil=(1, 1))
    try:
        fshape = B.conv_plan_output_shape(fwd, 2)
        fflops = B.conv_plan_flops(fwd)
    finally:
        B.conv_plan_destroy(fwd)
    for kind in ("data", "weight"):
        h = _bwd_plan(kind)
        try:
            assert B.conv_plan_output_shape(h, 2) == fshape          # dy's extents
            assert B.conv_plan_flops(h) == fflops
            d = B.conv_plan_describe(h)
            if kind == "data":
                # unit stride: the forward kernels on the transposed problem (C and K swapped)
                assert "direction=bwd_data(transposed_forward)" in d and d.startswith("variant=tc_bf16"), d
                assert B.conv_prepacked_weight_bytes(h) > 0
            else:
                assert "direction=bwd_weight" in d, d
                assert B.conv_prepacked_weight_bytes(h) == 0
                with pytest.raises(B.ConvError) as e:
                    B.conv_prepack_weights(h, 4096, 4096, 0)
                assert e.value.status == B.CONV_ERR_INVALID_ARG
        finally:
            B.conv_plan_destroy(h)
    # stride 2 (4 phases), and padding beyond the filter's reach (1 phase, negative padding):
    # stride phases on the forward kernels
    for kw, nph in ((dict(stride=(2, 2)), 4), (dict(pad=(3, 1)), 1), (dict(stride=(2, 3), filt=(1, 1), pad=(0, 0)), 1)):
        h = _bwd_plan("data", **kw)
        try:
            d = dict(kv.split("=", 1) for kv in B.conv_plan_describe(h).split())
            assert d["direction"] == "bwd_data(phases)" and d["phases"] == str(nph), d
            assert d["variant"] == "tc_bf16"
            # a 1x1 filter at stride 2 x 3 reaches one input pixel in 6: the rest are cleared
            assert d["zero_fill"] == ("1" if kw.get("filt") == (1, 1) else "0"), d
        finally:
            B.conv_plan_destroy(h)
    # channel counts the tensor-core path cannot take: the gather kernel
    h = _bwd_plan("data", C=6, K=10, stride=(2, 2), dtype=B.CONV_F32)
    try:
        assert "direction=bwd_data(gather)" in B.conv_plan_describe(h)
    finally:
        B.conv_plan_destroy(h)


def test_backward_entry_points_check_direction_and_arguments(lib):
    fwd = plan()
    dg = _bwd_plan("data")
    wg = _bwd_plan("weight")
    try:
        for h in (dg, wg):       # a backward plan is refused by the forward entry points
            assert lib.conv_fwd(h, 4096, 4096, 4096, 4096, None) == B.CONV_ERR_INVALID_ARG
            assert lib.conv_fwd_static_scratch(h, 4096, 4096, 4096, 4096, None) == B.CONV_ERR_INVALID_ARG
        assert lib.conv_bwd_data(fwd, 4096, 4096, 4096, None) == B.CONV_ERR_INVALID_ARG
        assert lib.conv_bwd_data(wg, 4096, 4096, 4096, None) == B.CONV_ERR_INVALID_ARG
        assert lib.conv_bwd_weight(dg, 4096, 4096, 4096, None) == B.CONV_ERR_INVALID_ARG
        assert lib.conv_bwd_data(dg, None, 4096, 4096, None) == B.CONV_ERR_INVALID_ARG
        assert lib.conv_bwd_weight(wg, 4096, None, 4096, None) == B.CONV_ERR_INVALID_ARG
        assert lib.conv_bwd_data(dg, 4100, 4096, 4096, None) == B.CONV_ERR_ALIGNMENT
        assert lib.conv_bwd_weight(wg, 4096, 4096, 4104, None) == B.CONV_ERR_ALIGNMENT
        assert lib.conv_tune_scratch_bytes(wg) == 0
        for kw in (dict(ndim=0), dict(N=0), dict(stride=(0, 1)), dict(spatial=(1, 1), pad=(0, 0))):
            for kind in ("data", "weight"):
                with pytest.raises(B.ConvError) as e:
                    _bwd_plan(kind, **kw)
                assert e.value.status == B.CONV_ERR_INVALID_ARG
    finally:
        for h in (fwd, dg, wg):
            B.conv_plan_destroy(h)


def test_backward_weight_splits_pixels_and_needs_a_workspace(lib):
    """A large reduction over output pixels is split across CTAs; the partials need a workspace."""
    layer = WORKLOADS["grouped2d_g8_c64_d1"].layers[0]
    h = B.conv_bwd_weight_plan_create(*layer.plan_args(B.CONV_BF16)[:11])
    try:
        d = dict(kv.split("=", 1) for kv in B.conv_plan_describe(h).split())
        assert int(d["splits"]) > 1 and B.conv_workspace_bytes(h) > 0
        assert lib.conv_bwd_weight(h, 4096, 4096, 4096, None) == B.CONV_ERR_WORKSPACE
    finally:
        B.conv_plan_destroy(h)


def test_every_plan_description_is_key_value_pairs(lib):
    """The benchmark and the tests read plan descriptions as space-separated key=value pairs."""
    for wl in WORKLOADS.values():
        for layer in wl.layers:
            args = layer.plan_args(wl.dtype_code)
            for create in (lambda: B.conv_plan_create(*args), lambda: B.conv_bwd_data_plan_create(*args[:11]),
                           lambda: B.conv_bwd_weight_plan_create(*args[:11])):
                h = create()
                try:
                    d = B.conv_plan_describe(h)
                finally:
                    B.conv_plan_destroy(h)
                assert all(len(kv.split("=", 1)) == 2 for kv in d.split()), d


def test_missing_library_fails_loudly(tmp_path):
    """Without the built library every entry point raises: there is no CPU or PyTorch fallback."""
    import subprocess
    import sys
    code = ("from convolution_forward_implicit_gb300 import binding as B\n"
            "try:\n"
            "    B.conv_plan_create(1, 1, 1, 80, 384, [3000], [3], [1], [1], [1], B.CONV_BF16, B.CONV_EPI_BIAS)\n"
            "except RuntimeError as e:\n"
            "    print('raised:', 'not built' in str(e))\n")
    env = dict(os.environ, CONVFWD_LIBRARY=str(tmp_path / "absent" / "libconvfwd.so"))
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "raised: True", out.stdout + out.stderr


def test_static_scratch_size_agrees_with_the_header(lib):
    """The allocation-free entry point's array: the library reports the size the header states."""
    src = open(os.path.join(ROOT, "include", "conv.h")).read()
    m = re.search(r"#define\s+CONV_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", src)
    assert m, "CONV_STATIC_SCRATCH_BYTES not found in include/conv.h"
    assert B.conv_static_scratch_bytes() == int(m.group(1)) << int(m.group(2))


@pytest.mark.parametrize("name,li,variant", [
    ("whisper_frontend_f32", 0, "tc_tf32x3"), ("whisper_frontend_f32", 1, "tc_tf32x3"),
    ("conv1d_f32_80to384_L3000", 0, "tc_tf32x3"), ("whisper_mlp_f32", 0, "tc_tf32x3"),
    ("whisper_frontend_bf16", 0, "tc_bf16"), ("sweep_bf16_n32", 1, "tc_bf16"), ("grouped2d_g32_c8_d1", 0, "tc_bf16"),
])
def test_default_arithmetic_is_the_one_the_header_documents(lib, name, li, variant):
    """include/conv.h: fp32 I/O runs as 3xTF32 on the tensor cores by default, bf16 I/O as
    bf16 tensor-core products; the FFMA kernel takes only what the tensor-core plans cannot."""
    layer = WORKLOADS[name].layers[li]
    h = B.conv_plan_create(*layer.plan_args(WORKLOADS[name].dtype_code))
    assert f"variant={variant} " in B.conv_plan_describe(h) + " "
    B.conv_plan_destroy(h)
    # channel counts the tensor-core plans cannot take fall back to the FFMA kernel
    h = B.conv_plan_create(1, 1, 1, 3, 5, (40,), (3,), (1,), (1,), (1,), B.CONV_F32, B.CONV_EPI_BIAS)
    assert "variant=simt_f32" in B.conv_plan_describe(h)
    B.conv_plan_destroy(h)


def _slab_units_expected(layer, d):
    """Units a slab plan's description implies: output tiles of BH x BW pixels per image and
    output plane, times groups and N tiles (packed groups count as one), halved (rounded up
    along M) on CTA pairs."""
    import math
    nd = len(layer.spatial)
    sp = (1,) * (3 - nd) + tuple(layer.spatial)
    f = (1,) * (3 - nd) + tuple(layer.filter)
    st = (1,) * (3 - nd) + tuple(layer.stride)
    pa = (0,) * (3 - nd) + tuple(layer.pad)
    di = (1,) * (3 - nd) + tuple(layer.dilation)
    out = [(sp[i] + 2 * pa[i] - di[i] * (f[i] - 1) - 1) // st[i] + 1 for i in range(3)]
    bh, bw = (int(v) for v in d["pixels"].split("x"))
    pack = int(d.get("pack", "1"))
    bn = int(d["tile"].split("x")[1])
    num_mt = layer.N * out[0] * math.ceil(out[1] / bh) * math.ceil(out[2] / bw)
    if d.get("cta_pair") == "m256":
        num_mt = math.ceil(num_mt / 2)
    return num_mt * (layer.G // pack) * math.ceil(pack * layer.K / bn)


@pytest.mark.parametrize("env", [{}, {"CONV_FORCE_SLAB_PAIR": "1"}, {"CONV_FORCE_SLAB_PAIR": "0"},
                                 {"CONV_FORCE_SLAB_BW": "20"}, {"CONV_FORCE_PAIR": "1"},
                                 {"CONV_FORCE_SLAB_PAIR": "1", "CONV_FORCE_SLAB_STREAM": "1"}])
def test_slab_plan_units_match_their_tiles(lib, env):
    """Every slab plan's unit count is the one its tile shape implies, whatever the rules
    tried on the way (narrower tiles for CTA pairs are dropped with the pairs when the pairs
    are not taken): the grouped workloads and small 2D/3D problems of every dilation."""
    from tests.test_parity_gpu import L
    layers = [WORKLOADS[n].layers[0] for n in ("grouped2d_g8_c64_d1", "grouped2d_g8_c64_d2", "grouped2d_g32_c8_d1",
                                                "grouped3d_g4_c64_d1", "grouped3d_g4_c64_d2")]
    layers += [L(3, 1, 2, 64, 64, (6, 24, 56), (3, 3, 3), (1, 1, 1), (1, 1, 1), (2, 2, 2)),
               L(2, 2, 1, 64, 32, (33, 54), (3, 3), (1, 1), (1, 1), (2, 2)),
               L(3, 2, 4, 64, 64, (7, 28, 40), (3, 3, 3), (1, 1, 1), (2, 2, 2), (2, 2, 2))]
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        seen = 0
        for layer in layers:
            h = B.conv_plan_create(*layer.plan_args(B.CONV_BF16))
            d = dict(kv.split("=", 1) for kv in B.conv_plan_describe(h).split())
            B.conv_plan_destroy(h)
            if d["gather"] != "tma-slab":
                continue
            seen += 1
            assert int(d["units"]) == _slab_units_expected(layer, d), (layer, env, d)
        assert seen
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
