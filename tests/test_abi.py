"""Host-side checks of the C ABI (no GPU needed): the library builds for sm_103a,
loads, exports every symbol include/wgrad.h declares, and validates arguments
before touching the device.  Only calls that fail validation are made here, so
nothing is ever launched."""
import os
import re

import numpy as np
import pytest

import oracle

from implicit_gemm_gb300 import binding, build
from tests.common import WORKLOADS, spec

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def header_symbols():
    with open(os.path.join(ROOT, "include", "wgrad.h")) as f:
        txt = f.read()
    return sorted(set(re.findall(r"WG_API\s+[\w\s\*]+?\b(wg_\w+)\s*\(", txt)))


def test_exports_every_declared_symbol(lib):
    syms = header_symbols()
    assert set(syms) == set(binding.EXPORTS), syms
    for s in syms:
        assert hasattr(lib, s), s


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert binding.wg_status_string(code) == name


def test_normalize_derives_output():
    assert binding.wg_problem_normalize(spec(2, 1, 1, 1, 1, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])) == [8, 8]
    assert binding.wg_problem_normalize(spec(3, 1, 4, 8, 8, [16, 16, 16], [3, 3, 3], [2, 2, 2], [1, 1, 1], [1, 1, 1],
                                             [1, 1, 1])) == [8, 8, 8]
    for sp in (spec(1, 1, 1, 8, 8, [11], [3], [2], [2], [2], [0]), spec(2, 1, 1, 8, 8, [7, 13], [2, 5], [3, 2], [2, 1],
                                                                     [0, 2], [3, 1])):
        assert binding.wg_problem_normalize(sp) == oracle.out_dims(sp)


@pytest.mark.parametrize("bad,status", [
    (dict(ndim=4), 1), (dict(G=0), 1), (dict(N=-1), 1), (dict(C=0), 1),
    (dict(filt=[11, 3]), 1), (dict(stride=[0, 1]), 1), (dict(dil=[1, 0]), 1), (dict(pad_l=[-1, 0]), 1),
    (dict(out=[7, 8]), 1), (dict(in_dtype="fp32"), 1),
])
def test_invalid_arguments(bad, status):
    s = spec(2, 1, 1, 16, 16, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    s.update(bad)
    with pytest.raises(binding.WgradError) as e:
        binding.wg_workspace_size(s)
    assert e.value.status == status


def test_not_supported_paths():
    s = spec(2, 1, 1, 4, 4, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])  # G*C = 4: rows not 16 bytes
    with pytest.raises(binding.WgradError) as e:
        binding.wg_workspace_size(s)
    assert e.value.status == 2
    s = spec(2, 1, 1, 16, 16, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], out_dtype="bf16")
    # Atomic adds into a 16-bit dW go through an fp32 copy in the workspace.
    assert binding.wg_workspace_size(s, split_k=2, mode="atomic") == 16 * 9 * 16 * 4
    assert binding.wg_workspace_size(s, split_k=2, mode="deterministic") == 2 * 16 * 9 * 16 * 4
    with pytest.raises(binding.WgradError) as e:
        binding.wg_workspace_size(s, group_merge=2)  # merge degree is a depthwise option
    assert e.value.status == 2
    with pytest.raises(binding.WgradError) as e:
        binding.wg_workspace_size(s, split_k=2, mode="direct")
    assert e.value.status == 1


def test_size_limits():
    # Tensors of 2^31 elements or more and split degrees above 65535 are refused
    # before anything is planned on a device.
    big = spec(2, 1, 70000, 128, 128, [128, 128], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    with pytest.raises(binding.WgradError) as e:
        binding.wg_workspace_size(big)
    assert e.value.status == 2 and "2^31" in binding.wg_last_error()
    small = spec(2, 1, 2, 16, 16, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    with pytest.raises(binding.WgradError) as e:
        binding.wg_workspace_size(small, split_k=70000, mode="deterministic")
    assert e.value.status == 2
    assert binding.wg_workspace_size(small, split_k=65535, mode="deterministic") > 0


def test_kernel_instance_choice():
    # The CTA-pair kernel serves the pair plans (automatic for long splits:
    # one or four splits of the 56x56 workload); the trimmed instance serves
    # single-CTA x-taps-on-columns plans with one M-tile per CTA in a split
    # mode (the 56x56 workload's automatic S = 75); every other plan takes the
    # general one.
    dense = WORKLOADS["2d_dense_n32_h56_c64_k64"][0]
    assert binding.wg_plan_string(dense).endswith("code=x1")
    assert binding.wg_plan_string(dense, 1, "direct").endswith("code=pair")
    assert binding.wg_plan_string(dense, 4, "deterministic").endswith("code=pair")
    assert binding.wg_plan_string(dense, kernel="igemm_pair").endswith("code=pair")
    assert binding.wg_plan_string(dense, 1, "direct", kernel="igemm_pair").endswith("code=pair")
    assert binding.wg_plan_string(dense, kernel="igemm_taps_mn").endswith("code=x1")
    direct = binding.wg_plan_string(dense, 1, "direct", kernel="igemm_taps_mn")
    assert "taps=mn" in direct and "mode=direct" in direct and direct.endswith("code=any")
    assert binding.wg_plan_string(dense, kernel="igemm_taps_m").endswith("code=any")
    for name in ("2d_grouped_g32_c8_k8_n32_h28", "3d_n4_d16_c128_k96_s2", "2d_1x1_n32_h56_c64_k256"):
        assert binding.wg_plan_string(WORKLOADS[name][0]).endswith("code=any"), name


def test_planner_measured_choices():
    # Choices the planner makes because they measured faster on GB300: the
    # 3-D stride-2 split-K = 8 mode takes two 128-pixel K-tiles per split in a
    # two-stage ring (no refill), not four 64-pixel ones; the 8x8 problem runs
    # five CTAs of one M-tile, not two of three; the 56x56 listed non-split and
    # split-K = 4 modes run on CTA pairs with the x taps on the columns, and
    # its automatic split degree on single CTAs.
    f = _plan_fields(binding.wg_plan_string(WORKLOADS["3d_n4_d16_c128_k96_s2"][0], 8, "atomic"))
    assert (f["KT"], f["per_split"], f["stages"], f["mt_per_cta"]) == ("128", "2", "2", "2"), f
    f = _plan_fields(binding.wg_plan_string(WORKLOADS["2d_tiny_n1_h8_c16_k32"][0]))
    assert (f["mt_per_cta"], f["grid"]) == ("1", "(5,1,1)"), f
    dense = WORKLOADS["2d_dense_n32_h56_c64_k64"][0]
    for S, mode in ((1, "direct"), (4, "deterministic")):
        f = _plan_fields(binding.wg_plan_string(dense, S, mode))
        assert (f["taps"], f["code"]) == ("mn", "pair"), (S, f)
    f = _plan_fields(binding.wg_plan_string(dense))
    assert (f["taps"], f["code"], f["S"]) == ("mn", "x1", "75"), f


def test_workspace_sizes():
    sp = WORKLOADS["2d_dense_n32_h56_c64_k64"][0]
    E = 1 * 64 * 9 * 64  # rows of 576 = 6 slices of 96: no padding
    assert binding.wg_workspace_size(sp, split_k=1) == 0
    assert binding.wg_workspace_size(sp, split_k=4, mode="deterministic", cluster=1) == 4 * E * 4
    # Clusters add their splits on chip: one partial sum per cluster reaches memory.
    assert binding.wg_workspace_size(sp, split_k=8, mode="deterministic", cluster=2) == 4 * E * 4
    assert binding.wg_workspace_size(sp, split_k=8, mode="deterministic", cluster=4) == 2 * E * 4
    # One cluster holds every split: its sums are final, no workspace.
    assert binding.wg_workspace_size(sp, split_k=4, mode="deterministic", cluster=4) == 0
    assert "mode=direct" in binding.wg_plan_string(sp, split_k=8, mode="direct", cluster=8)
    sp5 = WORKLOADS["3d_n4_d16_c128_k96_s2"][0]
    assert binding.wg_workspace_size(sp5, split_k=8, mode="atomic") == 0
    assert binding.wg_workspace_size(sp5, split_k=8, mode="deterministic", cluster=1) == 8 * 96 * 27 * 128 * 4
    # Rows (g, k) of T*C = 9*12 = 108 elements, one slice of 108 each.
    sp6 = spec(2, 2, 1, 12, 8, [9, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    assert binding.wg_workspace_size(sp6, split_k=5, mode="deterministic") == 5 * 2 * 8 * 108 * 4
    # Rows of 37*4 = 148 elements: no multiple of 4 in 64..128 divides 148 -> two slices of 128.
    sp7 = spec(1, 2, 1, 4, 8, [50], [37], [1], [1], [0], [0])
    assert binding.wg_workspace_size(sp7, split_k=5, mode="deterministic") == 5 * 16 * 256 * 4


def test_cluster_option_checks():
    sp = WORKLOADS["2d_dense_n32_h56_c64_k64"][0]
    for bad in (3, 16, -1):
        with pytest.raises(binding.WgradError) as e:
            binding.wg_plan_string(sp, cluster=bad)
        assert e.value.status == 1
    with pytest.raises(binding.WgradError) as e:
        binding.wg_plan_string(sp, split_k=6, cluster=4)
    assert e.value.status == 1 and "divide" in binding.wg_last_error()
    with pytest.raises(binding.WgradError) as e:
        binding.wg_plan_string(sp, split_k=4, mode="direct", cluster=2)
    assert e.value.status == 1
    dw = WORKLOADS["2d_depthwise_g512_n64_h28"][0]
    with pytest.raises(binding.WgradError) as e:
        binding.wg_plan_string(dw, cluster=2)
    assert e.value.status == 2
    # Automatic choice: grid z a multiple of the cluster size.
    for name in WORKLOADS:
        ps = binding.wg_plan_string(WORKLOADS[name][0])
        if "igemm" in ps:
            S, q = int(re.search(r" S=(\d+)", ps).group(1)), int(re.search(r"cluster=(\d+)", ps).group(1))
            assert S % q == 0, ps


def test_launch_argument_checks_before_device(lib):
    sp = spec(2, 1, 1, 16, 16, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    with pytest.raises(binding.WgradError) as e:
        binding.wg_conv_bwd_weight(sp, 0, 4096, 8192)
    assert e.value.status == 1
    with pytest.raises(binding.WgradError) as e:
        binding.wg_conv_bwd_weight(sp, 4096 + 8, 8192, 12288)
    assert e.value.status == 3
    with pytest.raises(binding.WgradError) as e:
        binding.wg_conv_bwd_weight(sp, 4096, 8192, 12288, split_k=3, mode="deterministic")
    assert e.value.status == 4
    assert "workspace" in binding.wg_last_error()


def test_host_entry_argument_checks_before_device(lib):
    # The host-buffer entry point validates before it enqueues anything: NULL host
    # buffers (1), unaligned device buffers (3), a missing workspace (4).
    sp = spec(2, 1, 1, 16, 16, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    for args, status in (((0, 64, 128, 4096, 8192, 12288), 1),
                         ((64, 0, 128, 4096, 8192, 12288), 1),
                         ((64, 128, 0, 4096, 8192, 12288), 1),
                         ((64, 128, 192, 4096 + 8, 8192, 12288), 3),
                         ((64, 128, 192, 4096, 8192, 0), 1)):
        with pytest.raises(binding.WgradError) as e:
            binding.wg_conv_bwd_weight_host(sp, *args)
        assert e.value.status == status, args
    with pytest.raises(binding.WgradError) as e:
        binding.wg_conv_bwd_weight_host(sp, 64, 128, 192, 4096, 8192, 12288, split_k=3, mode="deterministic")
    assert e.value.status == 4


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_plans_for_workloads(name):
    sp = WORKLOADS[name][0]
    ps = binding.wg_plan_string(sp)
    kind = "depthwise" if sp["C"] == 1 and sp["K"] == 1 else "igemm_tcgen05"
    assert f"kernel={kind}" in ps
    m = re.search(r"smem=(\d+)", ps)
    assert int(m.group(1)) <= 232448


def test_depthwise_merge_degrees():
    sp = WORKLOADS["2d_depthwise_g512_n64_h28"][0]
    for gm in (1, 2, 4, 8):
        assert f"Gm={gm} " in binding.wg_plan_string(sp, group_merge=gm)


def test_mark_event_can_be_cleared_without_device(lib):
    # Setting and clearing the measurement hook touches no device state.
    binding.wg_set_mark_event(None)
    assert lib.wg_set_mark_event(None) == 0


def test_kernel_selector():
    dw = WORKLOADS["2d_depthwise_g512_n64_h28"][0]
    assert "kernel=depthwise" in binding.wg_plan_string(dw)
    ps = binding.wg_plan_string(dw, kernel="igemm")
    # Block-diagonal tensor-core plan: 64 groups per tile, windows 8-aligned.
    assert "kernel=igemm_tcgen05" in ps and " Gm=64 " in ps and "gblocks=8 " in ps
    dense = WORKLOADS["2d_dense_n32_h56_c64_k64"][0]
    with pytest.raises(binding.WgradError) as e:
        binding.wg_plan_string(dense, kernel="depthwise")
    assert e.value.status == 2
    with pytest.raises(binding.WgradError) as e:
        lib_opts = binding.make_options()
        lib_opts.kernel = 6
        p = binding.make_problem(dense)
        import ctypes
        buf = ctypes.create_string_buffer(256)
        binding._check(binding.load().wg_plan_string(ctypes.byref(p), ctypes.byref(lib_opts), buf, len(buf)))
    assert e.value.status == 1


def test_tap_form_selector():
    # x taps on the MMA columns: stride 1, no group fold, K a multiple of 64,
    # 2 <= X <= 4 and no cluster; NOT_SUPPORTED (2) otherwise when forced.
    ok = [spec(2, 1, 2, 64, 64, [13, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
          spec(2, 1, 2, 64, 128, [9, 14], [3, 4], [1, 1], [1, 1], [1, 2], [1, 1]),
          spec(1, 1, 3, 40, 64, [50], [2], [1], [3], [3], [3]),
          spec(3, 2, 2, 72, 64, [5, 6, 7], [3, 3, 3], [1, 1, 1], [1, 1, 1], [1, 1, 1], [1, 1, 1]),
          spec(2, 32, 2, 8, 8, [9, 10], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])]  # 8 groups folded: k window 64
    for sp in ok:
        f = _plan_fields(binding.wg_plan_string(sp, kernel="igemm_taps_mn"))
        assert f["taps"] == "mn" and f["Nmma"] == str(64 * sp["filt"][-1]) and f["Nt"] == "64", f
        assert int(f["tmem_cols"]) >= int(f["mt_per_cta"]) * int(f["Nmma"])
        assert _plan_fields(binding.wg_plan_string(sp, kernel="igemm_taps_m"))["taps"] == "m"
    bad = [spec(2, 1, 2, 64, 64, [13, 11], [3, 3], [2, 2], [1, 1], [1, 1], [1, 1]),   # stride 2
           spec(2, 1, 2, 64, 96, [13, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),   # K = 96
           spec(2, 1, 2, 64, 64, [13, 11], [3, 1], [1, 1], [1, 1], [1, 0], [1, 0]),   # X = 1
           spec(2, 1, 2, 64, 64, [13, 11], [3, 5], [1, 1], [1, 1], [1, 2], [1, 2]),   # X = 5
           spec(2, 2, 2, 24, 40, [13, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])]   # folded k window 80
    for sp in bad:
        with pytest.raises(binding.WgradError) as e:
            binding.wg_plan_string(sp, kernel="igemm_taps_mn")
        assert e.value.status == 2, sp
    with pytest.raises(binding.WgradError) as e:
        binding.wg_plan_string(ok[0], 4, "deterministic", 0, cluster=2, kernel="igemm_taps_mn")
    assert e.value.status == 2
    # Depthwise problems run on the tensor cores under either tap form selector.
    dw = WORKLOADS["2d_depthwise_g512_n64_h28"][0]
    assert "kernel=igemm_tcgen05" in binding.wg_plan_string(dw, kernel="igemm_taps_m")


def test_pair_selector():
    # The CTA-pair form: the x-taps-on-columns tile with K = 64 (no fold), one
    # 64-channel chunk (C <= 64) and a 2-D filter of 3 or 4 rows: the split's
    # two M-tiles on the two CTAs of a cluster (grid x = 2).
    ok = [spec(2, 1, 2, 64, 64, [13, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
          spec(2, 1, 2, 40, 64, [9, 14], [4, 3], [1, 1], [1, 2], [2, 1], [1, 1]),
          spec(2, 2, 3, 64, 64, [7, 10], [3, 2], [1, 1], [2, 1], [2, 0], [2, 1]),
          spec(2, 1, 1, 16, 64, [20, 19], [3, 4], [1, 1], [1, 1], [1, 2], [1, 1])]
    for sp in ok:
        for mode in ("auto", "deterministic", "direct"):
            f = _plan_fields(binding.wg_plan_string(sp, 1 if mode == "direct" else 0, mode, kernel="igemm_pair"))
            assert f["code"] == "pair" and f["taps"] == "mn" and f["mranges"] == "2" and f["mt_per_cta"] == "1", f
            assert f["grid"].startswith("(2,") and f["Nmma"] == str(64 * sp["filt"][-1]), f
    bad = [spec(2, 1, 2, 64, 128, [13, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),  # K = 128
           spec(2, 1, 2, 96, 64, [13, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),   # C = 96: two chunks
           spec(2, 1, 2, 64, 64, [13, 11], [2, 3], [1, 1], [1, 1], [1, 1], [1, 1]),   # 2 taps along h
           spec(2, 1, 2, 64, 64, [13, 11], [5, 3], [1, 1], [1, 1], [2, 1], [2, 1]),   # 5 taps along h
           spec(3, 1, 2, 64, 64, [5, 6, 7], [3, 3, 3], [1, 1, 1], [1, 1, 1], [1, 1, 1], [1, 1, 1]),  # 3-D
           spec(1, 1, 3, 64, 64, [50], [3], [1], [1], [1], [1]),                        # 1-D
           spec(2, 32, 2, 8, 8, [9, 10], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),     # folded groups
           spec(2, 1, 2, 64, 64, [13, 11], [3, 3], [2, 2], [1, 1], [1, 1], [1, 1])]   # stride 2
    for sp in bad:
        with pytest.raises(binding.WgradError) as e:
            binding.wg_plan_string(sp, kernel="igemm_pair")
        assert e.value.status == 2, sp
    with pytest.raises(binding.WgradError) as e:
        binding.wg_plan_string(ok[0], 4, "deterministic", 0, cluster=2, kernel="igemm_pair")
    assert e.value.status == 2
    # The single-CTA selector never takes the pair.
    assert _plan_fields(binding.wg_plan_string(ok[0], kernel="igemm_taps_mn"))["code"] != "pair"


def test_dgrad_plans_and_limits():
    dense = WORKLOADS["2d_dense_n32_h56_c64_k64"][0]
    ps = binding.wg_bwd_data_plan_string(dense)
    assert "kernel=dgrad_tcgen05" in ps and "box=(w8,h16)" in ps
    one_d = spec(1, 1, 2, 16, 24, [300], [5], [1], [2], [4], [4])
    assert "box=(w128,h1)" in binding.wg_bwd_data_plan_string(one_d)
    assert "phases=4 " in binding.wg_bwd_data_plan_string(spec(2, 1, 1, 16, 16, [9, 9], [3, 3], [2, 2]))
    for bad, status in ((spec(2, 1, 1, 16, 16, [40, 9], [3, 3], [9, 1]), 2),     # stride above 8
                        (spec(2, 1, 1, 4, 8, [9, 9], [3, 3]), 2),                # G*C not a multiple of 8
                        (spec(2, 1, 1, 0, 8, [9, 9], [3, 3]), 1)):               # C = 0
        with pytest.raises(binding.WgradError) as e:
            binding.wg_bwd_data_plan_string(bad)
        assert e.value.status == status


def test_dgrad_group_fold():
    # Small C and K: Gm groups share a tile through a block-diagonal copy of W in the workspace.
    sp = WORKLOADS["2d_grouped_g32_c8_k8_n32_h28"][0]
    ps = binding.wg_bwd_data_plan_string(sp)
    assert " Gm=8 " in ps and "grid=(" in ps
    assert binding.wg_bwd_data_workspace_size(sp) == 4 * 64 * 9 * 64 * 2
    assert binding.wg_bwd_data_workspace_size(WORKLOADS["2d_dense_n32_h56_c64_k64"][0]) == 0
    folded = spec(2, 2, 1, 4, 8, [9, 9], [3, 3])  # C = 4: supported only through the fold
    assert " Gm=2 " in binding.wg_bwd_data_plan_string(folded)


def _plan_fields(ps):
    return {k: v for k, v in re.findall(r"(\w+)=(\S+)", ps)}


def test_planner_choices_on_default_caps():
    # With the GB300 defaults (no device): the headline plan, split degrees below
    # the device-filling one where the cold HBM read bounds the main loop, and
    # explicit split degrees that keep well-shaped pixel tiles (a cost floor
    # must not make every tiling tie).
    dense = _plan_fields(binding.wg_plan_string(WORKLOADS["2d_dense_n32_h56_c64_k64"][0]))
    assert (dense["taps"], dense["S"], dense["mt_per_cta"], dense["box"]) == ("mn", "75", "1", "(w32,h8,d1,n1)")
    dense = _plan_fields(binding.wg_plan_string(WORKLOADS["2d_dense_n32_h56_c64_k64"][0], kernel="igemm_taps_m"))
    assert (dense["S"], dense["mt_per_cta"], dense["box"]) == ("75", "3", "(w8,h7,d1,n4)")
    # Depthwise vector width: two channels (one packed word) whatever the
    # filter, stride or problem size -- no threshold on anything -- unless the
    # caller asks for a width.
    dwp = _plan_fields(binding.wg_plan_string(WORKLOADS["2d_depthwise_g512_n64_h28"][0]))
    assert (dwp["kernel"], dwp["Gm"]) == ("depthwise", "2")
    small = _plan_fields(binding.wg_plan_string(spec(2, 64, 2, 1, 1, [9, 13], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])))
    assert small["Gm"] == "2"
    strided = _plan_fields(binding.wg_plan_string(spec(2, 64, 2, 1, 1, [9, 13], [3, 3], [2, 2], [1, 1], [1, 1],
                                                       [1, 1])))
    assert strided["Gm"] == "2"
    for g in (1, 2, 4, 8):  # an explicit merge degree is kept
        p = _plan_fields(binding.wg_plan_string(WORKLOADS["2d_depthwise_g512_n64_h28"][0], 0, "auto", g))
        assert p["Gm"] == str(g)
    # 8 groups of C = K = 8 folded into a 64-wide window: the column form too.
    grouped = _plan_fields(binding.wg_plan_string(WORKLOADS["2d_grouped_g32_c8_k8_n32_h28"][0]))
    assert (grouped["taps"], grouped["Gm"], grouped["Nmma"], grouped["S"]) == ("mn", "8", "192", "38")
    one = _plan_fields(binding.wg_plan_string(WORKLOADS["2d_1x1_n32_h56_c64_k256"][0]))
    assert int(one["S"]) < 150
    for S in (75, 100, 150):
        p = _plan_fields(binding.wg_plan_string(WORKLOADS["2d_1x1_n32_h56_c64_k256"][0], S, "deterministic", 0))
        h = int(p["box"].split(",")[1][1:])
        assert p["S"] == str(S) and h >= 4, p["box"]


def _dg_fields(ps):
    return {k: v for k, v in re.findall(r"(\w+)=(\S+)", ps)}


def test_dgrad_persistent_plans():
    # Two CTAs per SM (shared memory and TMEM of both fit) come first; W stays
    # resident when one (channel tile, group) covers the problem.
    nsm = 152
    dense = _dg_fields(binding.wg_bwd_data_plan_string(WORKLOADS["2d_dense_n32_h56_c64_k64"][0]))
    assert dense["w_resident"] == "1" and int(dense["smem"]) <= 232448 // 2 - 1024
    assert dense["grid"] == f"({2 * nsm},1,1)" and int(dense["tmem_cols"]) <= 256
    grouped = _dg_fields(binding.wg_bwd_data_plan_string(WORKLOADS["2d_grouped_g32_c8_k8_n32_h28"][0]))
    assert grouped["w_resident"] == "0"  # four group blocks: W streamed with each patch
    # C = 256 takes two 128-channel tiles (TMEM for two accumulators of two CTAs).
    wide = _dg_fields(binding.wg_bwd_data_plan_string(WORKLOADS["2d_1x1s2_n32_h56_c256_k128"][0]))
    assert wide["Nt"] == "128" and wide["ctiles"] == "2" and wide["w_resident"] == "0"
    # Never more CTAs than tiles.
    tiny = _dg_fields(binding.wg_bwd_data_plan_string(spec(2, 1, 1, 16, 16, [8, 8], [3, 3], [1, 1], [1, 1],
                                                           [1, 1], [1, 1])))
    assert tiny["grid"] == "(1,1,1)"


def test_dgrad_launch_checks_before_device(lib):
    sp = spec(2, 1, 1, 16, 16, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    with pytest.raises(binding.WgradError) as e:
        binding.wg_conv_bwd_data(sp, 0, 4096, 8192)
    assert e.value.status == 1
    with pytest.raises(binding.WgradError) as e:
        binding.wg_conv_bwd_data(sp, 4096, 8192 + 4, 12288)
    assert e.value.status == 3


def test_planner_invariants_on_random_problems():
    # Seeded random problems (1-, 2- and 3-D, strides, dilations, groups, both
    # tile forms and the depthwise kernel): every plan is either refused with
    # NOT_SUPPORTED or satisfies the limits the kernels rely on.
    rng = np.random.default_rng(20261202)
    checked = {"m": 0, "mn": 0, "depthwise": 0}
    for _ in range(400):
        nd = int(rng.integers(1, 4))
        G = int(rng.choice([1, 1, 2, 4, 8, 32]))
        C = int(rng.choice([1, 8, 16, 24, 40, 64, 72, 128]))
        K = int(rng.choice([1, 8, 16, 32, 64, 96, 128, 256]))
        if C == 1 or K == 1:
            C = K = 1
            G = int(rng.choice([8, 16, 64, 512]))
        if (G * C) % 8 or (G * K) % 8:
            continue
        filt = [int(rng.choice([1, 2, 3, 3, 4, 5])) for _ in range(nd)]
        stride = [int(rng.choice([1, 1, 1, 2, 3])) for _ in range(nd)]
        dil = [int(rng.choice([1, 1, 2])) for _ in range(nd)]
        inn = [int(rng.integers(1, 40)) for _ in range(nd)]
        pl = [int(rng.integers(0, f)) for f in filt]
        pr = [int(rng.integers(0, f)) for f in filt]
        sp = spec(nd, G, int(rng.integers(1, 9)), C, K, inn, filt, stride, dil, pl, pr)
        try:
            binding.wg_problem_normalize(sp)
        except binding.WgradError:
            continue  # no output position
        for kernel in ("auto", "igemm_taps_m", "igemm_taps_mn"):
            for split_k, mode in ((0, "auto"), (1, "direct"), (7, "deterministic")):
                try:
                    ps = binding.wg_plan_string(sp, split_k, mode, 0, kernel=kernel)
                except binding.WgradError as e:
                    assert e.status == 2, (sp, kernel, split_k, mode, e)
                    continue
                f = _plan_fields(ps)
                assert int(f["smem"]) <= 232448, ps
                if f["kernel"] == "depthwise":
                    checked["depthwise"] += 1
                    continue
                w, h, d, n = (int(v[1:]) for v in f["box"].strip("()").split(","))
                KT = w * h * d * n
                assert KT == int(f["KT"]) and KT % 16 == 0 and KT <= 256, ps
                assert int(f["stage_bytes"]) % 1024 == 0, ps
                assert int(f["mt_per_cta"]) * int(f["Nmma"]) <= int(f["tmem_cols"]) <= 512, ps
                if f["taps"] == "mn":
                    checked["mn"] += 1
                    assert sp["stride"] == [1] * nd and int(f["Nmma"]) == 64 * filt[-1] <= 256, ps
                    assert " halo " in ps, ps
                else:
                    checked["m"] += 1
                    if kernel == "igemm_taps_mn":
                        raise AssertionError(f"forced column form planned as rows: {ps}")
    assert min(checked.values()) > 20, checked

