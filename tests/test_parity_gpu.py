"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by element.

* every full-size workload in the launch configurations the bench times (and the
  other listed modes), every element compared;
* small problems spanning several tiles and ragged tails over 1-D/2-D/3-D,
  strides, dilations, asymmetric pads, group sizes (cpg 4, 8, 12, 24, 64, 128),
  16-bit outputs, both input dtypes and every split mode;
* integer-valued inputs (exact in bf16/fp16, partial sums below 2^24): the GPU
  result must equal the oracle bit for bit in every mode;
* deterministic split-K repeats bitwise; dW pre-filled with NaN must come back
  fully written.
"""
import numpy as np
import pytest

import oracle
from implicit_gemm_gb300 import binding, build
from tests.common import WORKLOADS, assert_close, make_inputs, spec, workload_inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    binding.load()


def to_dev(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


_TDT = {"fp32": "float32", "bf16": "bfloat16", "fp16": "float16"}


def run_gpu(sp, x, dy, split_k=0, mode="auto", gm=0, xd=None, dyd=None, cluster=0, kernel="auto"):
    xd = to_dev(x, sp["in_dtype"]) if xd is None else xd
    dyd = to_dev(dy, sp["in_dtype"]) if dyd is None else dyd
    out = torch.full((sp["G"], sp["K"], *sp["filt"], sp["C"]), float("nan"),
                     dtype=getattr(torch, _TDT[sp["out_dtype"]]), device="cuda")
    binding.conv_bwd_weight(sp, xd, dyd, split_k, mode, gm, out=out, cluster=cluster, kernel=kernel)
    binding.wg_check_status()
    return out.float().cpu().numpy().astype(np.float64)


def ref(sp, x, dy):
    dt = sp["in_dtype"]
    return oracle.wgrad(sp, oracle.decode(x, dt), oracle.decode(dy, dt))


_WCACHE = {}


def workload(name):
    if name not in _WCACHE:
        sp, (x, dy) = workload_inputs(name)
        _WCACHE.clear()
        _WCACHE[name] = (sp, x, dy, ref(sp, x, dy))
    return _WCACHE[name]


# (workload, split_k, mode, group_merge, cluster)
WORKLOAD_MODES = [
    ("2d_tiny_n1_h8_c16_k32", 0, "auto", 0, 0),
    ("2d_tiny_n1_h8_c16_k32", 4, "direct", 0, 4),
    ("2d_dense_n32_h56_c64_k64", 1, "direct", 0, 0),
    ("2d_dense_n32_h56_c64_k64", 4, "deterministic", 0, 1),
    ("2d_dense_n32_h56_c64_k64", 0, "auto", 0, 0),
    ("2d_dense_n32_h56_c64_k64", 0, "auto", 0, 1),
    ("2d_dense_n32_h56_c64_k64", 0, "auto", 0, 2),
    ("2d_dense_n32_h56_c64_k64", 0, "auto", 0, 4),
    ("2d_dense_n32_h56_c64_k64", 8, "direct", 0, 8),
    ("2d_grouped_g32_c8_k8_n32_h28", 0, "auto", 0, 0),
    ("2d_grouped_g32_c8_k8_n32_h28", 0, "atomic", 0, 0),
    ("2d_grouped_g32_c8_k8_n32_h28", 0, "deterministic", 0, 0),
    ("2d_grouped_g32_c8_k8_n32_h28", 32, "deterministic", 0, 4),
    ("2d_grouped_g32_c8_k8_n32_h28", 16, "atomic", 0, 8),
    ("2d_depthwise_g512_n64_h28", 0, "auto", 0, 0),
    ("2d_depthwise_g512_n64_h28", 0, "deterministic", 0, 0),
    ("2d_depthwise_g512_n64_h28", 0, "deterministic", 1, 0),
    ("2d_depthwise_g512_n64_h28", 0, "deterministic", 2, 0),
    ("2d_depthwise_g512_n64_h28", 0, "deterministic", 4, 0),
    ("2d_depthwise_g512_n64_h28", 0, "deterministic", 8, 0),
    ("2d_depthwise_g512_n64_h28", 0, "auto", 2, 0),
    ("2d_depthwise_g512_n64_h28", 0, "atomic", 8, 0),
    ("2d_depthwise_g512_n64_h28", 1, "direct", 8, 0),
    ("3d_n4_d16_c128_k96_s2", 8, "atomic", 0, 0),
    ("3d_n4_d16_c128_k96_s2", 8, "deterministic", 0, 1),
    ("3d_n4_d16_c128_k96_s2", 16, "deterministic", 0, 2),
    ("3d_n4_d16_c128_k96_s2", 0, "auto", 0, 0),
    ("3d_n4_d16_c128_k96_s2", 0, "deterministic", 0, 0),
    ("2d_1x1_n32_h56_c64_k256", 0, "auto", 0, 0),
    ("2d_1x1_n32_h56_c64_k256", 0, "atomic", 0, 0),
    ("2d_1x1_n32_h56_c64_k256", 0, "deterministic", 0, 0),
    ("2d_1x1s2_n32_h56_c256_k128", 0, "auto", 0, 0),
    ("2d_1x1s2_n32_h56_c256_k128", 0, "deterministic", 0, 0),
    ("2d_1x1s2_n32_h56_c256_k128", 1, "direct", 0, 0),
]


@pytest.mark.parametrize("name,split_k,mode,gm,cluster", WORKLOAD_MODES,
                         ids=[f"{w[0]}-S{w[1]}-{w[2]}-gm{w[3]}-cl{w[4]}" for w in WORKLOAD_MODES])
def test_workload_full(name, split_k, mode, gm, cluster):
    sp, x, dy, (dw, A) = workload(name)
    if not _supported(sp, split_k, mode, gm, cluster):
        pytest.skip("the planner reports this combination as not supported")
    got = run_gpu(sp, x, dy, split_k, mode, gm, cluster=cluster)
    assert_close(got, dw, A, sp["out_dtype"], f"{name} S={split_k} {mode} gm={gm} cluster={cluster}")


def _supported(sp, split_k, mode, gm, cluster):
    """False where the planner answers WG_ERR_NOT_SUPPORTED (e.g. a cluster whose
    partial sums do not fit shared memory); any other error propagates."""
    try:
        binding.wg_plan_string(sp, split_k, mode, gm, cluster=cluster)
    except binding.WgradError as e:
        if e.status == 2:
            return False
        raise
    return True


SMALL = [
    # (spec, modes)
    spec(2, 1, 2, 16, 16, [9, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 1, 3, 64, 64, [13, 10], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], out_dtype="bf16"),
    spec(2, 1, 2, 128, 32, [7, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 1, 2, 24, 40, [10, 7], [3, 2], [2, 1], [1, 2], [0, 1], [2, 0]),
    spec(2, 4, 2, 4, 4, [6, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 2, 2, 12, 12, [7, 7], [3, 3], [1, 1], [2, 2], [2, 2], [2, 2]),
    spec(2, 6, 1, 8, 16, [8, 12], [1, 1]),
    spec(2, 3, 2, 24, 8, [11, 6], [5, 3], [2, 2], [1, 1], [2, 1], [2, 1], in_dtype="fp16", out_dtype="fp16"),
    spec(2, 2, 2, 64, 72, [6, 6], [2, 2], [3, 3], [1, 1], [0, 1], [1, 0]),
    spec(1, 2, 3, 16, 8, [37], [5], [1], [2], [3], [1]),
    spec(1, 1, 2, 48, 24, [29], [3], [2], [1], [1], [0], in_dtype="fp16"),
    spec(3, 1, 2, 32, 16, [5, 6, 7], [3, 3, 3], [1, 1, 1], [1, 1, 1], [1, 1, 1], [1, 1, 1]),
    spec(3, 2, 1, 8, 8, [7, 6, 9], [2, 3, 3], [2, 1, 2], [1, 2, 1], [0, 1, 1], [1, 1, 0]),
    spec(3, 1, 3, 128, 96, [9, 9, 9], [3, 3, 3], [2, 2, 2], [1, 1, 1], [1, 1, 1], [1, 1, 1], in_dtype="fp16"),
    # 1x1: stride 2 pad 0 (strided GEMM), wide channels with a ragged pixel count, 3-D
    spec(2, 1, 2, 48, 40, [11, 9], [1, 1], [2, 2]),
    spec(2, 1, 3, 256, 96, [7, 5], [1, 1], out_dtype="bf16"),
    spec(3, 2, 2, 16, 24, [3, 5, 4], [1, 1, 1], [1, 2, 1], in_dtype="fp16"),
    # depthwise: fast 3x3 window, generic taps, stride, ragged channel block, 1-D
    spec(2, 64, 2, 1, 1, [9, 13], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 72, 3, 1, 1, [10, 7], [3, 2], [2, 1], [1, 2], [1, 0], [0, 1]),
    spec(2, 16, 2, 1, 1, [8, 9], [1, 3], [1, 2], [1, 1], [0, 1], [0, 1], in_dtype="fp16", out_dtype="bf16"),
    spec(1, 24, 3, 1, 1, [40], [3], [1], [1], [1], [1]),
    spec(3, 8, 2, 1, 1, [5, 5, 5], [3, 3, 3], [1, 1, 1], [1, 1, 1], [1, 1, 1], [1, 1, 1]),
]
# (split_k, mode, cluster): 0 = automatic; cluster > 1 adds splits on chip.
MODES = [(0, "auto", 0), (1, "direct", 0), (3, "deterministic", 0), (5, "atomic", 0), (64, "deterministic", 1),
         (64, "deterministic", 8), (8, "deterministic", 2), (4, "direct", 4), (8, "atomic", 8),
         (16, "deterministic", 4)]


def _ids(sp):
    return (f"{sp['ndim']}d_G{sp['G']}_C{sp['C']}_K{sp['K']}_in{'x'.join(map(str, sp['in']))}_f"
            f"{'x'.join(map(str, sp['filt']))}_s{''.join(map(str, sp['stride']))}_{sp['in_dtype']}_{sp['out_dtype']}")


@pytest.mark.parametrize("sp", SMALL, ids=_ids)
def test_small_problems_all_modes(sp):
    x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 7, 8)
    dw, A = ref(sp, x, dy)
    for split_k, mode, cl in MODES:
        if (mode == "atomic" and sp["out_dtype"] != "fp32") or not _supported(sp, split_k, mode, 0, cl):
            continue
        got = run_gpu(sp, x, dy, split_k, mode, cluster=cl)
        assert_close(got, dw, A, sp["out_dtype"], f"{_ids(sp)} S={split_k} {mode} cluster={cl}")


@pytest.mark.parametrize("sp", [SMALL[i] for i in (0, 3, 4, 10, 12, 14, 16, 17, 18)], ids=_ids)
def test_integer_inputs_bitwise(sp):
    x, dy = make_inputs(sp, ("int", -2, 2), 17, 18)
    dw, _ = ref(sp, x, dy)
    assert np.all(np.abs(dw) < 2 ** 24)
    for split_k, mode, cl in MODES:
        if (mode == "atomic" and sp["out_dtype"] != "fp32") or not _supported(sp, split_k, mode, 0, cl):
            continue
        got = run_gpu(sp, x, dy, split_k, mode, cluster=cl)
        np.testing.assert_array_equal(got, dw, err_msg=f"{_ids(sp)} S={split_k} {mode} cluster={cl}")


@pytest.mark.parametrize("gm", [1, 2, 4, 8])
def test_depthwise_merge_degrees_bitwise_equal(gm):
    sp = spec(2, 64, 3, 1, 1, [11, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    x, dy = make_inputs(sp, ("int", -2, 2), 27, 28)
    dw, _ = ref(sp, x, dy)
    got = run_gpu(sp, x, dy, 3, "deterministic", gm)
    np.testing.assert_array_equal(got, dw)


@pytest.mark.parametrize("name", ["2d_dense_n32_h56_c64_k64", "2d_depthwise_g512_n64_h28", "3d_n4_d16_c128_k96_s2"])
def test_deterministic_mode_repeats_bitwise(name):
    sp, x, dy, _ = workload(name)
    xd, dyd = to_dev(x, sp["in_dtype"]), to_dev(dy, sp["in_dtype"])
    a = run_gpu(sp, x, dy, 0, "deterministic", xd=xd, dyd=dyd)
    b = run_gpu(sp, x, dy, 0, "deterministic", xd=xd, dyd=dyd)
    assert np.array_equal(a.view(np.int64), b.view(np.int64))


@pytest.mark.parametrize("split_k,mode", [(8, "atomic"), (8, "deterministic"), (0, "auto")])
def test_3d_ragged_gemmk(split_k, mode):
    # The 3-D stride-2 geometry (C 128, K 96, 3x3x3, pad 1) on 3 images of 13^3:
    # output 7^3, GemmK = 3 * 343 = 1029, not a multiple of any K-tile, in the
    # 3-D workload's modes.
    sp = spec(3, 1, 3, 128, 96, [13, 13, 13], [3, 3, 3], [2, 2, 2], [1, 1, 1], [1, 1, 1], [1, 1, 1],
              in_dtype="fp16", out_dtype="fp32")
    assert binding.wg_problem_normalize(sp) == [7, 7, 7]
    x, dy = make_inputs(sp, ("normal", 0.0, 0.5), 47, 48)
    dw, A = ref(sp, x, dy)
    got = run_gpu(sp, x, dy, split_k, mode)
    assert_close(got, dw, A, sp["out_dtype"], f"3-D ragged S={split_k} {mode}")


DEGENERATE = [
    # the filter covers the whole image: one output position per image
    spec(2, 2, 3, 16, 24, [7, 9], [7, 9]),
    # a 1x1 image with a 1x1 filter; a 1x1 image with a 3x3 filter and pad 1
    spec(2, 1, 5, 16, 16, [1, 1], [1, 1]),
    spec(2, 1, 4, 32, 16, [1, 1], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    # stride larger than the filter: input positions no tap reaches
    spec(2, 1, 2, 16, 16, [13, 13], [2, 2], [5, 5]),
]


@pytest.mark.parametrize("sp", DEGENERATE, ids=_ids)
def test_degenerate_shapes_bitwise(sp):
    x, dy = make_inputs(sp, ("int", -2, 2), 67, 68)
    dw, _ = ref(sp, x, dy)
    for split_k, mode in ((0, "auto"), (1, "direct"), (0, "atomic")):
        got = run_gpu(sp, x, dy, split_k, mode)
        np.testing.assert_array_equal(got, dw, err_msg=f"{_ids(sp)} {mode}")


LARGE = [
    # wide channels: 8 channel chunks per tap, two N-tiles of K
    spec(2, 1, 2, 512, 512, [7, 7], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], out_dtype="bf16"),
    # large filter, large stride (11x11, stride 4), narrow input channels
    spec(2, 1, 2, 8, 64, [35, 39], [11, 11], [4, 4], [1, 1], [2, 3], [2, 1]),
    # long 1-D signal, 31 dilated taps
    spec(1, 2, 2, 16, 16, [1500], [31], [1], [3], [45], [45], in_dtype="fp16"),
    # anisotropic 3-D filter with groups
    spec(3, 4, 2, 32, 32, [6, 9, 12], [3, 5, 7], [1, 1, 1], [1, 1, 1], [1, 2, 3], [1, 2, 3]),
    # many images of 2x2
    spec(2, 1, 512, 32, 48, [2, 2], [2, 2], [1, 1], [1, 1], [0, 0], [0, 0]),
]


@pytest.mark.parametrize("sp", LARGE, ids=_ids)
def test_large_and_unusual_shapes(sp):
    x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 57, 58)
    dw, A = ref(sp, x, dy)
    for split_k, mode in ((0, "auto"), (0, "atomic")):
        if mode == "atomic" and sp["out_dtype"] != "fp32":
            continue
        got = run_gpu(sp, x, dy, split_k, mode)
        assert_close(got, dw, A, sp["out_dtype"], f"{_ids(sp)} {mode}")


def test_more_splits_than_tiles():
    sp = spec(2, 1, 1, 16, 32, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    x, dy = make_inputs(sp, ("int", -2, 2), 37, 38)
    dw, _ = ref(sp, x, dy)
    for split_k, mode, cl in ((7, "deterministic", 0), (7, "atomic", 0), (8, "direct", 8), (16, "deterministic", 4),
                              (16, "atomic", 8)):
        got = run_gpu(sp, x, dy, split_k, mode, cluster=cl)
        np.testing.assert_array_equal(got, dw, err_msg=f"S={split_k} {mode} cluster={cl}")


def test_status_clear_after_runs():
    binding.wg_check_status()


# The depthwise problems again on the tensor-core kernel (block-diagonal tiles).
DW_SMALL = [sp for sp in SMALL if sp["C"] == 1 and sp["K"] == 1]


@pytest.mark.parametrize("sp", DW_SMALL, ids=_ids)
def test_depthwise_on_tensor_cores(sp):
    x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 47, 48)
    dw, A = ref(sp, x, dy)
    for split_k, mode in ((0, "auto"), (1, "direct"), (5, "deterministic"), (3, "atomic")):
        if mode == "atomic" and sp["out_dtype"] != "fp32":
            continue
        got = run_gpu(sp, x, dy, split_k, mode, kernel="igemm")
        assert_close(got, dw, A, sp["out_dtype"], f"{_ids(sp)} igemm S={split_k} {mode}")
    xi, dyi = make_inputs(sp, ("int", -2, 2), 57, 58)
    dwi, _ = ref(sp, xi, dyi)
    np.testing.assert_array_equal(run_gpu(sp, xi, dyi, 4, "deterministic", kernel="igemm"), dwi)


@pytest.mark.parametrize("split_k,mode", [(0, "auto"), (0, "atomic")])
def test_depthwise_workload_on_tensor_cores(split_k, mode):
    sp, x, dy, (dw, A) = workload("2d_depthwise_g512_n64_h28")
    got = run_gpu(sp, x, dy, split_k, mode, kernel="igemm")
    assert_close(got, dw, A, sp["out_dtype"], f"depthwise igemm S={split_k} {mode}")


# Folded groups whose CTAs cover whole groups write their split's dW block from
# shared memory in dW order (plan "out=staged"): 16 groups of 4 channels per
# 64-channel window, both tile forms, atomic and two-stage modes, 16-bit dW
# through the two-stage path.
STAGED_SP = spec(2, 64, 8, 4, 4, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])


def test_staged_output_folded_groups():
    sp = STAGED_SP
    xi, dyi = make_inputs(sp, ("int", -2, 2), 71, 72)
    dwi, _ = ref(sp, xi, dyi)
    x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 73, 74)
    dw, A = ref(sp, x, dy)
    seen = 0
    for kernel in ("auto", "igemm_taps_m", "igemm_taps_mn"):
        for split_k, mode in ((0, "auto"), (0, "deterministic"), (0, "atomic")):
            plan = binding.wg_plan_string(sp, split_k, mode, 0, kernel=kernel)
            seen += "out=staged" in plan
            got = run_gpu(sp, xi, dyi, split_k, mode, kernel=kernel)
            np.testing.assert_array_equal(got, dwi, err_msg=f"{kernel} {mode}: {plan}")
            got = run_gpu(sp, x, dy, split_k, mode, kernel=kernel)
            assert_close(got, dw, A, sp["out_dtype"], f"{kernel} {mode}")
        for odt in ("bf16", "fp16"):
            s16 = dict(sp, out_dtype=odt)
            got = run_gpu(s16, x, dy, 0, "deterministic", kernel=kernel)
            assert_close(got, dw, A, odt, f"{kernel} deterministic {odt}")
    assert seen >= 5, "the staged output was not exercised"
