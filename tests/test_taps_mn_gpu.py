"""GPU parity of the tensor-core kernel's x-taps-on-columns tile (kernel
"igemm_taps_mn": D[(z, y, c), (x, k)] summed over pixels shifted by x along W)
against the fp64 oracle.

The form changes what the MMA rows and columns mean, the pixel range along W
(Wo + (X-1)*dil_w positions, dY zero outside [0, Wo)), the dY staging (one
patch per K-tile read as X row-shifted column blocks) and the epilogue's tap of
each column block, so it is checked on its own: ragged images, dilation,
asymmetric pads, X = 2, 3 and 4, 1-D and 3-D, K and C above 64, groups (and
small groups folded into one tile), channel counts that are not multiples of
64, every split mode, integer inputs
bit for bit, and the 56x56 workload at full size in both tile forms.
"""
import numpy as np
import pytest

import oracle
from implicit_gemm_gb300 import binding, build
from tests.common import assert_close, make_inputs, spec, workload_inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    binding.load()


_TDT = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}


def to_dev(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


def run_gpu(sp, x, dy, split_k, mode, kernel):
    out = torch.full((sp["G"], sp["K"], *sp["filt"], sp["C"]), float("nan"), dtype=_TDT[sp["out_dtype"]],
                     device="cuda")
    binding.conv_bwd_weight(sp, to_dev(x, sp["in_dtype"]), to_dev(dy, sp["in_dtype"]), split_k, mode, 0, out=out,
                            kernel=kernel)
    binding.wg_check_status()
    return out.float().cpu().numpy().astype(np.float64)


def ref(sp, x, dy):
    dt = sp["in_dtype"]
    return oracle.wgrad(sp, oracle.decode(x, dt), oracle.decode(dy, dt))


CASES = [
    # 3x3 pad 1 on a ragged image (Wo = 11: 13 shifted positions along W)
    spec(2, 1, 2, 64, 64, [13, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    # dilation 2 in both dims, 16-bit dW
    spec(2, 1, 3, 64, 64, [9, 20], [3, 3], [1, 1], [2, 2], [2, 2], [2, 2], out_dtype="bf16"),
    # X = 2 with asymmetric pads (N = 128 per MMA)
    spec(2, 1, 2, 64, 64, [10, 12], [2, 2], [1, 1], [1, 1], [0, 1], [1, 0]),
    # X = 4 (N = 256), Y = 3, asymmetric pads
    spec(2, 1, 2, 64, 64, [9, 14], [3, 4], [1, 1], [1, 1], [1, 2], [1, 1]),
    # 1-D, dilation 3, fp16
    spec(1, 1, 3, 64, 64, [50], [3], [1], [3], [3], [3], in_dtype="fp16"),
    # 3-D: the (z, y) taps stay on the rows
    spec(3, 1, 2, 64, 64, [5, 6, 7], [3, 3, 3], [1, 1, 1], [1, 1, 1], [1, 1, 1], [1, 1, 1]),
    # two N-tiles of K; two channel chunks per (z, y)
    spec(2, 1, 2, 64, 128, [8, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 1, 2, 128, 64, [8, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], in_dtype="fp16", out_dtype="fp16"),
    # groups; a partial channel chunk; groups of 72 channels (two chunks, the window not 64-aligned)
    spec(2, 2, 2, 64, 64, [7, 10], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 1, 2, 40, 64, [9, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 3, 2, 72, 64, [6, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    # a 3x3 image, one image
    spec(2, 1, 1, 64, 64, [3, 3], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    # small groups folded into one tile (block-diagonal mask): 8 groups of 8 per
    # 64-wide window; a 128-wide k window; 12 groups of 16; 10 groups (the last
    # block half empty)
    spec(2, 32, 2, 8, 8, [9, 10], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 8, 3, 8, 16, [14, 14], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], out_dtype="bf16"),
    spec(2, 12, 2, 16, 16, [7, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], in_dtype="fp16"),
    spec(2, 10, 2, 8, 8, [8, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    # no padding, so the shifted range reaches past the image on both sides
    spec(2, 1, 4, 64, 64, [12, 30], [3, 3], [1, 1], [1, 1], [0, 0], [0, 0]),
]
MODES = [(0, "auto"), (1, "direct"), (3, "deterministic"), (5, "atomic"), (64, "deterministic")]


def _ids(sp):
    return (f"{sp['ndim']}d_G{sp['G']}_C{sp['C']}_K{sp['K']}_in{'x'.join(map(str, sp['in']))}_f"
            f"{'x'.join(map(str, sp['filt']))}_d{''.join(map(str, sp['dil']))}_{sp['in_dtype']}_{sp['out_dtype']}")


@pytest.mark.parametrize("sp", CASES, ids=_ids)
def test_taps_mn_all_modes(sp):
    x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 71, 72)
    dw, A = ref(sp, x, dy)
    for split_k, mode in MODES:
        if mode == "atomic" and sp["out_dtype"] != "fp32":
            continue
        plan = binding.wg_plan_string(sp, split_k, mode, 0, kernel="igemm_taps_mn")
        assert " taps=mn " in plan, plan
        got = run_gpu(sp, x, dy, split_k, mode, "igemm_taps_mn")
        assert_close(got, dw, A, sp["out_dtype"], f"{_ids(sp)} S={split_k} {mode}: {plan}")


@pytest.mark.parametrize("sp", [CASES[i] for i in (0, 2, 3, 4, 5, 7, 10, 12, 14, 15, 16)], ids=_ids)
def test_taps_mn_integer_inputs_bitwise(sp):
    x, dy = make_inputs(sp, ("int", -2, 2), 73, 74)
    dw, _ = ref(sp, x, dy)
    assert np.all(np.abs(dw) < 2 ** 24)
    for split_k, mode in MODES:
        if mode == "atomic" and sp["out_dtype"] != "fp32":
            continue
        got = run_gpu(sp, x, dy, split_k, mode, "igemm_taps_mn")
        np.testing.assert_array_equal(got, dw, err_msg=f"{_ids(sp)} S={split_k} {mode}")


@pytest.mark.parametrize("kernel", ["igemm_taps_mn", "igemm_taps_m"])
def test_56x56_workload_both_forms(kernel):
    sp, (x, dy) = workload_inputs("2d_dense_n32_h56_c64_k64")
    dw, A = ref(sp, x, dy)
    plan = binding.wg_plan_string(sp, 0, "auto", 0, kernel=kernel)
    assert (" taps=mn " in plan) == (kernel == "igemm_taps_mn"), plan
    got = run_gpu(sp, x, dy, 0, "auto", kernel)
    assert_close(got, dw, A, sp["out_dtype"], plan)
