"""GPU parity of the CTA-pair form of the x-taps-on-columns tile (kernel
"igemm_pair": a split's two M-tiles on the two CTAs of a cluster sharing
M = 256 MMAs, tcgen05 .cta_group::2) against the fp64 oracle.

What the pair changes, and so what is checked here: rank 1's X patch is loaded
pair_dh rows further down (its atoms y = 2, 3 at rank 0's offsets), each CTA
stages 32 of the 64 output channels of dY (64-byte swizzle, B atoms of 32
columns one dil_w row apart), rank 1's loads are counted on rank 0's barrier,
and the TMEM columns are ordered (k half, x block, k).  Cases: ragged images,
dilation, asymmetric pads, X = 2, 3, 4 and Y = 3, 4 (the second M-tile half
padding, or full), C below 64, two groups, one image of 3x3, no padding, every
split mode and output type, integer inputs bit for bit, the 56x56 workload at
full size against the single-CTA form, and the two-stage result repeated bit
for bit.
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


def run_gpu(sp, x, dy, split_k, mode, kernel="igemm_pair"):
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
    # 3x3 pad 1 on a ragged image
    spec(2, 1, 2, 64, 64, [13, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    # dilation 2 in both dims (rank 1's patch 4 rows down), 16-bit dW
    spec(2, 1, 3, 64, 64, [9, 20], [3, 3], [1, 1], [2, 2], [2, 2], [2, 2], out_dtype="bf16"),
    # X = 2 (N = 128: 64 columns per CTA) with asymmetric pads
    spec(2, 1, 2, 64, 64, [10, 12], [3, 2], [1, 1], [1, 1], [1, 0], [1, 1]),
    # X = 4 (N = 256), Y = 3
    spec(2, 1, 2, 64, 64, [9, 14], [3, 4], [1, 1], [1, 1], [1, 2], [1, 1]),
    # Y = 4: rank 1's second atom is y = 3, not padding
    spec(2, 1, 2, 64, 64, [12, 9], [4, 3], [1, 1], [1, 1], [2, 1], [1, 1]),
    spec(2, 1, 2, 64, 64, [11, 13], [4, 4], [1, 1], [1, 1], [2, 2], [1, 1], in_dtype="fp16", out_dtype="fp16"),
    # C below 64: rows past the channels are discarded
    spec(2, 1, 2, 40, 64, [9, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 1, 1, 16, 64, [20, 19], [3, 4], [1, 1], [1, 1], [1, 2], [1, 1]),
    # two groups of 64 -> 64
    spec(2, 2, 2, 64, 64, [7, 10], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    # a 3x3 image, one image
    spec(2, 1, 1, 64, 64, [3, 3], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    # no padding: the shifted range reaches past the image on both sides
    spec(2, 1, 4, 64, 64, [12, 30], [3, 3], [1, 1], [1, 1], [0, 0], [0, 0]),
    # many K-tiles
    spec(2, 1, 8, 64, 64, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], in_dtype="fp16"),
]
MODES = [(0, "auto"), (1, "direct"), (3, "deterministic"), (5, "atomic"), (64, "deterministic")]


def _ids(sp):
    return (f"{sp['ndim']}d_G{sp['G']}_C{sp['C']}_K{sp['K']}_in{'x'.join(map(str, sp['in']))}_f"
            f"{'x'.join(map(str, sp['filt']))}_d{''.join(map(str, sp['dil']))}_{sp['in_dtype']}_{sp['out_dtype']}")


@pytest.mark.parametrize("sp", CASES, ids=_ids)
def test_pair_all_modes(sp):
    x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 81, 82)
    dw, A = ref(sp, x, dy)
    for split_k, mode in MODES:
        plan = binding.wg_plan_string(sp, split_k, mode, 0, kernel="igemm_pair")
        assert plan.endswith("code=pair"), plan
        got = run_gpu(sp, x, dy, split_k, mode)
        assert_close(got, dw, A, sp["out_dtype"], f"{_ids(sp)} S={split_k} {mode}: {plan}")


def _random_pair_problems(count, seed):
    # Seeded random problems the pair form admits: 2-D, stride 1, K = 64 (no
    # group fold), C <= 64, 3 or 4 filter rows, 2-4 columns.
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        G = int(rng.choice([1, 1, 2, 3]))
        C = int(rng.choice([8, 16, 24, 32, 40, 56, 64]))
        if (G * C) % 8:
            continue
        filt = [int(rng.choice([3, 4])), int(rng.choice([2, 3, 4]))]
        dil = [int(rng.choice([1, 1, 2])), int(rng.choice([1, 1, 2]))]
        inn = [int(rng.integers(filt[i] * dil[i], 24)) for i in range(2)]
        pl = [int(rng.integers(0, filt[i])) for i in range(2)]
        pr = [int(rng.integers(0, filt[i])) for i in range(2)]
        sp = spec(2, G, int(rng.integers(1, 4)), C, 64, inn, filt, [1, 1], dil, pl, pr,
                  str(rng.choice(["bf16", "fp16"])), str(rng.choice(["fp32", "bf16", "fp16"])))
        try:
            binding.wg_plan_string(sp, 0, "auto", 0, kernel="igemm_pair")
        except binding.WgradError:
            continue
        out.append(sp)
    return out


def test_pair_random_problems():
    for sp in _random_pair_problems(12, 4242):
        x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 85, 86)
        dw, A = ref(sp, x, dy)
        for split_k, mode in ((0, "auto"), (1, "direct"), (7, "deterministic"), (3, "atomic")):
            got = run_gpu(sp, x, dy, split_k, mode)
            assert_close(got, dw, A, sp["out_dtype"], f"{_ids(sp)} S={split_k} {mode}")


@pytest.mark.parametrize("sp", [CASES[i] for i in (0, 1, 2, 3, 4, 6, 8, 10)], ids=_ids)
def test_pair_integer_inputs_bitwise(sp):
    x, dy = make_inputs(sp, ("int", -2, 2), 83, 84)
    dw, _ = ref(sp, x, dy)
    assert np.all(np.abs(dw) < 2 ** 24)
    for split_k, mode in MODES:
        if mode == "atomic" and sp["out_dtype"] != "fp32":
            continue
        got = run_gpu(sp, x, dy, split_k, mode)
        np.testing.assert_array_equal(got, dw, err_msg=f"{_ids(sp)} S={split_k} {mode}")


def test_56x56_workload_pair_and_single():
    sp, (x, dy) = workload_inputs("2d_dense_n32_h56_c64_k64")
    dw, A = ref(sp, x, dy)
    assert binding.wg_plan_string(sp, kernel="igemm_pair").endswith("code=pair")
    got = run_gpu(sp, x, dy, 0, "auto")
    assert_close(got, dw, A, sp["out_dtype"], binding.wg_plan_string(sp, kernel="igemm_pair"))
    single = run_gpu(sp, x, dy, 0, "auto", kernel="igemm_taps_mn")
    assert_close(single, dw, A, sp["out_dtype"], "single-CTA form")
    # Two-stage: the same bits on every call.
    again = run_gpu(sp, x, dy, 0, "deterministic")
    np.testing.assert_array_equal(again, run_gpu(sp, x, dy, 0, "deterministic"))
