"""GPU parity of the backward-data (dgrad) kernel against the fp64 oracle, element
by element, through the C ABI.

* small problems over 1-D/2-D/3-D, groups, dilations, asymmetric pads, K and C
  below, at and above one 64-channel chunk, filters whose taps do not all fit
  one stage, 16-bit outputs and both input dtypes;
* integer-valued inputs: the result must equal the oracle bit for bit;
* strides (each dim's positions split into phases with their own taps), including
  phases no tap reaches, which must come out zero;
* the 56x56, C = K = 64 and 3-D stride-2 shapes of the weight-gradient workloads at
  full size;
* dX pre-filled with NaN must come back fully written.
"""
import numpy as np
import pytest

import oracle
from implicit_gemm_gb300 import binding, build, synth
from tests.common import assert_close, make_inputs, spec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

_TDT = {"fp32": "float32", "bf16": "bfloat16", "fp16": "float16"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    binding.load()


def _dev(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)


def _w_bits(sp, dist, seed):
    sh = oracle.shapes(sp)["dw"]
    return synth.tensor_bits(seed, int(np.prod(sh)), sp["in_dtype"], *dist).reshape(sh)


def run_gpu(sp, dy, w):
    dt = sp["in_dtype"]
    out = torch.full((sp["N"], *sp["in"], sp["G"], sp["C"]), float("nan"),
                     dtype=getattr(torch, _TDT[sp["out_dtype"]]), device="cuda")
    binding.conv_bwd_data(sp, _dev(dy, dt), _dev(w, dt), out=out)
    binding.wg_check_status()
    return out.float().cpu().numpy().astype(np.float64)


def ref(sp, dy, w):
    dt = sp["in_dtype"]
    return oracle.dgrad(sp, oracle.decode(dy, dt), oracle.decode(w, dt))


SMALL = [
    spec(2, 1, 2, 16, 16, [9, 11], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 1, 1, 64, 64, [20, 19], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], out_dtype="bf16"),
    spec(2, 1, 2, 128, 96, [10, 13], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 2, 2, 24, 40, [11, 9], [3, 2], [1, 1], [1, 2], [0, 1], [2, 0]),
    spec(2, 4, 2, 8, 8, [7, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 1, 1, 32, 16, [30, 33], [5, 5], [1, 1], [1, 1], [2, 2], [2, 2]),
    spec(2, 2, 3, 16, 24, [7, 6], [1, 1]),
    spec(1, 1, 2, 16, 24, [300], [5], [1], [2], [4], [4]),
    spec(1, 2, 1, 8, 16, [50], [3], [1], [1], [1], [2]),
    spec(3, 1, 1, 16, 16, [5, 6, 7], [3, 3, 3], [1, 1, 1], [1, 1, 1], [1, 1, 1], [1, 1, 1]),
    spec(3, 2, 2, 8, 8, [4, 5, 6], [2, 3, 3], [1, 1, 1], [2, 1, 1], [1, 0, 1], [0, 2, 1]),
    spec(2, 1, 2, 24, 16, [9, 10], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], in_dtype="fp16", out_dtype="fp16"),
    spec(2, 1, 1, 64, 256, [12, 12], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 1, 2, 256, 64, [9, 8], [1, 1]),
    # strides: phases with different tap lists, strides beyond the filter
    # (phases no tap reaches must come out zero), stride with dilation, 1-D, 3-D
    spec(2, 1, 2, 16, 32, [13, 11], [3, 3], [2, 2], [1, 1], [1, 1], [1, 1]),
    spec(2, 1, 2, 64, 48, [14, 15], [1, 1], [2, 2]),
    spec(2, 2, 1, 8, 16, [10, 9], [3, 2], [2, 1], [1, 2], [0, 1], [2, 0]),
    spec(2, 1, 1, 16, 16, [11, 10], [1, 2], [3, 3], [1, 1], [0, 0], [0, 0]),
    spec(2, 1, 2, 24, 8, [12, 12], [3, 3], [2, 2], [2, 2], [2, 1], [1, 2], in_dtype="fp16", out_dtype="fp16"),
    spec(1, 1, 2, 16, 24, [100], [5], [3], [2], [4], [1]),
    spec(3, 1, 2, 16, 16, [7, 8, 9], [3, 3, 3], [2, 2, 2], [1, 1, 1], [1, 1, 1], [1, 1, 1]),
    # group folds (block-diagonal W): full blocks, a partial last block, C = 4, strided
    spec(2, 32, 2, 8, 8, [9, 10], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    spec(2, 12, 2, 8, 8, [7, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], out_dtype="bf16"),
    spec(2, 4, 2, 4, 12, [8, 7], [3, 2], [1, 1], [1, 1], [1, 0], [1, 1]),
    spec(2, 16, 1, 8, 16, [11, 12], [3, 3], [2, 2], [1, 1], [1, 1], [1, 1]),
]


def _ids(sp):
    return (f"{sp['ndim']}d_G{sp['G']}_C{sp['C']}_K{sp['K']}_in{'x'.join(map(str, sp['in']))}_f"
            f"{'x'.join(map(str, sp['filt']))}_{sp['in_dtype']}_{sp['out_dtype']}")


@pytest.mark.parametrize("sp", SMALL, ids=_ids)
def test_dgrad_small(sp):
    _, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 301, 302)
    w = _w_bits(sp, ("uniform", -1.0, 1.0), 303)
    dx, A = ref(sp, dy, w)
    got = run_gpu(sp, dy, w)
    assert_close(got, dx, A, sp["out_dtype"], _ids(sp))


@pytest.mark.parametrize("sp", [SMALL[i] for i in (0, 3, 4, 5, 7, 10, 12, 14, 16, 17, 19, 20, 21, 22, 23, 24)],
                         ids=_ids)
def test_dgrad_integer_bitwise(sp):
    sp = dict(sp, out_dtype="fp32")
    _, dy = make_inputs(sp, ("int", -2, 2), 311, 312)
    w = _w_bits(sp, ("int", -2, 2), 313)
    dx, _ = ref(sp, dy, w)
    assert np.all(np.abs(dx) < 2 ** 24)
    np.testing.assert_array_equal(run_gpu(sp, dy, w), dx)


def test_dgrad_dense_56x56_full():
    sp = spec(2, 1, 32, 64, 64, [56, 56], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], out_dtype="bf16")
    _, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 321, 322)
    w = _w_bits(sp, ("uniform", -1.0, 1.0), 323)
    dx, A = ref(sp, dy, w)
    got = run_gpu(sp, dy, w)
    assert_close(got, dx, A, sp["out_dtype"], "dgrad 56x56")


def test_dgrad_repeats_bitwise():
    sp = SMALL[2]
    _, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 331, 332)
    w = _w_bits(sp, ("uniform", -1.0, 1.0), 333)
    a, b = run_gpu(sp, dy, w), run_gpu(sp, dy, w)
    assert np.array_equal(a.view(np.int64), b.view(np.int64))


def test_dgrad_3d_stride2_full():
    # The geometry of the 3-D weight-gradient workload (16^3, C 128, K 96, stride 2).
    sp = spec(3, 1, 4, 128, 96, [16, 16, 16], [3, 3, 3], [2, 2, 2], [1, 1, 1], [1, 1, 1], [1, 1, 1],
              in_dtype="fp16", out_dtype="fp32")
    _, dy = make_inputs(sp, ("normal", 0.0, 0.5), 341, 342)
    w = _w_bits(sp, ("normal", 0.0, 0.5), 343)
    dx, A = ref(sp, dy, w)
    got = run_gpu(sp, dy, w)
    assert_close(got, dx, A, sp["out_dtype"], "dgrad 3-D stride 2")


def test_dgrad_grouped_full():
    # The geometry of the grouped weight-gradient workload (G 32, C = K = 8, 28x28).
    sp = spec(2, 32, 32, 8, 8, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    _, dy = make_inputs(sp, ("normal", 0.0, 1.0), 351, 352)
    w = _w_bits(sp, ("normal", 0.0, 1.0), 353)
    dx, A = ref(sp, dy, w)
    got = run_gpu(sp, dy, w)
    assert_close(got, dx, A, sp["out_dtype"], "dgrad grouped")
