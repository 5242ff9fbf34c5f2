"""GPU parity on seeded random problems: 1-, 2- and 3-D, strides, dilations,
asymmetric pads, groups (folded or not), depthwise, 16-bit and fp32 dW, through
every kernel selector that accepts the problem (automatic, every tap on the MMA
rows, the x taps on the columns, their CTA-pair form, the depthwise kernel) in
the automatic, direct, deterministic and atomic split modes (a 16-bit dW
through its fp32 copy and the cast kernel), each compared with the fp64 oracle.
"""
import numpy as np
import pytest

import oracle
from implicit_gemm_gb300 import binding, build
from tests.common import assert_close, make_inputs, spec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

_TDT = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    binding.load()


def _problems(count, seed):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        nd = int(rng.choice([1, 2, 2, 2, 3]))
        G = int(rng.choice([1, 1, 2, 4, 8]))
        C = int(rng.choice([8, 16, 24, 40, 64, 72, 128]))
        K = int(rng.choice([8, 16, 32, 64, 64, 96, 128]))
        if rng.random() < 0.15:
            C = K = 1
            G = int(rng.choice([8, 16, 24, 64]))
        if (G * C) % 8 or (G * K) % 8:
            continue
        lim = {1: 48, 2: 14, 3: 7}[nd]
        filt = [int(rng.choice([1, 2, 3, 3, 4])) for _ in range(nd)]
        stride = [int(rng.choice([1, 1, 1, 2])) for _ in range(nd)]
        dil = [int(rng.choice([1, 1, 2])) for _ in range(nd)]
        inn = [int(rng.integers(2, lim + 1)) for _ in range(nd)]
        pl = [int(rng.integers(0, f)) for f in filt]
        pr = [int(rng.integers(0, f)) for f in filt]
        in_dtype = str(rng.choice(["bf16", "fp16"]))
        out_dtype = str(rng.choice(["fp32", "fp32", "bf16", "fp16"]))
        sp = spec(nd, G, int(rng.integers(1, 4)), C, K, inn, filt, stride, dil, pl, pr, in_dtype, out_dtype)
        try:
            binding.wg_problem_normalize(sp)
        except binding.WgradError:
            continue
        out.append(sp)
    return out


PROBLEMS = _problems(40, 1202)


def _id(sp):
    return (f"{sp['ndim']}d_G{sp['G']}_C{sp['C']}_K{sp['K']}_in{'x'.join(map(str, sp['in']))}_f"
            f"{'x'.join(map(str, sp['filt']))}_s{''.join(map(str, sp['stride']))}"
            f"_d{''.join(map(str, sp['dil']))}_{sp['in_dtype']}_{sp['out_dtype']}")


def _run(sp, x, dy, split_k, mode, kernel):
    out = torch.full((sp["G"], sp["K"], *sp["filt"], sp["C"]), float("nan"), dtype=_TDT[sp["out_dtype"]],
                     device="cuda")
    idt = torch.bfloat16 if sp["in_dtype"] == "bf16" else torch.float16
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(idt)
    dyd = torch.from_numpy(np.ascontiguousarray(dy).view(np.int16)).cuda().view(idt)
    binding.conv_bwd_weight(sp, xd, dyd, split_k, mode, 0, out=out, kernel=kernel)
    binding.wg_check_status()
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("sp", PROBLEMS, ids=_id)
def test_random_problem_every_kernel(sp):
    x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 81, 82)
    dt = sp["in_dtype"]
    dw, A = oracle.wgrad(sp, oracle.decode(x, dt), oracle.decode(dy, dt))
    ran = 0
    for kernel in ("auto", "igemm_taps_m", "igemm_taps_mn", "igemm_pair", "depthwise"):
        for split_k, mode in ((0, "auto"), (1, "direct"), (6, "deterministic"), (5, "atomic")):
            try:
                plan = binding.wg_plan_string(sp, split_k, mode, 0, kernel=kernel)
            except binding.WgradError as e:
                assert e.status == 2, e  # not supported for this problem: skipped
                continue
            got = _run(sp, x, dy, split_k, mode, kernel)
            assert_close(got, dw, A, sp["out_dtype"], f"{_id(sp)} {kernel} S={split_k} {mode}: {plan}")
            ran += 1
    assert ran >= 3
