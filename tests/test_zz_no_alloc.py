"""GPU test of wg_conv_bwd_weight_noalloc, the entry point for callers that cannot
allocate device memory (a plug-in whose host owns every device allocation, code
under a fixed memory budget, a path that cannot take cudaMalloc's implicit
synchronisation).  It takes its split-K workspace from an array compiled into
the library instead of from the caller.

Each case calls it twice in a row through the C ABI and compares both results
with the regular entry point's, within the parity tests' tolerance.  Collected
last (file name) so that a run stopping at the first failure has run every
other test before it; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import oracle
from implicit_gemm_gb300 import binding, build
from tests.common import assert_close, make_inputs, spec, workload_inputs

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


def _out(sp):
    return torch.full((sp["G"], sp["K"], *sp["filt"], sp["C"]), float("nan"),
                      dtype=getattr(torch, _TDT[sp["out_dtype"]]), device="cuda")


CASES = [
    ("small_split4", spec(2, 2, 2, 24, 16, [11, 9], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]), 4, "deterministic", 0),
    ("dense_56x56_auto", None, 0, "auto", 0),
    ("depthwise_3d_split3", spec(3, 8, 2, 1, 1, [5, 6, 5], [3, 3, 3], [1, 1, 1], [1, 1, 1], [1, 1, 1], [1, 1, 1]),
     3, "deterministic", 0),
    ("depthwise_2d_auto_split", spec(2, 64, 3, 1, 1, [12, 10], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]), 0,
     "deterministic", 8),
    # The automatic split degree's partial sums need more than the 16 MiB array
    # (S = 8 partials of 2.25 MiB): the call caps the split degree to 7.
    ("capped_auto_split", spec(2, 1, 8, 256, 256, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]), 0,
     "deterministic", 0),
    # One partial sum of dW is 9 MiB, so not even two fit: the call runs one
    # split (direct mode, no workspace).
    ("direct_when_two_partials_do_not_fit", spec(2, 1, 8, 512, 512, [14, 14], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
     0, "deterministic", 0),
]

SCRATCH_BYTES = 16 << 20


@pytest.mark.parametrize("name,sp,split_k,mode,gm", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_regular_entry_twice(name, sp, split_k, mode, gm):
    if sp is None:
        sp, (x, dy) = workload_inputs("2d_dense_n32_h56_c64_k64")
    else:
        x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 91, 92)
    dt = sp["in_dtype"]
    if name in ("capped_auto_split", "direct_when_two_partials_do_not_fit"):
        # the case must reach the branch it is named for
        assert binding.wg_workspace_size(sp, split_k, mode, gm) > SCRATCH_BYTES
    ref_dw, A = oracle.wgrad(sp, oracle.decode(x, dt), oracle.decode(dy, dt))
    xd, dyd = _dev(x, dt), _dev(dy, dt)
    ref = _out(sp)
    binding.conv_bwd_weight(sp, xd, dyd, split_k, mode, gm, out=ref)
    binding.wg_check_status()
    ref_np = ref.float().cpu().numpy().astype(np.float64)
    first = None
    for call in range(2):
        got = _out(sp)
        binding.wg_conv_bwd_weight_noalloc(sp, xd, dyd, got, split_k, mode, gm)
        binding.wg_check_status()
        got_np = got.float().cpu().numpy().astype(np.float64)
        assert_close(got_np, ref_np, A, sp["out_dtype"], f"{name} call {call}")
        assert_close(got_np, ref_dw, A, sp["out_dtype"], f"{name} call {call} against the oracle")
        if first is None:
            first = got_np
        elif "mode=atomic" not in binding.wg_plan_string(sp, split_k, mode, gm):
            # the same bits again (atomic adds may sum in another order)
            np.testing.assert_array_equal(got_np, first)


def test_noalloc_rejects_oversized_split():
    sp, (x, dy) = workload_inputs("2d_dense_n32_h56_c64_k64")
    xd, dyd = _dev(x, sp["in_dtype"]), _dev(dy, sp["in_dtype"])
    out = _out(sp)
    with pytest.raises(binding.WgradError) as e:
        binding.wg_conv_bwd_weight_noalloc(sp, xd, dyd, out, 200, "deterministic", cluster=1)
    assert e.value.status == 4
    assert "scratch" in binding.wg_last_error()
