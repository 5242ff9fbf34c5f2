"""The deterministic mode's reduction order, bit for bit.

After a deterministic call the workspace still holds the fp32 partial sums of
every split.  This test re-adds them on the host in the order the header
documents -- for S >= 8 four contiguous ranges of splits, each summed in index
order in fp32, then the four range sums in range order; for S < 8 index order --
rounds to the output type (round to nearest even) and requires dW to match bit
for bit, for split degrees below and above 8, 16-bit and fp32 dW, 2-D and 3-D
problems, a grouped one, and depthwise problems (whose workspace holds all of
dW as one row).  The workspace layout is the documented one: dW as
rows of L = T*C elements per (g, k), rows cut into slices of W elements, the S
partials of a slice stored together.
"""
import numpy as np
import pytest

from implicit_gemm_gb300 import binding, build
from tests.common import make_inputs, spec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    binding.load()


def _slice_width(L):
    if L <= 128:
        return -(-L // 4) * 4
    for w in range(128, 63, -4):
        if L % w == 0:
            return w
    return 128


def _rne_bf16(a32):
    u = a32.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _expected(ws, sp, S, out_dtype, depthwise_kernel):
    T = int(np.prod(sp["filt"]))
    # Tensor-core kernel: one row per (g, k); depthwise kernel: all of dW as one row.
    rows, L = (1, sp["G"] * T) if depthwise_kernel else (sp["G"] * sp["K"], T * sp["C"])
    W = _slice_width(L)
    nj = -(-L // W)
    part = ws[: rows * nj * S * W].reshape(rows, nj, S, W)
    G = 4 if S >= 8 else 1
    sums = []
    for g in range(G):
        s0, s1 = S * g // G, S * (g + 1) // G
        a = part[:, :, s0, :].copy()
        for s in range(s0 + 1, s1):
            a = (a + part[:, :, s, :]).astype(np.float32)
        sums.append(a)
    tot = sums[0]
    for a in sums[1:]:
        tot = (tot + a).astype(np.float32)
    dw = tot.reshape(rows, nj * W)[:, :L].reshape(-1)
    if out_dtype == "fp32":
        return dw.view(np.uint32)
    if out_dtype == "bf16":
        return _rne_bf16(dw)
    return dw.astype(np.float16).view(np.uint16)


CASES = [
    # (spec, split_k): S >= 8 and S < 8, 16-bit and fp32 dW, a split degree of
    # several hundred, grouped, 3-D strided.
    (spec(2, 1, 8, 64, 64, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "bf16"), 40),
    (spec(2, 1, 8, 64, 64, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32"), 5),
    (spec(2, 1, 8, 64, 64, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "bf16"), 392),
    (spec(2, 4, 4, 16, 24, [20, 20], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "fp16", "fp16"), 12),
    (spec(3, 1, 2, 32, 32, [8, 8, 8], [3, 3, 3], [2, 2, 2], [1, 1, 1], [1, 1, 1], [1, 1, 1], "fp16", "fp32"), 16),
    # depthwise kernel
    (spec(2, 512, 8, 1, 1, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32"), 19),
    (spec(2, 64, 4, 1, 1, [20, 20], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "bf16"), 6),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_reduction_order_bitwise(case):
    sp, S = CASES[case]
    plan = binding.wg_plan_string(sp, S, "deterministic", 0)
    assert f" S={S} " in plan
    depthwise_kernel = plan.startswith("kernel=depthwise")
    x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), 500 + case, 600 + case)
    idt = torch.bfloat16 if sp["in_dtype"] == "bf16" else torch.float16
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(idt).cuda()
    dyd = torch.from_numpy(np.ascontiguousarray(dy).view(np.int16)).view(idt).cuda()
    odt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[sp["out_dtype"]]
    n_dw = sp["G"] * sp["K"] * int(np.prod(sp["filt"])) * sp["C"]
    dw = torch.empty(n_dw, dtype=odt, device="cuda")
    nb = binding.wg_workspace_size(sp, S, "deterministic", 0)
    ws = torch.empty(nb // 4, dtype=torch.float32, device="cuda")
    binding.wg_conv_bwd_weight(sp, xd, dyd, dw, S, "deterministic", 0, ws, nb)
    binding.wg_check_status()
    got = dw.cpu().view(torch.int32 if odt == torch.float32 else torch.int16).numpy()
    want = _expected(ws.cpu().numpy(), sp, S, sp["out_dtype"], depthwise_kernel)
    np.testing.assert_array_equal(got.view(want.dtype), want, err_msg=plan)
