"""GPU tests of wg_conv_bwd_weight_host: inputs and result in host memory.

The call copies X and dY into the caller's device buffers, computes exactly as
wg_conv_bwd_weight on them and copies dW back, so deterministic and direct plans
must give the device entry point's dW bit for bit; atomic plans add in another
order and are checked against it within a few fp32 ulps.  Device-entry results
are themselves checked against the oracle by the parity tests.  Cases: dense,
depthwise, 1x1 and grouped workloads, direct and split modes on a 7-image batch,
atomic mode, a cluster plan, pageable host memory, and staging buffers
pre-filled with NaN (every byte must be copied).
"""
import numpy as np
import pytest

from implicit_gemm_gb300 import binding, build
from tests.common import WORKLOADS, make_inputs, spec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

_TDT = {"fp32": "float32", "bf16": "bfloat16", "fp16": "float16"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    binding.load()


def _tensors(sp, seed):
    x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), seed, seed + 1)
    idt = torch.bfloat16 if sp["in_dtype"] == "bf16" else torch.float16
    xh = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(idt)
    dyh = torch.from_numpy(np.ascontiguousarray(dy).view(np.int16)).view(idt)
    return xh, dyh


def _dw_shape(sp):
    return (sp["G"] * sp["K"] * int(np.prod(sp["filt"])) * sp["C"],)


def _run_both(sp, seed, pinned=True, **kw):
    xh, dyh = _tensors(sp, seed)
    odt = getattr(torch, _TDT[sp["out_dtype"]])
    mode = kw.get("mode", "auto")
    if mode == "atomic":
        odt = torch.float32
    # Device entry point on resident inputs.
    x, dy = xh.cuda(), dyh.cuda()
    dw_ref = torch.empty(_dw_shape(sp), dtype=odt, device="cuda")
    nb = binding.wg_workspace_size(sp, kw.get("split_k", 0), mode, 0, cluster=kw.get("cluster", 0))
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    binding.wg_conv_bwd_weight(sp, x, dy, dw_ref, workspace=ws, ws_bytes=nb, **kw)
    # Host entry point: staging buffers full of NaN, result into host memory.
    if pinned:
        xh, dyh = xh.pin_memory(), dyh.pin_memory()
    x_dev = torch.full_like(x, float("nan"))
    dy_dev = torch.full_like(dy, float("nan"))
    dw_dev = torch.full_like(dw_ref, float("nan"))
    dw_host = torch.full(_dw_shape(sp), float("nan"), dtype=odt)
    if pinned:
        dw_host = dw_host.pin_memory()
    ws2 = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    binding.wg_conv_bwd_weight_host(sp, xh, dyh, dw_host, x_dev, dy_dev, dw_dev, workspace=ws2, ws_bytes=nb, **kw)
    torch.cuda.synchronize()
    binding.wg_check_status()
    assert torch.equal(x_dev.view(torch.int16).cpu(), xh.view(torch.int16))
    assert torch.equal(dy_dev.view(torch.int16).cpu(), dyh.view(torch.int16))
    return dw_ref.cpu(), dw_host.clone()


def _bits(t):
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16).numpy()


@pytest.mark.parametrize("name", ["2d_dense_n32_h56_c64_k64", "2d_depthwise_g512_n64_h28", "2d_1x1_n32_h56_c64_k256",
                                  "2d_grouped_g32_c8_k8_n32_h28"])
def test_host_entry_bitwise_equals_device_entry(name):
    # Two-stage mode, so that both entry points give one bit pattern.
    sp = WORKLOADS[name][0]
    ref, got = _run_both(sp, 401, mode="deterministic")
    np.testing.assert_array_equal(_bits(got), _bits(ref))


def test_host_entry_direct_and_split_modes():
    sp = spec(2, 1, 7, 64, 64, [112, 96], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32")
    for kw in ({"split_k": 0, "mode": "deterministic"}, {"split_k": 1, "mode": "direct"},
               {"split_k": 13, "mode": "deterministic"}):
        ref, got = _run_both(sp, 411, **kw)
        np.testing.assert_array_equal(_bits(got), _bits(ref), err_msg=str(kw))


def test_host_entry_atomic_within_tolerance():
    sp = spec(2, 1, 16, 64, 64, [56, 56], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32")
    ref, got = _run_both(sp, 421, split_k=40, mode="atomic")
    r, g = ref.double().numpy(), got.double().numpy()
    # The same products summed in another order: a few ulps of fp32 over 40 partials.
    assert np.max(np.abs(g - r)) <= 1e-5 * (np.max(np.abs(r)) + 1.0)


def test_host_entry_cluster_plan_and_pageable_memory():
    sp = spec(2, 1, 16, 64, 64, [56, 56], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "bf16")
    ref, got = _run_both(sp, 431, split_k=32, mode="deterministic", cluster=2)
    np.testing.assert_array_equal(_bits(got), _bits(ref))
    ref, got = _run_both(sp, 441, pinned=False, mode="deterministic")
    np.testing.assert_array_equal(_bits(got), _bits(ref))
