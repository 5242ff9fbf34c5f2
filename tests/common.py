"""Shared helpers for the parity tests: workloads, input generation, the tolerance rule.

The tolerance is the one the weight-gradient task states for this path:
|gpu - ref| <= 1e-3 * A + 1e-6 per element, A = sum |dY * X| (from the oracle),
plus one unit in the last place of the reference when dW is stored in a 16-bit
format (bf16: 2^(floor(log2|v|) - 7); fp16: 2^(floor(log2|v|) - 10), with the
smallest normal's ulp for tiny values).
"""
from __future__ import annotations

import numpy as np

import oracle
from implicit_gemm_gb300 import synth


def spec(ndim, G, N, C, K, inn, filt, stride=None, dil=None, pl=None, pr=None, in_dtype="bf16",
         out_dtype="fp32"):
    one, zero = [1] * ndim, [0] * ndim
    return {"ndim": ndim, "G": G, "N": N, "C": C, "K": K, "in": list(inn), "filt": list(filt),
            "stride": list(stride or one), "dil": list(dil or one), "pad_l": list(pl or zero),
            "pad_r": list(pr or zero), "in_dtype": in_dtype, "out_dtype": out_dtype}


# The five workloads the path is measured on (names say what they are).
WORKLOADS = {
    "2d_tiny_n1_h8_c16_k32": (spec(2, 1, 1, 16, 32, [8, 8], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32"),
                              ("uniform", -1.0, 1.0), 1),
    "2d_dense_n32_h56_c64_k64": (spec(2, 1, 32, 64, 64, [56, 56], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16",
                                      "bf16"), ("uniform", -1.0, 1.0), 2),
    "2d_grouped_g32_c8_k8_n32_h28": (spec(2, 32, 32, 8, 8, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16",
                                          "fp32"), ("normal", 0.0, 1.0), 3),
    "2d_depthwise_g512_n64_h28": (spec(2, 512, 64, 1, 1, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16",
                                       "fp32"), ("uniform", -1.0, 1.0), 4),
    "3d_n4_d16_c128_k96_s2": (spec(3, 1, 4, 128, 96, [16, 16, 16], [3, 3, 3], [2, 2, 2], [1, 1, 1], [1, 1, 1],
                                   [1, 1, 1], "fp16", "fp32"), ("normal", 0.0, 0.5), 5),
    # 1x1 filters: stride 1 pad 0 (a plain batched GEMM) and stride 2 pad 0 (a strided GEMM).
    "2d_1x1_n32_h56_c64_k256": (spec(2, 1, 32, 64, 256, [56, 56], [1, 1], [1, 1], [1, 1], [0, 0], [0, 0], "bf16",
                                     "fp32"), ("uniform", -1.0, 1.0), 6),
    "2d_1x1s2_n32_h56_c256_k128": (spec(2, 1, 32, 256, 128, [56, 56], [1, 1], [2, 2], [1, 1], [0, 0], [0, 0],
                                        "bf16", "fp32"), ("uniform", -1.0, 1.0), 7),
}


def make_inputs(sp, dist=("uniform", -1.0, 1.0), seed_x=1000, seed_dy=2000):
    """Seeded X and dY as 16-bit words in the problem's input dtype."""
    sh = oracle.shapes(sp)
    nx, ndy = int(np.prod(sh["x"])), int(np.prod(sh["dy"]))
    x = synth.tensor_bits(seed_x, nx, sp["in_dtype"], *dist).reshape(sh["x"])
    dy = synth.tensor_bits(seed_dy, ndy, sp["in_dtype"], *dist).reshape(sh["dy"])
    return x, dy


def workload_inputs(name):
    sp, dist, i = WORKLOADS[name]
    return sp, make_inputs(sp, dist, 1000 + i, 2000 + i)


def ulp(v, out_dtype):
    a = np.abs(np.asarray(v, dtype=np.float64))
    if out_dtype == "bf16":
        mant, emin = 7, -126
    elif out_dtype == "fp16":
        mant, emin = 10, -14
    else:
        return np.zeros_like(a)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** emin)))
    return 2.0 ** (e - mant)


def tolerance(ref, A, out_dtype):
    return 1e-3 * np.asarray(A) + 1e-6 + ulp(ref, out_dtype)


def assert_close(gpu, ref, A, out_dtype, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert not np.isnan(gpu).any(), f"{what}: {int(np.isnan(gpu).sum())} elements unwritten or NaN"
    err = np.abs(gpu - ref)
    tol = tolerance(ref, A, out_dtype)
    bad = err > tol
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} elements out of tolerance; first flat index {i}: "
                             f"gpu {gpu.ravel()[i]!r} ref {ref.ravel()[i]!r} tol {tol.ravel()[i]!r} "
                             f"max err/tol {float(np.max(err / tol)):.3g}")
