"""Pins for the fp64 oracle, each independent of the oracle's own code.

* hand-worked golden cases (tests/golden/hand_worked.json);
* an explicit im2col-then-matmul written here from the definition;
* PyTorch's fp64 CPU autograd weight gradient (a library cross-check);
* the adjoint identity <dW, W'> = <dY, conv_fwd(X, W')>, with the forward
  convolution itself pinned to PyTorch;
* 1x1/stride 1/pad 0 reduces to the matmul dY_g^T X_g;
* depthwise (cpg = kpg = 1) equals G independent single-channel problems;
* a filter covering the whole image has the closed form dW = sum_n dY[n] X[n];
* linearity in dY and the absolute-sum output A.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from implicit_gemm_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _prob(ndim, G, N, C, K, inn, filt, stride=None, dil=None, pl=None, pr=None):
    one = [1] * ndim
    zero = [0] * ndim
    return {"ndim": ndim, "G": G, "N": N, "C": C, "K": K, "in": list(inn), "filt": list(filt),
            "stride": list(stride or one), "dil": list(dil or one), "pad_l": list(pl or zero),
            "pad_r": list(pr or zero)}


def _rand(p, seed):
    sh = oracle.shapes(p)
    x = synth.values(seed, int(np.prod(sh["x"])), "uniform").reshape(sh["x"])
    dy = synth.values(seed + 1, int(np.prod(sh["dy"])), "uniform").reshape(sh["dy"])
    return x, dy


def im2col_wgrad(p, x, dy):
    """Weight gradient via an explicit zero-padded im2col matrix and a matmul."""
    nd, G, N, C, K = p["ndim"], p["G"], p["N"], p["C"], p["K"]
    out = oracle.out_dims(p)
    pads = [(0, 0)] + [(p["pad_l"][i], p["pad_r"][i]) for i in range(nd)] + [(0, 0), (0, 0)]
    xp = np.pad(x, pads)
    taps = list(itertools.product(*[range(f) for f in p["filt"]]))
    cols = []
    for t in taps:
        sl = [slice(None)]
        for i in range(nd):
            start = t[i] * p["dil"][i]
            sl.append(slice(start, start + p["stride"][i] * (out[i] - 1) + 1, p["stride"][i]))
        cols.append(xp[tuple(sl)])  # (N, *out, G, C)
    P = N * int(np.prod(out))
    colm = np.stack(cols, axis=-2).reshape(P, G, len(taps), C)  # (P, G, T, C)
    dym = dy.reshape(P, G, K)
    dw = np.empty((G, K, len(taps), C))
    for g in range(G):
        dw[g] = (dym[:, g, :].T @ colm[:, g].reshape(P, len(taps) * C)).reshape(K, len(taps), C)
    return dw.reshape(G, K, *p["filt"], C)


def torch_wgrad(p, x, dy):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    nd, G, N, C, K = p["ndim"], p["G"], p["N"], p["C"], p["K"]
    perm_in = (0, nd + 1, nd + 2) + tuple(range(1, nd + 1))
    xt = torch.from_numpy(np.ascontiguousarray(x)).permute(*perm_in).reshape(N, G * C, *p["in"])
    pad = []
    for i in reversed(range(nd)):
        pad += [p["pad_l"][i], p["pad_r"][i]]
    xt = F.pad(xt, pad)
    w = torch.zeros(G * K, C, *p["filt"], dtype=torch.float64, requires_grad=True)
    conv = {1: F.conv1d, 2: F.conv2d, 3: F.conv3d}[nd]
    yt = conv(xt, w, stride=p["stride"], dilation=p["dil"], groups=G)
    out = oracle.out_dims(p)
    dyt = torch.from_numpy(np.ascontiguousarray(dy)).permute(*perm_in).reshape(N, G * K, *out)
    assert tuple(yt.shape) == (N, G * K, *out)
    yt.backward(dyt)
    g = w.grad.reshape(G, K, C, *p["filt"]).numpy()
    return np.moveaxis(g, 2, -1)


def torch_fwd(p, x, w):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    nd, G, N, C, K = p["ndim"], p["G"], p["N"], p["C"], p["K"]
    perm_in = (0, nd + 1, nd + 2) + tuple(range(1, nd + 1))
    xt = torch.from_numpy(np.ascontiguousarray(x)).permute(*perm_in).reshape(N, G * C, *p["in"])
    pad = []
    for i in reversed(range(nd)):
        pad += [p["pad_l"][i], p["pad_r"][i]]
    xt = F.pad(xt, pad)
    wt = torch.from_numpy(np.ascontiguousarray(np.moveaxis(w, -1, 2))).reshape(G * K, C, *p["filt"])
    conv = {1: F.conv1d, 2: F.conv2d, 3: F.conv3d}[nd]
    yt = conv(xt, wt, stride=p["stride"], dilation=p["dil"], groups=G)
    out = oracle.out_dims(p)
    y = yt.reshape(N, G, K, *out).numpy()
    return np.moveaxis(np.moveaxis(y, 1, -1), 1, -1)  # (N, *out, G, K)


SMALL = [
    _prob(1, 1, 2, 3, 2, [9], [3], [1], [1], [1], [1]),
    _prob(1, 2, 1, 2, 3, [11], [3], [2], [2], [2], [0]),
    _prob(2, 1, 2, 3, 4, [6, 7], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1]),
    _prob(2, 3, 1, 2, 2, [7, 5], [3, 2], [2, 1], [1, 2], [0, 1], [2, 0]),
    _prob(2, 2, 2, 4, 3, [5, 6], [2, 3], [2, 2], [2, 1], [1, 2], [1, 1]),
    _prob(3, 1, 1, 2, 2, [5, 4, 5], [3, 2, 3], [2, 1, 2], [1, 2, 1], [1, 0, 1], [1, 1, 0]),
    _prob(3, 2, 2, 1, 2, [4, 5, 4], [2, 3, 2], [1, 2, 1], [2, 1, 1], [0, 1, 1], [1, 0, 1]),
]


def test_hand_worked_golden():
    with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    assert len(cases) >= 4
    for c in cases:
        dw, ab = oracle.wgrad(c["problem"], np.array(c["x"], float), np.array(c["dy"], float))
        assert dw.ravel().tolist() == c["dw"], c["name"]
        assert np.all(ab.ravel() >= np.abs(dw.ravel()))


@pytest.mark.parametrize("p", SMALL, ids=lambda p: f"{p['ndim']}d_G{p['G']}")
def test_matches_im2col_matmul(p):
    x, dy = _rand(p, 11)
    dw, _ = oracle.wgrad(p, x, dy)
    ref = im2col_wgrad(p, x, dy)
    np.testing.assert_allclose(dw, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("p", SMALL, ids=lambda p: f"{p['ndim']}d_G{p['G']}")
def test_matches_torch_autograd(p):
    x, dy = _rand(p, 21)
    dw, _ = oracle.wgrad(p, x, dy)
    np.testing.assert_allclose(dw, torch_wgrad(p, x, dy), rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("p", SMALL, ids=lambda p: f"{p['ndim']}d_G{p['G']}")
def test_forward_matches_torch_and_adjoint(p):
    x, dy = _rand(p, 31)
    sh = oracle.shapes(p)
    w = synth.values(77, int(np.prod(sh["dw"])), "normal", 0.0, 1.0).reshape(sh["dw"])
    y = oracle.conv_fwd(p, x, w)
    np.testing.assert_allclose(y, torch_fwd(p, x, w), rtol=1e-11, atol=1e-11)
    dw, _ = oracle.wgrad(p, x, dy)
    lhs = float(np.sum(dw * w))
    rhs = float(np.sum(dy * y))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, np.sum(np.abs(dw * w)))


def test_one_by_one_is_matmul():
    p = _prob(2, 3, 2, 5, 4, [4, 6], [1, 1])
    x, dy = _rand(p, 41)
    dw, _ = oracle.wgrad(p, x, dy)
    P = 2 * 4 * 6
    xm, dym = x.reshape(P, 3, 5), dy.reshape(P, 3, 4)
    for g in range(3):
        np.testing.assert_allclose(dw[g].reshape(4, 5), dym[:, g, :].T @ xm[:, g, :], rtol=1e-13, atol=1e-13)


def test_depthwise_equals_per_channel_dense():
    G = 6
    p = _prob(2, G, 2, 1, 1, [7, 6], [3, 3], [1, 2], [1, 1], [1, 1], [1, 0])
    x, dy = _rand(p, 51)
    dw, _ = oracle.wgrad(p, x, dy)
    for g in range(G):
        q = dict(p, G=1)
        d1, _ = oracle.wgrad(q, np.ascontiguousarray(x[..., g:g + 1, :]), np.ascontiguousarray(dy[..., g:g + 1, :]))
        np.testing.assert_array_equal(dw[g:g + 1], d1)


def test_full_image_filter_closed_form():
    p = _prob(2, 2, 3, 3, 2, [4, 5], [4, 5])
    x, dy = _rand(p, 61)
    assert oracle.out_dims(p) == [1, 1]
    dw, _ = oracle.wgrad(p, x, dy)
    ref = np.einsum("ngk,nyxgc->gkyxc", dy.reshape(3, 2, 2), x)
    np.testing.assert_allclose(dw, ref, rtol=1e-13, atol=1e-13)


def test_linearity_and_abs_sum():
    p = SMALL[4]
    x, dy = _rand(p, 71)
    dw, ab = oracle.wgrad(p, x, dy)
    dw3, ab3 = oracle.wgrad(p, x, -3.0 * dy)
    np.testing.assert_allclose(dw3, -3.0 * dw, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(ab3, 3.0 * ab, rtol=1e-13, atol=1e-13)
    dwa, _ = oracle.wgrad(p, np.abs(x), np.abs(dy))
    np.testing.assert_allclose(ab, dwa, rtol=1e-13, atol=1e-13)


def test_sampled_matches_full():
    p = SMALL[3]
    x, dy = _rand(p, 81)
    dw, ab = oracle.wgrad(p, x, dy)
    idx = np.array([0, 5, dw.size // 2, dw.size - 1], dtype=np.int64)
    s, a = oracle.wgrad_at(p, x, dy, idx)
    np.testing.assert_array_equal(s, dw.ravel()[idx])
    np.testing.assert_array_equal(a, ab.ravel()[idx])


def test_integer_inputs_exact():
    p = _prob(2, 2, 2, 3, 2, [6, 6], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1])
    sh = oracle.shapes(p)
    x = synth.values(5, int(np.prod(sh["x"])), "int", -2, 2).reshape(sh["x"])
    dy = synth.values(6, int(np.prod(sh["dy"])), "int", -2, 2).reshape(sh["dy"])
    dw, _ = oracle.wgrad(p, x, dy)
    ref = im2col_wgrad(p, x.astype(np.int64), dy.astype(np.int64))
    np.testing.assert_array_equal(dw, ref)


def test_output_size_rule():
    # Standard rule: floor((in + pl + pr - d(f-1) - 1)/s) + 1, checked against torch's output shape.
    torch = pytest.importorskip("torch")
    for inn, f, s, d, pl, pr in [(8, 3, 1, 1, 1, 1), (56, 3, 1, 1, 1, 1), (16, 3, 2, 1, 1, 1), (13, 3, 2, 1, 1, 1),
                                 (7, 2, 3, 2, 0, 2), (5, 5, 1, 1, 0, 0)]:
        p = _prob(1, 1, 1, 1, 1, [inn], [f], [s], [d], [pl], [pr])
        xt = torch.nn.functional.pad(torch.zeros(1, 1, inn), [pl, pr])
        yt = torch.nn.functional.conv1d(xt, torch.zeros(1, 1, f), stride=s, dilation=d)
        assert oracle.out_dims(p) == [yt.shape[-1]]


def test_decode_exact():
    w = np.arange(0, 65536, dtype=np.uint16)
    bf = oracle.decode(w, "bf16")
    ref = synth.bits_to_f32(w, "bf16").astype(np.float64)
    np.testing.assert_array_equal(np.isnan(bf), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(bf[ok], ref[ok])
    hf = oracle.decode(w, "fp16")
    ref = w.view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(np.isnan(hf), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(hf[ok], ref[ok])


# ----------------------------------------------------------------- backward-data
def _rand_w(p, seed):
    sh = oracle.shapes(p)
    return synth.values(seed, int(np.prod(sh["dw"])), "uniform").reshape(sh["dw"])


def torch_dgrad(p, dy, w):
    """PyTorch's fp64 CPU autograd input gradient of the padded grouped convolution."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    nd, G, N, C, K = p["ndim"], p["G"], p["N"], p["C"], p["K"]
    x0 = torch.zeros(N, G * C, *p["in"], dtype=torch.float64, requires_grad=True)
    pad = []
    for i in reversed(range(nd)):
        pad += [p["pad_l"][i], p["pad_r"][i]]
    wt = torch.from_numpy(np.ascontiguousarray(np.moveaxis(w, -1, 2))).reshape(G * K, C, *p["filt"])
    conv = {1: F.conv1d, 2: F.conv2d, 3: F.conv3d}[nd]
    yt = conv(F.pad(x0, pad), wt, stride=p["stride"], dilation=p["dil"], groups=G)
    out = oracle.out_dims(p)
    perm_in = (0, nd + 1, nd + 2) + tuple(range(1, nd + 1))
    dyt = torch.from_numpy(np.ascontiguousarray(dy)).permute(*perm_in).reshape(N, G * K, *out)
    yt.backward(dyt)
    g = x0.grad.reshape(N, G, C, *p["in"]).numpy()
    return np.moveaxis(np.moveaxis(g, 1, -1), 1, -1)  # (N, *in, G, C)


def scatter_dgrad(p, dy, w):
    """Pure-Python scatter form: every (output position, tap) adds dY * W to the
    input position it reads."""
    nd, G, N, C, K = p["ndim"], p["G"], p["N"], p["C"], p["K"]
    out = oracle.out_dims(p)
    dx = np.zeros((N, *p["in"], G, C))
    for n in range(N):
        for o in itertools.product(*[range(v) for v in out]):
            for t in itertools.product(*[range(f) for f in p["filt"]]):
                i = tuple(o[j] * p["stride"][j] - p["pad_l"][j] + t[j] * p["dil"][j] for j in range(nd))
                if any(i[j] < 0 or i[j] >= p["in"][j] for j in range(nd)):
                    continue
                for g in range(G):
                    dx[(n, *i, g)] += dy[(n, *o, g)] @ w[(g, slice(None), *t)]
    return dx


@pytest.mark.parametrize("p", SMALL, ids=lambda p: f"{p['ndim']}d_G{p['G']}")
def test_dgrad_matches_torch_autograd(p):
    _, dy = _rand(p, 61)
    w = _rand_w(p, 63)
    dx, _ = oracle.dgrad(p, dy, w)
    np.testing.assert_allclose(dx, torch_dgrad(p, dy, w), rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("p", SMALL[:5], ids=lambda p: f"{p['ndim']}d_G{p['G']}")
def test_dgrad_matches_scatter(p):
    _, dy = _rand(p, 71)
    w = _rand_w(p, 73)
    dx, _ = oracle.dgrad(p, dy, w)
    np.testing.assert_allclose(dx, scatter_dgrad(p, dy, w), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("p", SMALL, ids=lambda p: f"{p['ndim']}d_G{p['G']}")
def test_dgrad_adjoint_of_forward(p):
    # <dgrad(dY, W), X'> = <dY, conv_fwd(X', W)> for any X'; conv_fwd is pinned to PyTorch above.
    xp, dy = _rand(p, 81)
    w = _rand_w(p, 83)
    dx, _ = oracle.dgrad(p, dy, w)
    lhs = float(np.sum(dx * xp))
    rhs = float(np.sum(dy * oracle.conv_fwd(p, xp, w)))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(rhs))


def test_dgrad_one_by_one_is_matmul():
    p = _prob(2, 3, 2, 5, 4, [3, 4], [1, 1])
    _, dy = _rand(p, 91)
    w = _rand_w(p, 93)
    dx, _ = oracle.dgrad(p, dy, w)
    for g in range(3):
        ref = dy[..., g, :].reshape(-1, 4) @ w[g].reshape(4, 5)
        np.testing.assert_allclose(dx[..., g, :].reshape(-1, 5), ref, rtol=1e-13, atol=1e-13)


def test_dgrad_abs_sum():
    p = SMALL[3]
    _, dy = _rand(p, 95)
    w = _rand_w(p, 97)
    dx, a = oracle.dgrad(p, dy, w)
    a2, _ = oracle.dgrad(p, np.abs(dy), np.abs(w))
    np.testing.assert_allclose(a, a2, rtol=1e-13, atol=1e-13)
    assert np.all(a + 1e-15 >= np.abs(dx))
