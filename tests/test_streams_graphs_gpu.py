"""GPU tests of the entry points under CUDA graph capture, on several streams at
once, and from several host threads.

* Graphs: a deterministic weight-gradient call (split-K kernel plus the
  reduction kernel it launches with programmatic dependent launch), an atomic
  one (the kernel that zeroes dW, then the split-K kernel launched as its
  programmatic dependent), an atomic depthwise one, a backward-data call and a
  host-buffer call are captured
  once and replayed with new input values copied into the same buffers; each
  replay must give the bits of an eager call on those values.
* Streams: four different problems launched on four streams without
  synchronising in between must each give the bits of a run alone.
* Threads: four host threads calling concurrently (the library caches plans
  and tensor maps under a lock) must give the same bits.
* Launch chain: a backward-data kernel writes the X of a weight-gradient call
  queued right behind it; the call's first kernel must wait for it.
"""
import threading

import numpy as np
import pytest

from implicit_gemm_gb300 import binding, build
from tests.common import make_inputs, spec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

_TDT = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    build.build()
    binding.load()


def _inputs(sp, seed):
    x, dy = make_inputs(sp, ("uniform", -1.0, 1.0), seed, seed + 1)
    idt = torch.bfloat16 if sp["in_dtype"] == "bf16" else torch.float16
    xt = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(idt)
    dyt = torch.from_numpy(np.ascontiguousarray(dy).view(np.int16)).view(idt)
    return xt, dyt


def _ndw(sp):
    return sp["G"] * sp["K"] * int(np.prod(sp["filt"])) * sp["C"]


def _bits(t):
    t = t.detach().cpu()
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16).numpy().copy()


class Call:
    """Device buffers and a workspace for one problem and plan."""

    def __init__(self, sp, split_k=0, mode="auto"):
        self.sp, self.split_k, self.mode = sp, split_k, mode
        xt, dyt = _inputs(sp, 900)
        self.x, self.dy = xt.cuda(), dyt.cuda()
        odt = torch.float32 if mode == "atomic" else _TDT[sp["out_dtype"]]
        self.dw = torch.empty(_ndw(sp), dtype=odt, device="cuda")
        self.nb = binding.wg_workspace_size(sp, split_k, mode, 0)
        self.ws = torch.empty(max(self.nb, 16), dtype=torch.uint8, device="cuda")

    def __call__(self, stream=None):
        binding.wg_conv_bwd_weight(self.sp, self.x, self.dy, self.dw, self.split_k, self.mode, 0, self.ws, self.nb,
                                   stream=stream)

    def load(self, seed):
        xt, dyt = _inputs(self.sp, seed)
        self.x.copy_(xt)
        self.dy.copy_(dyt)


DENSE = spec(2, 1, 8, 64, 64, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "bf16")


DEPTHWISE = spec(2, 256, 32, 1, 1, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32")


@pytest.mark.parametrize("sp,split_k,mode", [(DENSE, 0, "deterministic"), (DENSE, 0, "auto"),
                                             (dict(DENSE, out_dtype="fp32"), 24, "atomic"),
                                             (DEPTHWISE, 0, "atomic")],
                         ids=["dense_deterministic", "dense_auto", "dense_atomic", "depthwise_atomic"])
def test_graph_replay_matches_eager(sp, split_k, mode):
    c = Call(sp, split_k, mode)
    atomic = "mode=atomic" in binding.wg_plan_string(sp, split_k, mode, 0)
    s = torch.cuda.Stream()
    eager, eager_f = {}, {}
    for seed in (910, 920, 930):
        c.load(seed)
        c()
        torch.cuda.synchronize()
        eager[seed] = _bits(c.dw)
        eager_f[seed] = c.dw.float().cpu().numpy()
    with torch.cuda.stream(s):
        c(s)  # first call outside the capture: plan, tensor maps, kernel attributes
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c(s)
    for seed in (910, 920, 930):
        c.load(seed)
        torch.cuda.synchronize()
        c.dw.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        got = _bits(c.dw)
        if atomic:
            # Atomic adds land in another order on every run: a few fp32 ulps of
            # the partial sums, which can be far larger than a cancelled result
            # (and one unit of a 16-bit dW where the cast rounds the other way).
            e = eager_f[seed]
            ulp = 0.0 if c.dw.dtype == torch.float32 else float(np.max(np.abs(e))) * 2.0 ** -7
            np.testing.assert_allclose(c.dw.float().cpu().numpy(), e, rtol=0,
                                       atol=1e-5 * float(np.max(np.abs(e))) + ulp)
        else:
            np.testing.assert_array_equal(got, eager[seed])
    binding.wg_check_status()


def test_graph_replay_dgrad_and_host_entry():
    sp = spec(2, 1, 4, 64, 64, [20, 20], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32")
    # backward-data
    dyt = torch.randn(sp["N"], 20, 20, 64, dtype=torch.float32).to(torch.bfloat16).cuda()
    w = torch.randn(_ndw(sp), dtype=torch.float32).to(torch.bfloat16).cuda()
    dx = torch.empty(sp["N"] * 20 * 20 * 64, dtype=torch.float32, device="cuda")
    binding.wg_conv_bwd_data(sp, dyt, w, dx)
    torch.cuda.synchronize()
    ref = _bits(dx)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        binding.wg_conv_bwd_data(sp, dyt, w, dx, stream=s)
    dx.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(dx), ref)
    # host entry: copies become memcpy nodes of the graph
    xt, dyh = _inputs(sp, 940)
    xh, dyh = xt.pin_memory(), dyh.pin_memory()
    dwh = torch.empty(_ndw(sp), dtype=torch.float32).pin_memory()
    xd, dyd = torch.empty_like(xh, device="cuda"), torch.empty_like(dyh, device="cuda")
    dwd = torch.empty(_ndw(sp), dtype=torch.float32, device="cuda")
    nb = binding.wg_workspace_size(sp, 0, "deterministic")
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    binding.wg_conv_bwd_weight_host(sp, xh, dyh, dwh, xd, dyd, dwd, mode="deterministic", workspace=ws, ws_bytes=nb)
    torch.cuda.synchronize()
    ref = dwh.clone()
    with torch.cuda.graph(g2 := torch.cuda.CUDAGraph(), stream=s):
        binding.wg_conv_bwd_weight_host(sp, xh, dyh, dwh, xd, dyd, dwd, mode="deterministic", workspace=ws,
                                        ws_bytes=nb, stream=s)
    dwh.fill_(float("nan"))
    xd.zero_()
    g2.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(dwh), _bits(ref))
    binding.wg_check_status()


PROBLEMS = [
    (DENSE, 0, "deterministic"),
    (spec(2, 512, 4, 1, 1, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32"), 0, "deterministic"),
    (spec(3, 1, 2, 32, 48, [8, 8, 8], [3, 3, 3], [2, 2, 2], [1, 1, 1], [1, 1, 1], [1, 1, 1], "fp16", "fp32"), 8,
     "deterministic"),
    (spec(2, 8, 4, 8, 16, [14, 14], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "bf16"), 0, "deterministic"),
]


def _alone():
    out = []
    for sp, k, mode in PROBLEMS:
        c = Call(sp, k, mode)
        c()
        torch.cuda.synchronize()
        out.append(_bits(c.dw))
    return out


def test_concurrent_streams_match_alone():
    ref = _alone()
    calls = [Call(sp, k, mode) for sp, k, mode in PROBLEMS]
    streams = [torch.cuda.Stream() for _ in calls]
    for rep in range(3):
        for c in calls:
            c.dw.fill_(float("nan"))
        torch.cuda.synchronize()
        for c, st in zip(calls, streams):
            c(st)
        torch.cuda.synchronize()
        for i, c in enumerate(calls):
            np.testing.assert_array_equal(_bits(c.dw), ref[i], err_msg=f"problem {i} rep {rep}")
    binding.wg_check_status()


def test_concurrent_host_threads_match_alone():
    ref = _alone()
    errors = []

    def worker(i):
        try:
            sp, k, mode = PROBLEMS[i]
            c = Call(sp, k, mode)
            st = torch.cuda.Stream()
            for _ in range(5):
                c(st)
            st.synchronize()
            np.testing.assert_array_equal(_bits(c.dw), ref[i], err_msg=f"thread {i}")
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(PROBLEMS))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    binding.wg_check_status()


# Every kernel of a call is launched as a programmatic dependent of the kernel
# before it and waits for it before reading X and dY.  Here the kernel before
# it is the library's own backward-data kernel, which lets its dependents
# launch at once and writes the X that the weight-gradient call reads: a call
# that read X before that kernel finished would see stale or partial values.
# Each mode's first kernel is covered: the split-K kernel (two-stage), the
# zeroing kernel (atomic, into dW or into the fp32 copy of a 16-bit dW), the
# depthwise kernel (depthwise, two-stage and atomic).
CHAIN = [
    ("two_stage", spec(2, 1, 8, 64, 64, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "bf16"),
     "deterministic"),
    ("atomic", spec(2, 1, 8, 64, 64, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32"), "atomic"),
    ("atomic_bf16_dw", spec(2, 1, 8, 64, 64, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "bf16"),
     "atomic"),
    ("depthwise_atomic", spec(2, 64, 8, 1, 1, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32"),
     "atomic"),
    ("depthwise_two_stage", spec(2, 64, 8, 1, 1, [28, 28], [3, 3], [1, 1], [1, 1], [1, 1], [1, 1], "bf16", "fp32"),
     "deterministic"),
]


@pytest.mark.parametrize("name,sp,mode", CHAIN, ids=[c[0] for c in CHAIN])
def test_call_waits_for_the_kernel_that_writes_its_input(name, sp, mode):
    torch.manual_seed(7)
    # Backward-data on the same geometry writes X (bf16) from dY1 and W.
    spd = dict(sp, out_dtype="bf16")
    n_x = sp["N"] * int(np.prod(sp["in"])) * sp["G"] * sp["C"]
    n_dy = sp["N"] * int(np.prod(sp["in"])) * sp["G"] * sp["K"]  # stride 1, same padding: out = in
    dy1 = [torch.randn(n_dy, device="cuda").to(torch.bfloat16) for _ in range(3)]
    w = torch.randn(_ndw(sp), device="cuda").to(torch.bfloat16)
    dy2 = torch.randn(n_dy, device="cuda").to(torch.bfloat16)
    x = torch.empty(n_x, dtype=torch.bfloat16, device="cuda")
    odt = torch.float32 if sp["out_dtype"] == "fp32" else torch.bfloat16
    nb_d = binding.wg_bwd_data_workspace_size(spd)
    ws_d = torch.empty(max(nb_d, 16), dtype=torch.uint8, device="cuda")
    nb = binding.wg_workspace_size(sp, 0, mode, 0)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    chained = []
    with torch.cuda.stream(s):
        for d in dy1:  # no synchronisation inside the chain
            binding.wg_conv_bwd_data(spd, d, w, x, ws_d, nb_d, stream=s)
            dw = torch.full((_ndw(sp),), float("nan"), dtype=odt, device="cuda")
            binding.wg_conv_bwd_weight(sp, x, dy2, dw, 0, mode, 0, ws, nb, stream=s)
            chained.append(dw)
    s.synchronize()
    binding.wg_check_status()
    for i, d in enumerate(dy1):
        # The same calls one at a time, with the device idle in between.
        binding.wg_conv_bwd_data(spd, d, w, x, ws_d, nb_d)
        torch.cuda.synchronize()
        ref = torch.empty((_ndw(sp),), dtype=odt, device="cuda")
        binding.wg_conv_bwd_weight(sp, x, dy2, ref, 0, mode, 0, ws, nb)
        torch.cuda.synchronize()
        got, want = chained[i].float().cpu().numpy(), ref.float().cpu().numpy()
        if mode == "deterministic":
            np.testing.assert_array_equal(got, want, err_msg=f"{name} call {i}")
        else:
            # adds in another order; with a 16-bit dW the cast may round one unit the other way
            m = float(np.max(np.abs(want)))
            np.testing.assert_allclose(got, want, rtol=0, atol=1e-4 * m + (m * 2.0 ** -7 if odt != torch.float32 else 0),
                                       err_msg=f"{name} call {i}")
    binding.wg_check_status()
