"""GPU runtime behaviour: bounded waits that run out, CUDA-graph capture.

The wait tests make a kernel wait for something that never comes (the
forward's TMA producers are told to stop early; a fused-schedule backward
launch whose dX tile depends on a dZ tile that is not scheduled) and check
that the wait gives up after its limit with FLP_ERR_TIMEOUT in the error
word, that the kernel returns on its own, and that the CUDA context keeps
working afterwards.  Nothing faults, traps or hangs the GPU.
"""
import math
import time

import numpy as np
import pytest
import torch

import oracle
from entropy_loss_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def flp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from entropy_loss_gb300 import build, flp as _flp
    build.build()
    _flp.load()
    return _flp


def test_bounded_wait_times_out_and_context_survives(flp):
    limit_ns = 200_000_000  # 0.2 s per wait
    ws = torch.empty(flp.SELFTEST_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")

    def outputs():
        o = flp.SELFTEST_OUTPUT_OFFSET
        return ws[o:o + 3 * 256 * 4].view(torch.float32).view(3, 256).cpu().double()

    assert flp.selftest_wait_timeout(-1, limit_ns, workspace=ws) == flp.FLP_OK  # no stall
    # all-zero logits over 512 classes: lse = entropy = log 512, logprob = -log 512
    lp, lse, ent = outputs()
    assert torch.allclose(lse, torch.full_like(lse, math.log(512)), atol=1e-5)
    assert torch.allclose(ent, torch.full_like(ent, math.log(512)), atol=1e-5)
    assert torch.allclose(lp, torch.full_like(lp, -math.log(512)), atol=1e-5)
    t0 = time.perf_counter()
    st = flp.selftest_wait_timeout(1, limit_ns, workspace=ws)
    elapsed = time.perf_counter() - t0
    assert st == flp.FLP_ERR_TIMEOUT
    assert elapsed < 5.0, f"timed-out kernel took {elapsed:.2f} s to return"
    # the merge saw the timeout bit: no row reports a stale or partial value
    assert torch.isnan(outputs()).all()
    assert flp.selftest_wait_timeout(0, limit_ns, workspace=ws) == flp.FLP_ERR_TIMEOUT  # before any data
    assert torch.isnan(outputs()).all()
    # the context still runs the real path correctly
    d = inputs.make_inputs(inputs.custom("after", 200, 64, 1000, w_std=0.05, seed=41))
    dev = torch.device("cuda")
    lp, lse, en = flp.forward(d["X"].to(dev), d["W"].to(dev), d["y"].to(dev))
    o_lp, o_lse, o_en = oracle.forward(inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"]),
                                       d["y"].numpy())
    assert np.abs(lp.cpu().double().numpy() - o_lp).max() < 2e-3
    assert np.abs(en.cpu().double().numpy() - o_en).max() < 2e-3


def test_dz_kernel_wait_times_out_and_context_survives(flp):
    """The split schedule's dZ kernel (256 x 512 tiles, two epilogue groups
    with store barriers) stalls, gives up after the bounded wait, reports the
    timeout, and leaves a context that still runs a correct split backward."""
    limit_ns = 200_000_000
    assert flp.selftest_dz_wait_timeout(-1, limit_ns) == flp.FLP_OK  # same launch, no stall
    for stall in (1, 0, 3):  # after the first stage, before any data, before the last of 4 stages
        t0 = time.perf_counter()
        st = flp.selftest_dz_wait_timeout(stall, limit_ns)
        elapsed = time.perf_counter() - t0
        assert st == flp.FLP_ERR_TIMEOUT, stall
        assert elapsed < 5.0, f"timed-out kernel took {elapsed:.2f} s to return"
    assert flp.selftest_dz_wait_timeout(-1, limit_ns) == flp.FLP_OK
    M, H, V = 300, 64, 1000
    d = inputs.make_inputs(inputs.custom("after_dz", M, H, V, w_std=0.05, seed=44))
    dev = torch.device("cuda")
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    ws = flp.alloc_workspace(M, H, V, True, device=dev)
    lp, lse, en = flp.forward(X, W, y, workspace=ws)
    dX, dW = flp.backward(X, W, y, lse, en, d["g_lp"].to(dev), d["g_ent"].to(dev), workspace=ws,
                          schedule="split")
    torch.cuda.synchronize()
    assert flp.get_error(ws) == flp.FLP_OK
    o_dx, o_dw = oracle.backward(inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"]), d["y"].numpy(),
                                 d["g_lp"].double().numpy(), d["g_ent"].double().numpy())
    for got, want in ((dX, o_dx), (dW, o_dw)):
        g = got.float().cpu().double().numpy()
        assert np.linalg.norm(g - want) / np.linalg.norm(want) < 1e-2


def test_fused_dependency_wait_times_out_and_context_survives(flp):
    limit_ns = 200_000_000
    assert flp.selftest_dependency_timeout(False, limit_ns) == flp.FLP_OK  # full schedule
    t0 = time.perf_counter()
    st = flp.selftest_dependency_timeout(True, limit_ns)
    elapsed = time.perf_counter() - t0
    assert st == flp.FLP_ERR_TIMEOUT
    assert elapsed < 5.0, f"timed-out kernel took {elapsed:.2f} s to return"
    assert flp.selftest_dependency_timeout(False, limit_ns) == flp.FLP_OK
    # the context still runs the real fused backward correctly
    M, H, V = 300, 64, 1000
    d = inputs.make_inputs(inputs.custom("after_dep", M, H, V, w_std=0.05, seed=43))
    dev = torch.device("cuda")
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    ws = flp.alloc_workspace(M, H, V, True, chunk_rows=256, device=dev)
    lp, lse, en = flp.forward(X, W, y, workspace=ws)
    dX, dW = flp.backward(X, W, y, lse, en, d["g_lp"].to(dev), d["g_ent"].to(dev), workspace=ws,
                          schedule="fused")
    torch.cuda.synchronize()
    assert flp.get_error(ws) == flp.FLP_OK
    o_dx, o_dw = oracle.backward(inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"]), d["y"].numpy(),
                                 d["g_lp"].double().numpy(), d["g_ent"].double().numpy())
    for got, want in ((dX, o_dx), (dW, o_dw)):
        g = got.float().cpu().double().numpy()
        assert np.linalg.norm(g - want) / np.linalg.norm(want) < 1e-2


@pytest.mark.parametrize("schedule", ["split", "fused", "vsplit"])
def test_cuda_graph_capture_and_replay(flp, schedule):
    dev = torch.device("cuda")
    d = inputs.make_inputs(inputs.custom("graph", 700, 136, 2100, w_std=0.05, ignore_frac=0.1,
                                         seed=42))
    M, H, V = 700, 136, 2100
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    g1, g2 = d["g_lp"].to(dev), d["g_ent"].to(dev)
    ws = flp.alloc_workspace(M, H, V, True, chunk_rows=256, device=dev)
    lp = torch.empty(M, device=dev)
    lse = torch.empty(M, device=dev)
    en = torch.empty(M, device=dev)
    dX = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(V, H, device=dev)

    def step():
        flp.forward(X, W, y, logprob=lp, lse=lse, entropy=en, workspace=ws)
        flp.backward(X, W, y, lse, en, g1, g2, dX=dX, dW=dW, workspace=ws, schedule=schedule)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (lp, lse, en, dX, dW)]
    for t in (lp, lse, en, dX, dW):
        t.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up on the side stream before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (lp, lse, en, dX, dW):
        t.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (lp, lse, en, dX, dW)):
        assert torch.equal(a, b)
    assert flp.get_error(ws) == flp.FLP_OK


@pytest.mark.parametrize("schedule", ["split", "fused", "vsplit"])
def test_repeated_backward_is_bit_stable(flp, schedule):
    """60 back-to-back full-size backward launches (headline shape) per
    schedule, every tenth checked bit for bit against the first: a race in the
    tile hand-off, the fused schedule's counters or the dW / dX adds would
    show as a changed bit or a timeout in the error word."""
    dev = torch.device("cuda")
    w = inputs.WORKLOADS["m4096_h4096_v131072"]
    d = inputs.make_inputs(w)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    g1, g2 = d["g_lp"].to(dev), d["g_ent"].to(dev)
    ws = flp.alloc_workspace(w.M, w.H, w.V, True, chunk_rows=1024 if schedule == "vsplit" else 0,
                             device=dev)
    fwd_ws = flp.alloc_workspace(w.M, w.H, w.V, True, device=dev)
    _, lse, en = flp.forward(X, W, y, workspace=fwd_ws)
    dX0, dW0 = flp.backward(X, W, y, lse, en, g1, g2, workspace=ws, schedule=schedule)
    dX0, dW0 = dX0.clone(), dW0.clone()
    dX, dW = torch.empty_like(dX0), torch.empty_like(dW0)
    for i in range(60):
        flp.backward(X, W, y, lse, en, g1, g2, dX=dX, dW=dW, workspace=ws, schedule=schedule)
        if i % 10 == 9:
            torch.cuda.synchronize()
            assert flp.get_error(ws) == flp.FLP_OK
            assert torch.equal(dX, dX0) and torch.equal(dW, dW0), f"launch {i} differs"
