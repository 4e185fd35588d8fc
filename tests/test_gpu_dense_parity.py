"""The backward with every row's upstream gradient live, against the oracle.

The other full-size tests keep gradients on a few rows so that the oracle can
form dW from those rows alone; here every non-ignored row carries a gradient,
as in the bench's step, at the headline's hidden size and vocabulary
(H = 4096, V = 131072, K = 131072 for the dX contraction):

* M = 512: every element of dX and dW against the oracle's full fp64 backward,
  for each backward schedule (one wave, two row waves, the fused launch, the
  vocabulary split) and with an fp32 dX / bf16 dW;
* M = 777, V = 50257: ragged row and vocabulary tails, two row waves, every
  element;
* the headline M = 4096 itself: the forward on every row, dX on 256 sampled
  rows, and dW on 256 sampled vocabulary rows plus the tile and chunk
  boundary rows, each a sum over all 4096 rows.

Per tensor: relative L2 within 1e-2, cosine > 0.999 and norm ratio within 2%
(the tolerances of the other parity tests); per row of dX and of dW: relative
L2 within 1e-2 as well, so one broken tile cannot hide in a global norm.
Ignored rows of dX are exactly zero.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from entropy_loss_gb300 import inputs

pytestmark = pytest.mark.gpu

ATOL_FWD = 2e-3
RTOL_GRAD = 1e-2


@pytest.fixture(scope="module")
def flp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from entropy_loss_gb300 import build, flp as _flp
    build.build()
    _flp.load()
    return _flp


def check_fwd(got, want, name):
    g = got.detach().double().cpu().numpy()
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    err = np.abs(g - want)
    assert err.max() <= ATOL_FWD, f"{name}: max abs err {err.max():.3e} at {int(err.argmax())}"


def check_dense(got, want_t, name, zero_rows=None):
    """got: GPU tensor [R, H]; want_t: fp64 GPU tensor of the oracle's values."""
    g = got.detach().double()
    diff = g - want_t
    nw = torch.linalg.vector_norm(want_t)
    rel = float(torch.linalg.vector_norm(diff) / nw)
    cos = float((g * want_t).sum() / (torch.linalg.vector_norm(g) * nw))
    ratio = float(torch.linalg.vector_norm(g) / nw)
    assert torch.isfinite(g).all(), f"{name}: non-finite values"
    assert rel <= RTOL_GRAD, f"{name}: rel L2 {rel:.3e}"
    assert cos > 0.999, f"{name}: cosine {cos}"
    assert abs(ratio - 1) < 0.02, f"{name}: norm ratio {ratio}"
    rn = torch.linalg.vector_norm(want_t, dim=1)
    live = rn > 0
    row_rel = torch.linalg.vector_norm(diff, dim=1)[live] / rn[live]
    worst = float(row_rel.max()) if row_rel.numel() else 0.0
    assert worst <= RTOL_GRAD, (f"{name}: worst row rel L2 {worst:.3e} at row "
                                f"{int(torch.nonzero(live).flatten()[int(row_rel.argmax())])}")
    assert not g[~live].any(), f"{name}: rows whose gradient is zero are not exactly zero"
    if zero_rows is not None and len(zero_rows):
        assert not g[torch.as_tensor(zero_rows, device=g.device)].any(), f"{name}: ignored rows not zero"
    return rel, worst


def _device_inputs(d, dev):
    g2 = d["g_ent"].to(dev) if d["g_ent"] is not None else None
    return d["X"].to(dev), d["W"].to(dev), d["y"].to(dev), d["g_lp"].to(dev), g2


def _run_backward(flp, X, W, y, lse, en, g1, g2, d, ws, schedule, dx_dtype=torch.bfloat16,
                  dw_dtype=torch.float32):
    dX, dW = flp.backward(X, W, y, lse, en, g1, g2, ignore_index=d["ignore_index"], scale=d["scale"],
                          compute_entropy=d["compute_entropy"], dx_dtype=dx_dtype, dw_dtype=dw_dtype,
                          workspace=ws, schedule=schedule)
    torch.cuda.synchronize()
    assert flp.get_error(ws) == flp.FLP_OK
    return dX, dW


def _full_dense(flp, w, variants):
    """Every element of dX and dW, every row's gradient live, against the
    oracle's full backward; `variants` lists (label, chunk_rows, schedule,
    dX dtype, dW dtype)."""
    dev = torch.device("cuda")
    d = inputs.make_inputs(w)
    X, W, y, g1, g2 = _device_inputs(d, dev)
    ent = d["compute_entropy"]
    Xb, Wb, yn = inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"]), d["y"].numpy()
    o_lp, o_lse, o_en = oracle.forward(Xb, Wb, yn, ignore_index=d["ignore_index"], scale=d["scale"],
                                       compute_entropy=ent)
    o_dx, o_dw = oracle.backward(Xb, Wb, yn, d["g_lp"].double().numpy(),
                                 d["g_ent"].double().numpy() if ent else None,
                                 ignore_index=d["ignore_index"], scale=d["scale"], compute_entropy=ent)
    want_dx = torch.from_numpy(o_dx).to(dev)
    del o_dx
    want_dw = torch.from_numpy(o_dw).to(dev)
    del o_dw
    ignored = np.flatnonzero(yn == d["ignore_index"])
    assert 0 < ignored.size < w.M
    report = {}
    for label, chunk_rows, schedule, dxt, dwt in variants:
        ws = flp.alloc_workspace(w.M, w.H, w.V, ent, chunk_rows=chunk_rows, device=dev)
        lp, lse, en = flp.forward(X, W, y, ignore_index=d["ignore_index"], scale=d["scale"],
                                  compute_entropy=ent, workspace=ws)
        torch.cuda.synchronize()
        check_fwd(lp, o_lp, f"{label} logprob")
        check_fwd(lse, o_lse, f"{label} lse")
        if ent:
            check_fwd(en, o_en, f"{label} entropy")
        plan = flp.backward_plan(w.M, w.H, w.V, ws.numel(), schedule)
        dX, dW = _run_backward(flp, X, W, y, lse, en, g1, g2, d, ws, schedule, dxt, dwt)
        report[label] = (plan, check_dense(dX, want_dx, f"{label} dX", zero_rows=ignored),
                         check_dense(dW, want_dw, f"{label} dW"))
        print(f"{w.name} {label}: plan {plan}; dX rel L2 {report[label][1][0]:.2e} (worst row "
              f"{report[label][1][1]:.2e}); dW rel L2 {report[label][2][0]:.2e} (worst row "
              f"{report[label][2][1]:.2e})")
        del dX, dW, ws
    return report


def test_dense_backward_every_element_m512_h4096_v131072(flp):
    """512 rows at the headline's H and V, every row live (5% ignored)."""
    w = inputs.custom("dense_m512_h4096_v131072", 512, 4096, 131072, ignore_frac=0.05, seed=1012)
    rep = _full_dense(flp, w, [
        ("split, one wave", 0, "split", torch.bfloat16, torch.float32),
        ("split, two 256-row waves", 256, "split", torch.bfloat16, torch.float32),
        ("fused", 0, "fused", torch.bfloat16, torch.float32),
        ("vocabulary split", 128, "vsplit", torch.bfloat16, torch.float32),
        ("split, fp32 dX, bf16 dW", 0, "split", torch.float32, torch.bfloat16),
    ])
    assert rep["split, two 256-row waves"][0][:2] == (256, 2)
    assert rep["vocabulary split"][0][2] == "vsplit" and rep["vocabulary split"][0][1] > 1


def test_dense_backward_every_element_ragged_m777_h4096_v50257(flp):
    """Ragged rows (3 pair tiles and 9 rows) and a ragged vocabulary (196
    tiles and 81 columns: the last wide dZ tile has a half past the end),
    two row waves of 512 and 265 rows, every row live."""
    w = inputs.custom("dense_m777_h4096_v50257", 777, 4096, 50257, ignore_frac=0.05, seed=1013)
    rep = _full_dense(flp, w, [
        ("split, two waves", 512, "split", torch.bfloat16, torch.float32),
        ("fused, two waves", 512, "fused", torch.bfloat16, torch.float32),
        ("auto", 0, "auto", torch.bfloat16, torch.float32),
    ])
    assert rep["split, two waves"][0][:2] == (512, 2)


def _sampled_dense(flp, w, schedules, n_rows=256, n_cols=256, seed=1014):
    """Every row live at the workload's full size: the forward on all rows,
    dX on a row sample (first, last and tile-boundary rows included), dW on a
    vocabulary sample plus the 256-column tile boundaries at both ends, every
    row-wave boundary's neighbourhood and every vocabulary-split chunk
    boundary, each dW row summed over all M rows; for each (label, chunk_rows,
    schedule)."""
    dev = torch.device("cuda")
    d = inputs.make_inputs(w)
    X, W, y, g1, g2 = _device_inputs(d, dev)
    ent = d["compute_entropy"]
    Xb, Wb, yn = inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"]), d["y"].numpy()
    M, H, V = w.M, w.H, w.V
    wss = {label: flp.alloc_workspace(M, H, V, ent, chunk_rows=cr, device=dev)
           for label, cr, _ in schedules}
    bounds = {0, V - 1}
    for label, _, sched in schedules:
        if flp.backward_plan(M, H, V, wss[label].numel(), sched)[2] != "vsplit":
            continue
        units = flp.backward_schedule(M, H, V, wss[label].numel(), "vsplit", 76)
        for li in range(0, int(units[:, 0].max()) + 1, 2):
            t = int(units[(units[:, 0] == li) & np.isin(units[:, 1], (0, 4)), 4].min())
            bounds |= {t * 256 - 1, t * 256, t * 256 + 255}
    for t in (1, (V - 1) // 256):
        bounds |= {t * 256 - 1, t * 256, t * 256 + 255}
    g = np.random.default_rng(seed)
    cols = np.unique(np.concatenate([g.choice(V, n_cols, replace=False),
                                     np.array(sorted(c for c in bounds if 0 <= c < V))]))
    rows = inputs.sample_rows(M, n_rows, seed=seed + 1).numpy()
    wave_edges = [r for k in range(8192, M, 8192) for r in (k - 1, k)]  # default row-wave boundaries
    rows = np.unique(np.concatenate([rows, np.array(wave_edges, dtype=rows.dtype)]))
    g_lp = d["g_lp"].double().numpy()
    g_ent = d["g_ent"].double().numpy() if ent else None
    o_dw, o_lp, o_lse, o_en = oracle.backward_dw_cols(
        Xb, Wb, yn, g_lp, g_ent, cols, ignore_index=d["ignore_index"], scale=d["scale"],
        compute_entropy=ent, with_forward=True)
    o_dx, _ = oracle.backward(Xb, Wb, yn, g_lp, g_ent, ignore_index=d["ignore_index"],
                              scale=d["scale"], compute_entropy=ent, rows=rows, want_dw=False)
    want_dw = torch.from_numpy(o_dw).to(dev)
    want_dx = torch.from_numpy(o_dx).to(dev)
    ridx = torch.as_tensor(rows, device=dev)
    cidx = torch.as_tensor(cols, device=dev)
    ignored = np.flatnonzero(yn[rows] == d["ignore_index"])
    first = schedules[0][0]
    lp, lse, en = flp.forward(X, W, y, ignore_index=d["ignore_index"], scale=d["scale"],
                              compute_entropy=ent, workspace=wss[first])
    torch.cuda.synchronize()
    assert flp.get_error(wss[first]) == flp.FLP_OK
    check_fwd(lp, o_lp, "logprob (all rows)")
    check_fwd(lse, o_lse, "lse (all rows)")
    if ent:
        check_fwd(en, o_en, "entropy (all rows)")
    for label, _, sched in schedules:
        plan = flp.backward_plan(M, H, V, wss[label].numel(), sched)
        dX, dW = _run_backward(flp, X, W, y, lse, en, g1, g2, d, wss[label], sched)
        rx = check_dense(dX[ridx], want_dx, f"{label} dX rows", zero_rows=ignored)
        rw = check_dense(dW[cidx], want_dw, f"{label} dW vocabulary rows")
        print(f"{w.name} {label}: plan {plan}; dX rows rel L2 {rx[0]:.2e} (worst {rx[1]:.2e}); dW "
              f"vocabulary rows rel L2 {rw[0]:.2e} (worst {rw[1]:.2e}); {len(rows)} rows, "
              f"{len(cols)} vocabulary rows")
        del dX, dW


def test_dense_backward_headline_sampled(flp):
    """The headline workload (M = 4096, H = 4096, V = 131072, every row live,
    5% ignored) in the bench's launch configuration, and with the fused and
    vocabulary-split schedules: the forward on all 4096 rows; dX on 256
    sampled rows (plus the first, last and tile-boundary rows); dW on 256
    sampled vocabulary rows plus every 256-column tile boundary row around
    the ends and the boundaries of the vocabulary-split chunks, each dW row a
    sum over all 4096 rows."""
    _sampled_dense(flp, inputs.WORKLOADS["m4096_h4096_v131072"],
                   [("split (the bench's)", 0, "auto"), ("fused", 0, "fused"),
                    ("vocabulary split", 1024, "vsplit")])


@pytest.mark.skipif(not os.environ.get("FLP_SLOW_PARITY"),
                    reason="the oracle's forward of every row takes 5-16 min here: set FLP_SLOW_PARITY=1")
@pytest.mark.parametrize("name", ["ragged_m20001_h4096_v128257", "m8192_h8192_v131072",
                                  "large_m32768_h5120_v152064"])
def test_dense_backward_large_workloads_sampled(flp, name):
    """The three largest workloads at full size in the bench's launch
    configuration (row waves of 8192: three for the ragged one, four for the
    large one; dW added across waves in fp32) with every row live: the
    forward on all rows, dX on ~256 rows, dW on ~270 vocabulary rows, each a
    sum over all rows (including the ragged vocabulary's tail tile)."""
    _sampled_dense(flp, inputs.WORKLOADS[name], [("split (the bench's)", 0, "auto")])


@pytest.mark.skipif(not os.environ.get("FLP_SLOW_PARITY"),
                    reason="the oracle's full backward at the headline shape takes ~6 min here: set FLP_SLOW_PARITY=1")
def test_dense_backward_every_element_headline(flp):
    """The headline workload exactly as the bench times it (M = 4096, H = 4096,
    V = 131072, every row live, one wave, the split schedule): every element
    of dX and dW against the oracle's full fp64 backward."""
    _full_dense(flp, inputs.WORKLOADS["m4096_h4096_v131072"],
                [("split (the bench's)", 0, "auto", torch.bfloat16, torch.float32)])
