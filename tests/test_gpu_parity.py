"""GPU path vs the fp64 oracle, through the C ABI (ctypes binding).

Tolerances (stated by the task's target for bf16 inputs with fp32
accumulation): logprob, lse and entropy within 2e-3 absolute; dX and dW within
1e-2 relative L2, plus gradient cosine > 0.999 and norm ratio within 2% (the
chunked GRPO page's gradient contract).
"""
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


def _np(t):
    return t.detach().float().cpu().double().numpy()


def check_fwd(got, want, name, atol=ATOL_FWD):
    g = _np(got)
    assert g.shape == want.shape
    err = np.abs(g - want)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    assert err.max() <= atol, f"{name}: max abs err {err.max():.3e} at {int(err.argmax())}"


def check_grad(got, want, name, rtol=RTOL_GRAD):
    g = _np(got)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    nw = np.linalg.norm(want)
    if nw == 0:
        assert np.linalg.norm(g) == 0, f"{name}: expected exact zero"
        return
    rel = np.linalg.norm(g - want) / nw
    cos = float(np.dot(g.ravel(), want.ravel()) / (np.linalg.norm(g) * nw))
    ratio = np.linalg.norm(g) / nw
    assert rel <= rtol, f"{name}: rel L2 {rel:.3e}"
    assert cos > 0.999, f"{name}: cosine {cos}"
    assert abs(ratio - 1) < 0.02, f"{name}: norm ratio {ratio}"


def run_case(flp, d, *, chunk_rows=0, dx_dtype=torch.bfloat16, check_backward=True, rows=None,
             dw_rows=None, schedule="auto"):
    dev = torch.device("cuda")
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    M, H = X.shape
    V = W.shape[0]
    ent = d["compute_entropy"]
    ws = flp.alloc_workspace(M, H, V, ent, chunk_rows=chunk_rows, device=dev)
    lp, lse, en = flp.forward(X, W, y, ignore_index=d["ignore_index"], scale=d["scale"],
                              compute_entropy=ent, workspace=ws)
    torch.cuda.synchronize()
    assert flp.get_error(ws) == flp.FLP_OK
    Xb, Wb = inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"])
    yn = d["y"].numpy()
    o_lp, o_lse, o_en = oracle.forward(Xb, Wb, yn, ignore_index=d["ignore_index"], scale=d["scale"],
                                       compute_entropy=ent, rows=rows)
    sel = slice(None) if rows is None else torch.as_tensor(rows)
    check_fwd(lp.cpu()[sel], o_lp, "logprob")
    check_fwd(lse.cpu()[sel], o_lse, "lse")
    if ent:
        check_fwd(en.cpu()[sel], o_en, "entropy")
    if not check_backward:
        return dict(lp=lp, lse=lse, en=en, ws=ws)
    g1 = d["g_lp"]
    g2 = d["g_ent"] if ent else None
    if dw_rows is not None:  # gradients only on a sample of rows: dW is then exact to compare
        mask = torch.zeros(M, dtype=torch.float32)
        mask[torch.as_tensor(dw_rows)] = 1
        g1 = g1 * mask
        g2 = None if g2 is None else g2 * mask
    dX, dW = flp.backward(X, W, y, lse, en, g1.to(dev), None if g2 is None else g2.to(dev),
                          ignore_index=d["ignore_index"], scale=d["scale"], compute_entropy=ent,
                          dx_dtype=dx_dtype, workspace=ws, schedule=schedule)
    torch.cuda.synchronize()
    assert flp.get_error(ws) == flp.FLP_OK
    g1n = g1.double().numpy()
    g2n = None if g2 is None else g2.double().numpy()
    if dw_rows is None and rows is None:
        o_dx, o_dw = oracle.backward(Xb, Wb, yn, g1n, g2n, ignore_index=d["ignore_index"],
                                     scale=d["scale"], compute_entropy=ent)
        check_grad(dX, o_dx, "dX")
        check_grad(dW, o_dw, "dW")
    else:
        if rows is not None:
            o_dx, _ = oracle.backward(Xb, Wb, yn, g1n, g2n, ignore_index=d["ignore_index"],
                                      scale=d["scale"], compute_entropy=ent, rows=rows,
                                      want_dw=False)
            if dw_rows is not None:
                keep = np.isin(rows, dw_rows)
                check_grad(dX.cpu()[torch.as_tensor(rows[keep])], o_dx[keep], "dX rows")
                assert np.all(_np(dX.cpu()[torch.as_tensor(rows[~keep])]) == 0)
            else:
                check_grad(dX.cpu()[torch.as_tensor(rows)], o_dx, "dX rows")
        if dw_rows is not None:
            _, o_dw = oracle.backward(Xb, Wb, yn, g1n, g2n, ignore_index=d["ignore_index"],
                                      scale=d["scale"], compute_entropy=ent, rows=dw_rows,
                                      want_dx=False)
            check_grad(dW, o_dw, "dW")
    return dict(lp=lp, lse=lse, en=en, dX=dX, dW=dW, ws=ws)


def case(M, H, V, seed=11, **kw):
    kw.setdefault("w_std", 0.05)
    kw.setdefault("ignore_frac", 0.1)
    return inputs.make_inputs(inputs.custom(f"m{M}_h{H}_v{V}", M, H, V, seed=seed, **kw))


# ----------------------------------------------------------------- small shapes

def test_tiny_workload(flp):
    run_case(flp, inputs.make_inputs(inputs.WORKLOADS["tiny"]))


@pytest.mark.parametrize("M,H,V", [
    (1, 64, 1), (1, 8, 2), (127, 64, 255), (128, 64, 256), (129, 72, 257),
    (300, 200, 3001), (5, 8, 50257 // 16), (513, 264, 1000),
    # around the 256-row pair tiles and 256-column vocabulary tiles, H < 64
    (255, 56, 511), (256, 128, 512), (257, 136, 513), (511, 64, 767), (512, 64, 1024),
])
def test_edge_shapes(flp, M, H, V):
    run_case(flp, case(M, H, V))


@pytest.mark.parametrize("ent", [True, False])
@pytest.mark.parametrize("scale", [0.5, 1.0, 1.0 / 0.7])
def test_scale_and_entropy_flag(flp, ent, scale):
    run_case(flp, case(200, 128, 1500, seed=3, scale=scale, compute_entropy=ent))


@pytest.mark.parametrize("schedule", ["split", "auto"])
def test_waves_and_ragged_tail(flp, schedule):
    # 700 rows in 256-row waves: three waves, the last one ragged; dW accumulates
    # across waves in fp32.  (auto takes the vocabulary split for such short waves.)
    run_case(flp, case(700, 136, 2100, seed=4), chunk_rows=256, schedule=schedule)


@pytest.mark.parametrize("schedule", ["split", "fused"])
@pytest.mark.parametrize("M,H,V,chunk", [
    (700, 136, 2100, 256),   # three 256-row waves, the last ragged
    (5000, 64, 1000, 512),   # ten waves
    (1200, 264, 3001, 0),    # one wave
    (257, 136, 513, 256),    # two waves, the second a single row
    (2600, 72, 5000, 1024),  # fused: dZ tiles of a wave wait on the previous wave's dX / dW tiles
    (1300, 512, 16500, 512), # wide (256 x 512) dX tiles in three waves
    (900, 640, 3001, 512),   # three 256-column tiles of H (the last half-filled): 256 x 256 dX and
                             # dW tiles, several per row tile, alternating accumulators, two waves
])
def test_schedules_match_oracle(flp, schedule, M, H, V, chunk):
    run_case(flp, case(M, H, V, seed=22), chunk_rows=chunk, schedule=schedule)


@pytest.mark.parametrize("M,H,V,chunk,ent,dx_f32,dw_bf16,acc", [
    (700, 136, 2100, 256, True, False, False, False),
    (700, 136, 2100, 256, False, True, False, True),
    (1200, 264, 3001, 0, True, False, True, False),
    (2600, 72, 5000, 1024, True, True, False, False),
    (4096, 512, 16384, 0, True, False, False, False),
    (16384, 64, 1000, 256, True, False, False, True),  # 64 waves: the fused schedule spans two launches
    (1300, 512, 16500, 512, True, True, False, True),   # wide dX tiles, three waves, slot layouts switching
    (1200, 264, 16500, 0, True, False, False, False),   # wide dX tiles whose second half is mostly beyond H
    (1000, 1024, 3000, 512, False, False, False, False),
    (900, 640, 3001, 512, True, True, False, True),      # three 256-column tiles of H: 256 x 256 dX / dW tiles
    (900, 640, 3001, 0, False, False, True, False),      # the same, one wave, bf16 dW
])
def test_fused_and_split_bit_identical(flp, M, H, V, chunk, ent, dx_f32, dw_bf16, acc):
    """Both schedules run every output tile with the same instructions in the
    same K order (and waves in the same order), so dX and dW agree bit for bit."""
    dev = torch.device("cuda")
    d = case(M, H, V, seed=23, compute_entropy=ent)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    g1 = d["g_lp"].to(dev)
    g2 = d["g_ent"].to(dev) if ent else None
    ws = flp.alloc_workspace(M, H, V, ent, chunk_rows=chunk, device=dev)
    lp, lse, en = flp.forward(X, W, y, compute_entropy=ent, workspace=ws)
    base = torch.randn(V, H, device=dev)
    outs = {}
    for sched in ("split", "fused"):
        dW = (base.clone() if acc else None)
        dX, dW = flp.backward(X, W, y, lse, en, g1, g2, compute_entropy=ent, workspace=ws,
                              dx_dtype=torch.float32 if dx_f32 else torch.bfloat16,
                              dw_dtype=torch.bfloat16 if dw_bf16 else torch.float32, dW=dW,
                              accumulate_dW=acc, schedule=sched)
        torch.cuda.synchronize()
        assert flp.get_error(ws) == flp.FLP_OK
        outs[sched] = (dX.clone(), dW.clone())
    assert torch.equal(outs["split"][0], outs["fused"][0])
    assert torch.equal(outs["split"][1], outs["fused"][1])


def _vsplit_workspace(flp, M, H, V, cols, dev):
    """Smallest workspace whose vocabulary-split chunks are `cols` columns wide."""
    Vp = -(-V // 256) * 256
    want = -(-Vp // cols)
    lo, hi = 0, 1 << 40
    while lo < hi:
        mid = (lo + hi) // 2
        try:
            ok = flp.backward_plan(M, H, V, mid, "vsplit")[1] <= want
        except flp.FlpError:
            ok = False
        hi, lo = (mid, lo) if ok else (hi, mid + 1)
    return torch.empty(lo, dtype=torch.uint8, device=dev)


@pytest.mark.parametrize("M,H,V,cols,dx_f32,dw_bf16,acc", [
    (700, 136, 2100, 768, False, False, False),   # 3 chunks; bf16 dX through the fp32 scratch
    (700, 512, 2100, 512, True, False, True),     # 5 chunks; fp32 dX added in place; wide dX tiles
    (1200, 264, 3001, 1024, False, True, False),  # bf16 dW, each tile written once
    (257, 72, 513, 256, False, False, False),     # three one-tile chunks
    (600, 512, 40000, 16384, False, False, False),  # wide dX tiles; a shorter last chunk
])
def test_vsplit_matches_oracle(flp, M, H, V, cols, dx_f32, dw_bf16, acc):
    """The vocabulary-split backward against the oracle; its dW against a
    one-wave split backward bit for bit (every dW tile has all rows as K in
    both), its dX within the tolerance (fp32 sums over the chunks)."""
    dev = torch.device("cuda")
    d = case(M, H, V, seed=24)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    g1, g2 = d["g_lp"].to(dev), d["g_ent"].to(dev)
    big = flp.alloc_workspace(M, H, V, True, device=dev)
    lp, lse, en = flp.forward(X, W, y, workspace=big)
    ws = _vsplit_workspace(flp, M, H, V, cols, dev)
    assert flp.backward_plan(M, H, V, ws.numel(), "vsplit")[1] == -(-(-(-V // 256) * 256) // cols)
    base = torch.randn(V, H, device=dev)
    dxt = torch.float32 if dx_f32 else torch.bfloat16
    dwt = torch.bfloat16 if dw_bf16 else torch.float32
    outs = {}
    for sched, w in (("vsplit", ws), ("split", big)):
        dW = base.clone() if acc else None
        dX, dW = flp.backward(X, W, y, lse, en, g1, g2, workspace=w, schedule=sched, dx_dtype=dxt,
                              dw_dtype=dwt, dW=dW, accumulate_dW=acc)
        torch.cuda.synchronize()
        assert flp.get_error(w) == flp.FLP_OK
        outs[sched] = (dX.clone(), dW.clone())
    assert torch.equal(outs["vsplit"][1], outs["split"][1])
    Xb, Wb = inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"])
    o_dx, o_dw = oracle.backward(Xb, Wb, d["y"].numpy(), d["g_lp"].double().numpy(),
                                 d["g_ent"].double().numpy())
    check_grad(outs["vsplit"][0], o_dx, "dX")
    want_dw = o_dw + (base.double().cpu().numpy() if acc else 0)
    check_grad(outs["vsplit"][1], want_dw, "dW", rtol=2e-2 if dw_bf16 else RTOL_GRAD)


@pytest.mark.parametrize("M", [4097, 5000])
def test_wave_boundaries_4096(flp, M):
    # 4096-row waves: one extra row (4097) and a two-wave tail (5000), the
    # boundary cases the native commit's "Correctness" section lists.
    run_case(flp, case(M, 64, 1000, seed=15), chunk_rows=4096)


def test_odd_vocabulary_50257(flp):
    # the odd vocabulary that exercises the vocabulary-tail path (chunked GRPO
    # page, "Correctness"): 50257 = 196 * 256 + 81
    run_case(flp, case(300, 64, 50257, seed=16))


def test_large_hidden_small_rows(flp):
    # a long K loop (H = 16384) on a handful of rows and a ragged vocabulary
    run_case(flp, case(70, 16384, 700, seed=17, w_std=0.01))


@pytest.mark.parametrize("scale", [-0.8, 0.0])
def test_negative_and_zero_scale(flp, scale):
    run_case(flp, case(200, 64, 777, seed=18, scale=scale))


def test_wide_ignore_index_and_far_bad_target(flp):
    dev = torch.device("cuda")
    d = case(150, 64, 500, seed=19)
    big = 1 << 40
    d["y"][d["y"] == -100] = big
    d["ignore_index"] = big
    run_case(flp, d)
    d["y"][3] = -(1 << 40)  # out of range, far beyond int32
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    ws = flp.alloc_workspace(150, 64, 500, True, device=dev)
    lp, _, _ = flp.forward(X, W, y, ignore_index=big, workspace=ws)
    assert flp.get_error(ws) == flp.FLP_ERR_BAD_TARGET and torch.isnan(lp[3])


def test_zero_rows(flp):
    dev = torch.device("cuda")
    X = torch.empty(0, 64, dtype=torch.bfloat16, device=dev)
    W = torch.randn(300, 64, device=dev).to(torch.bfloat16)
    y = torch.empty(0, dtype=torch.int64, device=dev)
    lp, lse, en = flp.forward(X, W, y)
    assert lp.numel() == 0
    dW = torch.full((300, 64), 7.0, device=dev)
    _, dW = flp.backward(X, W, y, lse, en, lp, en, dW=dW)
    torch.cuda.synchronize()
    assert torch.all(dW == 0)
    dW.fill_(7.0)
    flp.backward(X, W, y, lse, en, lp, en, dW=dW, accumulate_dW=True)
    torch.cuda.synchronize()
    assert torch.all(dW == 7.0)


def test_dw_bf16_single_wave(flp):
    dev = torch.device("cuda")
    d = case(300, 200, 3001, seed=20)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    g1, g2 = d["g_lp"].to(dev), d["g_ent"].to(dev)
    ws = flp.alloc_workspace(300, 200, 3001, True, device=dev)
    lp, lse, en = flp.forward(X, W, y, workspace=ws)
    _, dW32 = flp.backward(X, W, y, lse, en, g1, g2, workspace=ws)
    dX, dW16 = flp.backward(X, W, y, lse, en, g1, g2, dw_dtype=torch.bfloat16, workspace=ws)
    torch.cuda.synchronize()
    assert dW16.dtype == torch.bfloat16
    # the bf16 output is the fp32 accumulator rounded once (RNE)
    assert torch.equal(dW16, dW32.to(torch.bfloat16))
    Xb, Wb = inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"])
    _, o_dw = oracle.backward(Xb, Wb, d["y"].numpy(), d["g_lp"].double().numpy(),
                              d["g_ent"].double().numpy())
    check_grad(dW16, o_dw, "dW bf16")
    # several row waves, or accumulation, need the fp32 dW
    small = flp.alloc_workspace(300, 200, 3001, True, chunk_rows=128, device=dev)
    with pytest.raises(flp.FlpError) as e:
        flp.backward(X, W, y, lse, en, g1, g2, dw_dtype=torch.bfloat16, workspace=small,
                     schedule="split")
    assert e.value.status == flp.FLP_ERR_UNSUPPORTED
    # the vocabulary split (what auto runs on that workspace) writes each dW tile once
    assert flp.backward_plan(300, 200, 3001, small.numel(), "auto")[2] == "vsplit"
    _, dW16v = flp.backward(X, W, y, lse, en, g1, g2, dw_dtype=torch.bfloat16, workspace=small)
    torch.cuda.synchronize()
    assert torch.equal(dW16v, dW16)
    with pytest.raises(flp.FlpError) as e:
        flp.backward(X, W, y, lse, en, g1, g2, dW=dW16, accumulate_dW=True, workspace=ws)
    assert e.value.status == flp.FLP_ERR_UNSUPPORTED


def test_dx_fp32(flp):
    run_case(flp, case(260, 96, 999, seed=5), dx_dtype=torch.float32)


def test_hot_rows_and_strongly_negative_logits(flp):
    # rows scaled x50 and x100 (logit std ~50 and ~100), and a row whose logits
    # are all -1000 (exp underflows without the max shift): feature 0 is zero
    # everywhere except that row, and W's column 0 is -1000.
    d = case(256, 64, 2000, seed=6, w_std=1.0 / 8)
    X = d["X"].float()
    X[:, 0] = 0
    X[3] *= 50
    X[77] *= 100
    X[100, :] = 0
    X[100, 0] = 1.0
    W = d["W"].float()
    W[:, 0] = -1000.0
    d["X"] = X.to(torch.bfloat16)
    d["W"] = W.to(torch.bfloat16)
    r = run_case(flp, d, check_backward=False)
    assert abs(float(r["en"][100]) - np.log(2000)) < 1e-3
    # Backward.  dX[:, 0] = -1000 * sum_j dZ_ij is zero in exact arithmetic but
    # not once dZ is rounded to bf16 (the contract's rounding point), so that
    # one column measures rounding noise times 1000; every other entry of dX and
    # all of dW are compared.
    dev = torch.device("cuda")
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    dX, dW = flp.backward(X, W, y, r["lse"], r["en"], d["g_lp"].to(dev), d["g_ent"].to(dev),
                          workspace=r["ws"])
    Xb, Wb = inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"])
    o_dx, o_dw = oracle.backward(Xb, Wb, d["y"].numpy(), d["g_lp"].double().numpy(),
                                 d["g_ent"].double().numpy())
    check_grad(dX[:, 1:], o_dx[:, 1:], "dX[:, 1:]")
    check_grad(dW, o_dw, "dW")


def test_all_rows_ignored_and_custom_ignore_index(flp):
    d = case(130, 64, 700, seed=7)
    d["y"][:] = -100
    r = run_case(flp, d)
    assert torch.all(r["lp"] == 0) and torch.all(r["en"] == 0)
    assert torch.all(r["dX"] == 0) and torch.all(r["dW"] == 0)
    d = case(130, 64, 700, seed=8)
    d["y"][d["y"] == -100] = 0  # -100 is an ordinary (out-of-range) target here
    d["y"][::3] = 5
    d["ignore_index"] = 5
    run_case(flp, d)


def test_zero_gradients_and_accumulate(flp):
    dev = torch.device("cuda")
    d = case(300, 64, 900, seed=9)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    ws = flp.alloc_workspace(300, 64, 900, True, device=dev)
    lp, lse, en = flp.forward(X, W, y, workspace=ws)
    dX, dW = flp.backward(X, W, y, lse, en, None, None, workspace=ws)
    torch.cuda.synchronize()
    assert torch.all(dX == 0) and torch.all(dW == 0)
    g1, g2 = d["g_lp"].to(dev), d["g_ent"].to(dev)
    _, dW1 = flp.backward(X, W, y, lse, en, g1, g2, workspace=ws)
    base = torch.randn(900, 64, device=dev)
    dW2 = base.clone()
    flp.backward(X, W, y, lse, en, g1, g2, dW=dW2, accumulate_dW=True, workspace=ws)
    torch.cuda.synchronize()
    torch.testing.assert_close(dW2, base + dW1, rtol=1e-6, atol=1e-6)


def test_determinism(flp):
    dev = torch.device("cuda")
    d = case(700, 136, 2100, seed=10)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    g1, g2 = d["g_lp"].to(dev), d["g_ent"].to(dev)
    ws = flp.alloc_workspace(700, 136, 2100, True, chunk_rows=256, device=dev)
    outs = []
    for _ in range(2):
        lp, lse, en = flp.forward(X, W, y, workspace=ws)
        dX, dW = flp.backward(X, W, y, lse, en, g1, g2, workspace=ws)
        outs.append([t.clone() for t in (lp, lse, en, dX, dW)])
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_bad_target_sets_error_word(flp):
    dev = torch.device("cuda")
    d = case(140, 64, 500, seed=12)
    d["y"][7] = 500
    d["y"][9] = -3
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    ws = flp.alloc_workspace(140, 64, 500, True, device=dev)
    lp, lse, en = flp.forward(X, W, y, workspace=ws)
    assert flp.get_error(ws) == flp.FLP_ERR_BAD_TARGET
    assert torch.isnan(lp[7]) and torch.isnan(lp[9])
    assert torch.isfinite(lp[:7]).all()
    # the next call clears the word
    d2 = case(140, 64, 500, seed=12)
    flp.forward(X, W, d2["y"].to(dev), workspace=ws)
    assert flp.get_error(ws) == flp.FLP_OK


def test_workspace_query_forms_agree(flp):
    """The six-argument query of the boundary contract sizes the default row
    waves (all M rows up to 8192) exactly as the wave-size variant with
    chunk_rows <= 0; a wave size changes only the backward bytes."""
    import ctypes
    lib = flp.load()
    for M, H, V, ent in ((4096, 4096, 131072, 1), (20001, 4096, 128257, 1), (300, 64, 999, 0)):
        a = [ctypes.c_size_t(0) for _ in range(6)]
        assert lib.flp_workspace_query(M, H, V, ent, ctypes.byref(a[0]), ctypes.byref(a[1])) == flp.FLP_OK
        assert lib.flp_workspace_query_ex(M, H, V, ent, 0, ctypes.byref(a[2]),
                                          ctypes.byref(a[3])) == flp.FLP_OK
        assert lib.flp_workspace_query_ex(M, H, V, ent, 1024, ctypes.byref(a[4]),
                                          ctypes.byref(a[5])) == flp.FLP_OK
        assert (a[0].value, a[1].value) == (a[2].value, a[3].value)
        assert a[4].value == a[0].value
        Vp = -(-V // 256) * 256
        assert a[1].value - a[5].value == (min(M + (-M % 128), 8192) - min(1024, M + (-M % 128))) * Vp * 2
        assert flp.backward_plan(M, H, V, a[1].value, "split")[0] == min(M + (-M % 128), 8192)


def test_argument_errors(flp):
    dev = torch.device("cuda")
    d = case(64, 64, 300, seed=13)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    fwd, bwd = flp.workspace_query(64, 64, 300, True)
    small = torch.empty(fwd - 1024, dtype=torch.uint8, device=dev)
    with pytest.raises(flp.FlpError) as e:
        flp.forward(X, W, y, workspace=small)
    assert e.value.status == flp.FLP_ERR_WORKSPACE
    tiny_ws = torch.empty(2048, dtype=torch.uint8, device=dev)
    lse = torch.zeros(64, device=dev)
    en = torch.zeros(64, device=dev)
    with pytest.raises(flp.FlpError) as e:
        flp.backward(X, W, y, lse, en, lse, en, workspace=tiny_ws)
    assert e.value.status == flp.FLP_ERR_WORKSPACE
    # host memory handed over as X is refused before any launch
    import ctypes
    Xh = d["X"].pin_memory()
    lib = flp.load()
    lp_, lse_, en_ = (torch.empty(64, device=dev) for _ in range(3))
    ws_ = flp.alloc_workspace(64, 64, 300, True, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.flp_forward(p(Xh), p(W), p(y), 64, 64, 300, -100, 1.0, 1, p(lp_), p(lse_), p(en_),
                         p(ws_), ws_.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == flp.FLP_ERR_INVALID_ARG
    assert b"not device memory" in lib.flp_last_error_message()
    Xo = torch.zeros(64, 60, dtype=torch.bfloat16, device=dev)
    Wo = torch.zeros(300, 60, dtype=torch.bfloat16, device=dev)
    ws = flp.alloc_workspace(64, 64, 300, True, device=dev)
    with pytest.raises(flp.FlpError) as e:
        flp.forward(Xo[:, :60], Wo, y, workspace=ws)
    assert e.value.status == flp.FLP_ERR_UNSUPPORTED


def test_binding_rejects_tensors_the_abi_cannot_describe(flp):
    """The C ABI takes bare pointers, so the binding refuses non-contiguous,
    wrongly typed or wrongly shaped tensors before calling it."""
    dev = torch.device("cuda")
    d = case(64, 64, 300, seed=25)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    lp, lse, en = flp.forward(X, W, y)
    g = torch.zeros(64, device=dev)
    bad = [
        dict(X=X.t().contiguous().t()),                      # transposed view
        dict(W=W.float()),                                   # fp32 weight
        dict(y=y.int()),                                     # int32 targets
        dict(lse=lse[:32]),                                  # short lse
        dict(dX=torch.empty(64, 64, dtype=torch.float16, device=dev)),
        dict(dW=torch.empty(64, 300, device=dev)),           # transposed dW shape
    ]
    for over in bad:
        a = dict(X=X, W=W, y=y, lse=lse, dX=None, dW=None)
        a.update(over)
        with pytest.raises(ValueError):
            flp.backward(a["X"], a["W"], a["y"], a["lse"], en, g, g, dX=a["dX"], dW=a["dW"])
    with pytest.raises(ValueError):
        flp.forward(X, W, y, logprob=torch.empty(64, dtype=torch.float64, device=dev))
    with pytest.raises(ValueError):
        flp.backward(X, W, y, lse, en, g, g, schedule="nope")


def test_autograd_wrapper(flp):
    dev = torch.device("cuda")
    d = case(200, 64, 1000, seed=14)
    X = d["X"].to(dev).requires_grad_(True)
    W = d["W"].to(dev).requires_grad_(True)
    y = d["y"].to(dev)
    lp, en = flp.fused_linear_logprob(X, W, y)
    (lp * d["g_lp"].to(dev)).sum().backward(retain_graph=True)
    Xb, Wb = inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"])
    o_dx, o_dw = oracle.backward(Xb, Wb, d["y"].numpy(), d["g_lp"].double().numpy(), None)
    check_grad(X.grad, o_dx, "dX")
    check_grad(W.grad, o_dw, "dW", rtol=2e-2)  # W.grad is rounded to bf16 (W's dtype)


def test_headline_schedules_agree_at_full_size(flp):
    """At the full headline shape: the fused backward equals the split one bit
    for bit; the vocabulary split on a 256 MiB workspace (six chunks) gives the
    same dW bits and a dX within rounding (fp32 sums over the chunks, then one
    bf16 rounding).  The split schedule itself is checked against the oracle
    below."""
    dev = torch.device("cuda")
    w = inputs.WORKLOADS["m4096_h4096_v131072"]
    d = inputs.make_inputs(w)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    g1, g2 = d["g_lp"].to(dev), d["g_ent"].to(dev)
    ws = flp.alloc_workspace(w.M, w.H, w.V, True, device=dev)
    small = flp.alloc_workspace(w.M, w.H, w.V, True, chunk_rows=1024, device=dev)
    lp, lse, en = flp.forward(X, W, y, workspace=ws)
    out = {}
    for sched, wsp in (("split", ws), ("fused", ws), ("vsplit", small)):
        dX, dW = flp.backward(X, W, y, lse, en, g1, g2, workspace=wsp, schedule=sched)
        torch.cuda.synchronize()
        assert flp.get_error(wsp) == flp.FLP_OK
        out[sched] = (dX, dW)
    assert flp.backward_plan(w.M, w.H, w.V, small.numel(), "vsplit")[1] == 6
    assert torch.equal(out["fused"][0], out["split"][0])
    assert torch.equal(out["fused"][1], out["split"][1])
    assert torch.equal(out["vsplit"][1], out["split"][1])
    a, b = out["vsplit"][0].float(), out["split"][0].float()
    assert float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b)) < 4e-3


# ------------------------------------------------- full-size workloads (sampled)

@pytest.mark.parametrize("name", sorted(inputs.WORKLOADS))
def test_workload_full_size_sampled(flp, name):
    """The workload at its full size in the launch configuration the bench
    times; forward on a seeded row sample (all tile boundaries near the end
    included), dX on those rows, and dW exactly, with upstream gradients kept
    on a sub-sample of rows so the oracle can form dW from them alone."""
    w = inputs.WORKLOADS[name]
    d = inputs.make_inputs(w)
    n = 48 if w.M * w.V < 4e9 else 24
    rows = inputs.sample_rows(w.M, n, seed=21).numpy()
    dw_rows = rows[::3]
    run_case(flp, d, rows=rows, dw_rows=dw_rows)
