"""The allocation-free forward (flp_forward_noalloc) against flp_forward.

flp_forward_noalloc serves callers that cannot call cudaMalloc and have no
workspace to hand (a host framework that owns all device memory, or a
latency-critical loop that cannot afford cudaMalloc's implicit device
synchronisation): its scratch is a fixed 16 MiB device array inside the
library.  Here it is called through the C ABI twice in a row, on two
different problems (so the second call runs on whatever the first left in the
shared array), and each result is compared with the workspace-based entry
point: bit for bit where that entry point's own plan fits the static array
(the same plan runs), else within the forward tolerance of the other GPU
tests, and then also against the fp64 oracle on a row sample.  This file is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from entropy_loss_gb300 import inputs

pytestmark = pytest.mark.gpu

ATOL_FWD = 2e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from entropy_loss_gb300 import build, flp
    build.build()
    return flp.load()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(lib, X, W, y, lp, lse, en, ent, scale, stream):
    M, H = X.shape
    V = W.shape[0]
    return lib.flp_forward_noalloc(_p(X), _p(W), _p(y), M, H, V, -100, scale, int(ent), _p(lp),
                                   _p(lse), _p(en if ent else None), ctypes.c_void_p(stream))


def test_noalloc_forward_matches_workspace_forward_twice(lib):
    from entropy_loss_gb300 import flp
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream().cuda_stream
    cases = [inputs.custom("a", 1000, 256, 20000, w_std=0.05, ignore_frac=0.1, seed=31),
             inputs.custom("b", 333, 136, 9001, w_std=0.08, ignore_frac=0.1, seed=32,
                           compute_entropy=False, scale=1.0 / 0.7)]
    for w in cases:
        d = inputs.make_inputs(w, with_grads=False)
        X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
        ent, scale = d["compute_entropy"], d["scale"]
        M = w.M
        lp = torch.full((M,), float("nan"), device=dev)
        lse = torch.full((M,), float("nan"), device=dev)
        en = torch.full((M,), float("nan"), device=dev) if ent else None
        st = _call_noalloc(lib, X, W, y, lp, lse, en, ent, scale, stream)
        assert st == flp.FLP_OK, lib.flp_last_error_message()
        r_lp, r_lse, r_en = flp.forward(X, W, y, scale=scale, compute_entropy=ent)
        torch.cuda.synchronize()
        f, _ = flp.workspace_query(M, w.H, w.V, ent)
        assert f <= flp.STATIC_SCRATCH_BYTES  # the workspace forward's own plan: same bits
        assert torch.equal(lp, r_lp)
        assert torch.equal(lse, r_lse)
        if ent:
            assert torch.equal(en, r_en)


def test_noalloc_takes_fewer_splits_when_the_default_plan_does_not_fit(lib):
    """12288 rows, H = 1024, a 128K vocabulary: flp_forward's own plan (128
    splits) needs 36 MiB of partials, so the allocation-free forward runs a
    plan with fewer splits that fits its 16 MiB (same values as flp_forward
    within the forward tolerance, and as the fp64 oracle on a row sample that
    includes the last pair tiles)."""
    from entropy_loss_gb300 import flp
    M, H, V = 12288, 1024, 131072
    f, _ = flp.workspace_query(M, H, V, True)
    assert f > flp.STATIC_SCRATCH_BYTES
    dev = torch.device("cuda")
    d = inputs.make_inputs(inputs.custom("c", M, H, V, w_std=0.05, ignore_frac=0.05, seed=33),
                           with_grads=False)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    lp = torch.full((M,), float("nan"), device=dev)
    lse = torch.full((M,), float("nan"), device=dev)
    en = torch.full((M,), float("nan"), device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    st = _call_noalloc(lib, X, W, y, lp, lse, en, True, 1.0, stream)
    assert st == flp.FLP_OK, lib.flp_last_error_message()
    r_lp, r_lse, r_en = flp.forward(X, W, y)
    torch.cuda.synchronize()
    torch.testing.assert_close(lp, r_lp, rtol=0, atol=ATOL_FWD)
    torch.testing.assert_close(lse, r_lse, rtol=0, atol=ATOL_FWD)
    torch.testing.assert_close(en, r_en, rtol=0, atol=ATOL_FWD)
    rows = inputs.sample_rows(M, 64, seed=34).numpy()
    o_lp, o_lse, o_en = oracle.forward(inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"]),
                                       d["y"].numpy(), rows=rows)
    sel = torch.as_tensor(rows, device=dev)
    for name, got, want in (("logprob", lp, o_lp), ("lse", lse, o_lse), ("entropy", en, o_en)):
        err = np.abs(got[sel].double().cpu().numpy() - want)
        assert err.max() <= ATOL_FWD, f"{name}: max abs err {err.max():.3e} against the oracle"


def test_noalloc_rejects_problems_beyond_the_static_scratch(lib):
    from entropy_loss_gb300 import flp
    # 2^20 rows need at least 3 x 8 MiB of partials (two per split) and 4 MiB
    # of target logits plus the header, beyond 16 MiB whatever the split count
    # or the vocabulary size; W matches V, so nothing could be read out of
    # bounds even if the size check were missing
    M, H, V = 1 << 20, 8, 16
    f, _ = flp.workspace_query(M, H, V, True)
    assert f > flp.STATIC_SCRATCH_BYTES
    dev = torch.device("cuda")
    X = torch.zeros(M, H, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(V, H, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(M, dtype=torch.int64, device=dev)
    out = torch.empty(M, device=dev)
    st = lib.flp_forward_noalloc(_p(X), _p(W), _p(y), M, H, V, -100, 1.0, 1, _p(out), _p(out),
                                 _p(out), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == flp.FLP_ERR_UNSUPPORTED
    assert b"static scratch" in lib.flp_last_error_message()
