"""Out-of-bounds write detection: every output and the workspace sit inside a
larger device buffer whose guard bands hold a known byte pattern; after the
forward and backward on ragged shapes (rows, vocabulary and hidden size not
multiples of the tiles, several waves) the guards must be untouched and the
outputs finite."""
import pytest
import torch

from entropy_loss_gb300 import inputs

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side (keeps 16-byte alignment)
PATTERN = 0xA5


@pytest.fixture(scope="module")
def flp():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from entropy_loss_gb300 import build, flp as _flp
    build.build()
    _flp.load()
    return _flp


class Guarded:
    def __init__(self, nbytes, dev):
        self.n = nbytes
        self.raw = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=dev)

    def view(self, dtype, shape):
        return self.raw[GUARD:GUARD + self.n].view(dtype).view(shape)

    def intact(self):
        return bool(torch.all(self.raw[:GUARD] == PATTERN)) and bool(
            torch.all(self.raw[GUARD + self.n:] == PATTERN))


@pytest.mark.parametrize("schedule", ["split", "fused", "vsplit"])
@pytest.mark.parametrize("M,H,V,chunk", [
    (300, 200, 3001, 128), (257, 72, 513, 0), (700, 136, 2100, 256),
    # wide dX tiles whose second 256-column half is mostly outside (H = 264)
    # or entirely inside H (H = 512), over several waves
    (300, 264, 16500, 256), (700, 512, 16500, 256),
])
def test_no_writes_outside_buffers(flp, M, H, V, chunk, schedule):
    if schedule == "fused" and chunk == 128:
        pytest.skip("fused waves are multiples of 256 rows")
    if schedule == "vsplit":
        try:
            flp.backward_plan(M, H, V, max(flp.workspace_query(M, H, V, True, chunk)), "vsplit")
        except flp.FlpError:
            pytest.skip("the workspace does not hold the vocabulary split's dX scratch and a dZ chunk")
    dev = torch.device("cuda")
    d = inputs.make_inputs(inputs.custom("guard", M, H, V, w_std=0.05, ignore_frac=0.1, seed=61))
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    f_bytes, b_bytes = flp.workspace_query(M, H, V, True, chunk)
    ws_g = Guarded(max(f_bytes, b_bytes), dev)
    lp_g, lse_g, en_g = (Guarded(M * 4, dev) for _ in range(3))
    dx_g, dxf_g, dw_g = Guarded(M * H * 2, dev), Guarded(M * H * 4, dev), Guarded(V * H * 4, dev)
    ws = ws_g.view(torch.uint8, (ws_g.n,))
    lp, lse, en = (g.view(torch.float32, (M,)) for g in (lp_g, lse_g, en_g))
    flp.forward(X, W, y, logprob=lp, lse=lse, entropy=en, workspace=ws)
    dX = dx_g.view(torch.bfloat16, (M, H))
    dW = dw_g.view(torch.float32, (V, H))
    flp.backward(X, W, y, lse, en, d["g_lp"].to(dev), d["g_ent"].to(dev), dX=dX, dW=dW, workspace=ws,
                 schedule=schedule)
    dXf = dxf_g.view(torch.float32, (M, H))
    flp.backward(X, W, y, lse, en, d["g_lp"].to(dev), d["g_ent"].to(dev), dX=dXf, dW=dW,
                 accumulate_dW=True, workspace=ws, schedule=schedule)
    torch.cuda.synchronize()
    assert flp.get_error(ws) == flp.FLP_OK
    for name, g in (("workspace", ws_g), ("logprob", lp_g), ("lse", lse_g), ("entropy", en_g),
                    ("dX bf16", dx_g), ("dX fp32", dxf_g), ("dW", dw_g)):
        assert g.intact(), f"write outside {name}"
    for t in (lp, lse, en, dX.float(), dXf, dW):
        assert torch.isfinite(t).all()
