"""Loss heads on the GPU (flp_loss) against the oracle, alone and chained
through the fused forward and backward."""
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


def _rand(seed, M):
    r = np.random.default_rng(seed)
    lp = r.normal(-3, 1.0, M).astype(np.float32)
    old = (lp + r.normal(0, 0.3, M)).astype(np.float32)
    adv = r.normal(0, 1, M).astype(np.float32)
    ref = (lp + r.normal(0, 0.2, M)).astype(np.float32)
    y = r.integers(0, 1000, M)
    y[r.random(M) < 0.1] = -100
    return lp, old, adv, ref, y


@pytest.mark.parametrize("M", [1, 1000, 5000, 70001])
def test_loss_heads_match_oracle(flp, M):
    dev = torch.device("cuda")
    lp, old, adv, ref, y = _rand(M, M)
    t = lambda a: torch.from_numpy(a).to(dev)
    yt = torch.from_numpy(y.astype(np.int64)).to(dev)
    for kind, kw, okw in (
        (flp.FLP_LOSS_NLL_MEAN, {}, {}),
        (flp.FLP_LOSS_CLIPPED_SURROGATE,
         dict(old_logprob=t(old), advantage=t(adv), eps_low=0.2, eps_high=0.28),
         dict(old_logprob=old, advantage=adv, eps_low=0.2, eps_high=0.28)),
        (flp.FLP_LOSS_CLIPPED_SURROGATE,
         dict(old_logprob=t(old), advantage=t(adv), ref_logprob=t(ref), beta=0.04),
         dict(old_logprob=old, advantage=adv, ref_logprob=ref, beta=0.04)),
    ):
        loss, grad, per = flp.loss(t(lp), yt, kind, **kw)
        o_per, o_grad, o_loss = oracle.loss(lp.astype(np.float64), y, kind,
                                            **{k: (v.astype(np.float64) if isinstance(v, np.ndarray) else v)
                                               for k, v in okw.items()})
        torch.cuda.synchronize()
        np.testing.assert_allclose(per.cpu().numpy(), o_per, rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(grad.cpu().numpy(), o_grad, rtol=1e-5, atol=1e-9)
        assert abs(float(loss.item()) - o_loss) <= 1e-5 * max(1.0, abs(o_loss))
        # deterministic
        loss2, grad2, _ = flp.loss(t(lp), yt, kind, **kw)
        assert torch.equal(loss, loss2) and torch.equal(grad, grad2)


def test_clipped_surrogate_through_forward_and_backward(flp):
    # lm_head forward -> clipped-surrogate loss -> its gradient into the fused
    # backward, against the oracle chained the same way
    dev = torch.device("cuda")
    d = inputs.make_inputs(inputs.custom("grpo", 600, 128, 3000, w_std=0.08, ignore_frac=0.1,
                                         seed=51), with_grads=False)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    lp, lse, en = flp.forward(X, W, y)
    r = np.random.default_rng(52)
    Xb, Wb = inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"])
    o_lp, _, _ = oracle.forward(Xb, Wb, d["y"].numpy())
    old = (o_lp + r.normal(0, 0.02, o_lp.shape)).astype(np.float32)  # ratios near 1
    adv = r.normal(0, 1, o_lp.shape).astype(np.float32)
    loss, grad, _ = flp.loss(lp, y, flp.FLP_LOSS_CLIPPED_SURROGATE,
                             old_logprob=torch.from_numpy(old).to(dev),
                             advantage=torch.from_numpy(adv).to(dev), eps_low=0.2, eps_high=0.2)
    dX, dW = flp.backward(X, W, y, lse, en, grad, None)
    _, o_grad, o_loss = oracle.loss(o_lp, d["y"].numpy(), oracle.LOSS_GRPO,
                                    old_logprob=old.astype(np.float64), advantage=adv.astype(np.float64))
    o_dx, o_dw = oracle.backward(Xb, Wb, d["y"].numpy(), o_grad, None)
    torch.cuda.synchronize()
    assert abs(float(loss.item()) - o_loss) < 2e-3
    for got, want, name in ((dX, o_dx, "dX"), (dW, o_dw, "dW")):
        g = got.float().cpu().double().numpy()
        rel = np.linalg.norm(g - want) / np.linalg.norm(want)
        assert rel < 1e-2, (name, rel)
