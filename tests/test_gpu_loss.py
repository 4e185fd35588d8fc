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
        (flp.FLP_LOSS_NLL_SUM, {}, {}),
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


def _offsets(seed, M, B):
    """Ragged, sorted sequence offsets over [0, M] with some empty sequences."""
    r = np.random.default_rng(seed)
    cuts = np.sort(r.integers(0, M + 1, B - 1))
    return np.concatenate([[0], cuts, [M]]).astype(np.int64)


@pytest.mark.parametrize("M,B", [(1, 1), (1000, 7), (5000, 300), (70001, 64), (70001, 2000)])
def test_policy_loss_matches_oracle(flp, M, B):
    """Every ratio level and aggregation (bnpo, grpo, dapo with and without
    num_items_in_batch) against the oracle; the token-level ratio with the
    token mean is also the clipped surrogate of flp_loss."""
    dev = torch.device("cuda")
    lp, old, adv, ref, y = _rand(M + 17, M)
    off = _offsets(M + B, M, B)
    t = lambda a: torch.from_numpy(a).to(dev)
    yt = torch.from_numpy(y.astype(np.int64)).to(dev)
    f64 = lambda a: a.astype(np.float64)
    for is_level in (flp.FLP_IS_TOKEN, flp.FLP_IS_SEQUENCE):
        for agg, norm in ((flp.FLP_AGG_TOKEN_MEAN, 0.0), (flp.FLP_AGG_SEQUENCE_MEAN, 0.0),
                          (flp.FLP_AGG_SUM_OVER, 0.0), (flp.FLP_AGG_SUM_OVER, 3.0 * M + 5)):
            for with_ref in (False, True):
                kw = dict(eps_low=0.2, eps_high=0.28, beta=0.04 if with_ref else 0.0,
                          is_level=is_level, aggregation=agg, normalizer=norm)
                loss, grad, per = flp.policy_loss(t(lp), yt, t(old), t(adv), seq_offsets=t(off),
                                                  ref_logprob=t(ref) if with_ref else None, **kw)
                o_per, o_grad, o_loss = oracle.policy_loss(
                    f64(lp), y, f64(old), f64(adv), off, ref_logprob=f64(ref) if with_ref else None, **kw)
                torch.cuda.synchronize()
                tag = (is_level, agg, norm, with_ref)
                np.testing.assert_allclose(per.cpu().numpy(), o_per, rtol=1e-6, atol=1e-6, err_msg=str(tag))
                np.testing.assert_allclose(grad.cpu().numpy(), o_grad, rtol=1e-5, atol=1e-10,
                                           err_msg=str(tag))
                assert abs(float(loss.item()) - o_loss) <= 1e-6 * max(1.0, abs(o_loss)), tag
                loss2, grad2, _ = flp.policy_loss(t(lp), yt, t(old), t(adv), seq_offsets=t(off),
                                                  ref_logprob=t(ref) if with_ref else None, **kw)
                assert torch.equal(loss, loss2) and torch.equal(grad, grad2), tag
    # no offsets: one sequence of every row
    loss, grad, _ = flp.policy_loss(t(lp), yt, t(old), t(adv), is_level=flp.FLP_IS_SEQUENCE)
    _, o_grad, o_loss = oracle.policy_loss(f64(lp), y, f64(old), f64(adv), None, is_level=1)
    torch.cuda.synchronize()
    np.testing.assert_allclose(grad.cpu().numpy(), o_grad, rtol=1e-5, atol=1e-10)
    assert abs(float(loss.item()) - o_loss) <= 1e-6 * max(1.0, abs(o_loss))


def test_dapo_sequence_loss_through_forward_and_backward(flp):
    """The page's benchmark configuration (dapo, sequence-level ratio,
    num_items_in_batch, beta = 0, eps 0.2 / 0.2) on four sequences of mixed
    lengths: lm_head forward -> policy loss -> its gradient into the fused
    backward, against the oracle chained the same way."""
    dev = torch.device("cuda")
    M = 900
    d = inputs.make_inputs(inputs.custom("dapo", M, 128, 3001, w_std=0.08, ignore_frac=0.1, seed=53),
                           with_grads=False)
    X, W, y = d["X"].to(dev), d["W"].to(dev), d["y"].to(dev)
    lp, lse, en = flp.forward(X, W, y)
    Xb, Wb = inputs.bf16_bits(d["X"]), inputs.bf16_bits(d["W"])
    o_lp, _, _ = oracle.forward(Xb, Wb, d["y"].numpy())
    r = np.random.default_rng(54)
    off = np.array([0, 150, 400, 700, M], dtype=np.int64)
    old = (o_lp + r.normal(0, 0.02, M)).astype(np.float32)
    adv = np.repeat(r.normal(0, 1, 4), np.diff(off)).astype(np.float32)  # one advantage per sequence
    n_items = 4 * 1000.0
    loss, grad, _ = flp.policy_loss(lp, y, torch.from_numpy(old).to(dev), torch.from_numpy(adv).to(dev),
                                    seq_offsets=torch.from_numpy(off).to(dev), is_level=flp.FLP_IS_SEQUENCE,
                                    aggregation=flp.FLP_AGG_SUM_OVER, normalizer=n_items)
    dX, dW = flp.backward(X, W, y, lse, en, grad, None)
    _, o_grad, o_loss = oracle.policy_loss(o_lp, d["y"].numpy(), old.astype(np.float64),
                                           adv.astype(np.float64), off, is_level=1, aggregation=2,
                                           normalizer=n_items)
    o_dx, o_dw = oracle.backward(Xb, Wb, d["y"].numpy(), o_grad, None)
    torch.cuda.synchronize()
    assert abs(float(loss.item()) - o_loss) < 2e-3  # the two chains differ by the forward's error
    for got, want, name in ((dX, o_dx, "dX"), (dW, o_dw, "dW")):
        g = got.float().cpu().double().numpy()
        rel = np.linalg.norm(g - want) / np.linalg.norm(want)
        assert rel < 1e-2, (name, rel)
