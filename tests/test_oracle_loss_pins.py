"""Pins for the oracle's loss heads (CPU only): closed forms of each branch of
the clipped surrogate, the KL term, the token-mean normalisation over valid
rows, and central finite differences of the scalar loss."""
import math

import numpy as np

import oracle


def test_nll_mean_closed_form():
    lp = np.array([-1.0, -2.5, 0.0, -0.25])
    y = np.array([3, -100, 7, 1])
    per, grad, loss = oracle.loss(lp, y, oracle.LOSS_NLL_MEAN)
    assert abs(loss - (1.0 + 0.0 + 0.25) / 3) < 1e-15
    np.testing.assert_allclose(grad, [-1 / 3, 0, -1 / 3, -1 / 3], atol=1e-15)
    np.testing.assert_allclose(per, [1.0, 0.0, 0.0, 0.25], atol=1e-15)


def test_all_rows_ignored_gives_zero():
    per, grad, loss = oracle.loss(np.array([-1.0, -2.0]), np.array([-100, -100]),
                                  oracle.LOSS_GRPO, old_logprob=np.zeros(2), advantage=np.ones(2))
    assert loss == 0.0 and not grad.any() and not per.any()


def test_grpo_on_policy_is_minus_mean_advantage():
    # lp == old: ratio 1, inside the clip range, surrogate = A
    lp = np.array([-0.7, -1.3, -2.0])
    adv = np.array([0.5, -2.0, 1.5])
    y = np.array([1, 2, 3])
    per, grad, loss = oracle.loss(lp, y, oracle.LOSS_GRPO, old_logprob=lp, advantage=adv)
    assert abs(loss - (-adv.mean())) < 1e-15
    np.testing.assert_allclose(grad, -adv / 3, atol=1e-15)


def test_grpo_clip_branches():
    eps = 0.2
    y = np.array([0, 0, 0, 0])
    old = np.zeros(4)
    lp = np.array([math.log(1.5), math.log(1.5), math.log(0.5), math.log(0.5)])
    adv = np.array([1.0, -1.0, 1.0, -1.0])
    per, grad, loss = oracle.loss(lp, y, oracle.LOSS_GRPO, old_logprob=old, advantage=adv,
                                  eps_low=eps, eps_high=eps)
    # r=1.5, A>0: clipped at 1.2 -> term -1.2, zero gradient
    # r=1.5, A<0: min(-1.5, -1.2) = -1.5 (unclipped) -> term 1.5, grad -(r A)/N = 1.5/4
    # r=0.5, A>0: min(0.5, 0.8) = 0.5 (unclipped) -> term -0.5, grad -0.5/4
    # r=0.5, A<0: min(-0.5, -0.8) = -0.8 (clipped) -> term 0.8, zero gradient
    np.testing.assert_allclose(per, [-1.2, 1.5, -0.5, 0.8], atol=1e-12)
    np.testing.assert_allclose(grad, [0.0, 1.5 / 4, -0.5 / 4, 0.0], atol=1e-12)
    assert abs(loss - (-1.2 + 1.5 - 0.5 + 0.8) / 4) < 1e-12


def test_kl_term_closed_form():
    lp = np.array([-1.0, -2.0])
    ref = np.array([-1.5, -2.0])
    y = np.array([0, 1])
    beta = 0.3
    per, grad, loss = oracle.loss(lp, y, oracle.LOSS_GRPO, old_logprob=lp, advantage=np.zeros(2),
                                  ref_logprob=ref, beta=beta)
    d = -0.5
    kl0 = math.exp(d) - d - 1
    np.testing.assert_allclose(per, [beta * kl0, 0.0], atol=1e-15)
    np.testing.assert_allclose(grad, [beta * (1 - math.exp(d)) / 2, 0.0], atol=1e-15)


def test_grpo_gradient_matches_finite_differences():
    r = np.random.default_rng(3)
    M = 9
    lp = r.normal(-2, 0.5, M)
    old = lp + r.normal(0, 0.1, M)  # ratios near 1, away from the clip edges
    adv = r.normal(0, 1, M)
    ref = lp + r.normal(0, 0.3, M)
    y = r.integers(0, 10, M)
    y[4] = -100
    kw = dict(old_logprob=old, advantage=adv, ref_logprob=ref, eps_low=0.3, eps_high=0.4, beta=0.05)
    _, grad, _ = oracle.loss(lp, y, oracle.LOSS_GRPO, **kw)
    eps = 1e-6
    for i in range(M):
        a, b = lp.copy(), lp.copy()
        a[i] += eps
        b[i] -= eps
        fd = (oracle.loss(a, y, oracle.LOSS_GRPO, **kw)[2] - oracle.loss(b, y, oracle.LOSS_GRPO, **kw)[2]) / (2 * eps)
        assert abs(fd - grad[i]) < 1e-8, (i, fd, grad[i])
    assert grad[4] == 0.0
