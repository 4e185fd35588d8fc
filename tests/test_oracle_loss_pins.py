"""Pins for the oracle's loss heads (CPU only): closed forms of each branch of
the clipped surrogate, the KL term, the token-mean normalisation over valid
rows, and central finite differences of the scalar loss."""
import math

import numpy as np
import pytest

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


# ------------------------------------------------ token-sum NLL

def test_nll_sum_closed_form():
    lp = np.array([-1.0, -2.5, 0.0, -0.25])
    y = np.array([3, -100, 7, 1])
    per, grad, loss = oracle.loss(lp, y, oracle.LOSS_NLL_SUM)
    assert loss == 1.25
    np.testing.assert_array_equal(grad, [-1.0, 0.0, -1.0, -1.0])
    np.testing.assert_array_equal(per, [1.0, 0.0, 0.0, 0.25])


# ------------------------------------------------ policy loss over sequences

def test_sequence_ratio_closed_form():
    """Two sequences; hand-derived values.  Sequence 0 has two tokens with
    lp - old = 0.1 and 0.3 (one ignored row between them): log r = 0.2,
    r = e^0.2 = 1.2214 > 1 + 0.2.  With A = +1 the clipped term wins
    (-1.2 each, zero gradient); with A = -1 the unclipped one (r each, and
    each lp_u gets -A r / n_b summed over the two tokens' weights).
    Sequence 1 has one token, lp - old = log 0.9 (inside the range)."""
    lp = np.array([-1.0, -5.0, -2.0, -0.5])
    old = np.array([-1.1, -5.0, -2.3, -0.5 - math.log(0.9)])
    y = np.array([4, -100, 2, 9])
    off = np.array([0, 3, 4])
    r0, r1 = math.exp(0.2), 0.9
    for A0, A1 in ((1.0, 2.0), (-1.0, 2.0)):
        adv = np.array([A0, 0.0, A0, A1])
        per, grad, loss = oracle.policy_loss(lp, y, old, adv, off, is_level=oracle.IS_SEQUENCE,
                                             aggregation=oracle.AGG_SUM_OVER, normalizer=5.0)
        t0 = -min(r0 * A0, 1.2 * A0)
        t1 = -r1 * A1
        np.testing.assert_allclose(per, [t0, 0.0, t0, t1], rtol=1e-14)
        assert abs(loss - (2 * t0 + t1) / 5.0) < 1e-14
        g0 = 0.0 if A0 > 0 else (2 * (-r0 * A0) / 5.0) / 2
        np.testing.assert_allclose(grad, [g0, 0.0, g0, -r1 * A1 / 5.0], rtol=1e-14, atol=1e-16)
    # aggregation: sequence mean (grpo) with the same terms, A0 = -1
    per, grad, loss = oracle.policy_loss(lp, y, old, np.array([-1.0, 0, -1.0, 2.0]), off,
                                         is_level=oracle.IS_SEQUENCE,
                                         aggregation=oracle.AGG_SEQUENCE_MEAN)
    t0, t1 = r0, -r1 * 2.0
    assert abs(loss - 0.5 * ((2 * t0) / 2 + t1 / 1)) < 1e-14


def _policy_case(seed, M=23):
    r = np.random.default_rng(seed)
    lp = r.normal(-2, 0.5, M)
    old = lp + r.normal(0, 0.05, M)  # ratios near 1, away from the clip edges
    adv = r.normal(0, 1, M)
    ref = lp + r.normal(0, 0.3, M)
    y = r.integers(0, 10, M)
    y[[3, 11]] = -100
    off = np.array([0, 5, 5, 12, 20, M])  # an empty sequence, ragged lengths
    return lp, y, old, adv, ref, off


@pytest.mark.parametrize("is_level", [0, 1])
@pytest.mark.parametrize("agg,norm", [(0, 0.0), (1, 0.0), (2, 0.0), (2, 57.0)])
def test_policy_loss_gradient_matches_finite_differences(is_level, agg, norm):
    lp, y, old, adv, ref, off = _policy_case(5)
    kw = dict(seq_offsets=off, ref_logprob=ref, eps_low=0.3, eps_high=0.4, beta=0.05,
              is_level=is_level, aggregation=agg, normalizer=norm)
    _, grad, _ = oracle.policy_loss(lp, y, old, adv, **kw)
    eps = 1e-6
    for i in range(lp.size):
        a, b = lp.copy(), lp.copy()
        a[i] += eps
        b[i] -= eps
        fd = (oracle.policy_loss(a, y, old, adv, **kw)[2] - oracle.policy_loss(b, y, old, adv, **kw)[2]) / (2 * eps)
        assert abs(fd - grad[i]) < 1e-8, (i, fd, grad[i])
    assert grad[3] == 0.0 and grad[11] == 0.0


def test_policy_loss_reductions():
    lp, y, old, adv, ref, off = _policy_case(6)
    kw = dict(ref_logprob=ref, eps_low=0.2, eps_high=0.28, beta=0.04)
    # token-level ratio, token mean: the clipped surrogate of flpo_loss
    p0, g0, l0 = oracle.loss(lp, y, oracle.LOSS_GRPO, old_logprob=old, advantage=adv, **kw)
    p1, g1, l1 = oracle.policy_loss(lp, y, old, adv, off, **kw)
    np.testing.assert_allclose(p1, p0, rtol=1e-14)
    np.testing.assert_allclose(g1, g0, rtol=1e-13, atol=1e-17)
    assert abs(l1 - l0) < 1e-14
    # dapo without num_items_in_batch normalises by the token count: bnpo
    _, g2, l2 = oracle.policy_loss(lp, y, old, adv, off, aggregation=oracle.AGG_SUM_OVER, **kw)
    np.testing.assert_allclose(g2, g0, rtol=1e-13, atol=1e-17)
    assert abs(l2 - l0) < 1e-14
    # ... and with it, the same sum over another denominator
    N = int((y != -100).sum())
    _, g3, l3 = oracle.policy_loss(lp, y, old, adv, off, aggregation=oracle.AGG_SUM_OVER,
                                   normalizer=4 * N, **kw)
    assert abs(4 * l3 - l0) < 1e-14
    np.testing.assert_allclose(4 * g3, g0, rtol=1e-13, atol=1e-17)
    # one token per sequence: the sequence-level ratio is the token-level one
    M = lp.size
    ones = np.arange(M + 1)
    for agg in (0, 1, 2):
        a = oracle.policy_loss(lp, y, old, adv, ones, aggregation=agg, is_level=1, **kw)
        b = oracle.policy_loss(lp, y, old, adv, ones, aggregation=agg, is_level=0, **kw)
        np.testing.assert_allclose(a[0], b[0], rtol=1e-14)
        np.testing.assert_allclose(a[1], b[1], rtol=1e-13, atol=1e-17)
    # sequences of equal token counts: the sequence mean is the token mean
    yy = np.zeros(20, dtype=np.int64)
    eq = np.array([0, 5, 10, 15, 20])
    c = oracle.policy_loss(lp[:20], yy, old[:20], adv[:20], eq, aggregation=1, is_level=1, **kw)
    d = oracle.policy_loss(lp[:20], yy, old[:20], adv[:20], eq, aggregation=0, is_level=1, **kw)
    assert abs(c[2] - d[2]) < 1e-14
    np.testing.assert_allclose(c[1], d[1], rtol=1e-13, atol=1e-17)
    # no offsets: one sequence of every row
    e = oracle.policy_loss(lp, y, old, adv, None, is_level=1, **kw)
    f = oracle.policy_loss(lp, y, old, adv, np.array([0, M]), is_level=1, **kw)
    np.testing.assert_array_equal(e[1], f[1])
