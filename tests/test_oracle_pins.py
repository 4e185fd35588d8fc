"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: a closed form, an
invariant of the mathematics, brute force written independently in pure
Python, or central finite differences of the oracle's own forward.  Together
they are chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a missing scale) fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def to_bf16_bits(a):
    """Round fp64 values to bf16 bit patterns (via fp32, RNE) with numpy."""
    f = np.asarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def rand_case(seed, M, H, V, xs=1.0, ws=0.5):
    r = rng(seed)
    X = r.normal(0, xs, (M, H))
    W = r.normal(0, ws, (V, H))
    y = r.integers(0, V, M)
    return X, W, y


# ---------------------------------------------------------------- closed forms

def test_golden_integer_logits():
    with open(os.path.join(GOLDEN, "integer_logits.json")) as f:
        case = json.load(f)
    X = np.array(case["X"], dtype=np.float64)
    W = np.array(case["W"], dtype=np.float64)
    y = np.array(case["y"], dtype=np.int64)
    lp, lse, ent = oracle.forward(X, W, y, ignore_index=case["ignore_index"], scale=case["scale"])
    env = {"log": math.log, "exp": math.exp, "e": math.e, "__builtins__": {}}
    for key, got in (("lse", lse), ("logprob", lp), ("entropy", ent)):
        want = np.array([eval(s, env) for s in case["expected"][key]])
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12, err_msg=key)


@pytest.mark.parametrize("V", [1, 7, 4096])
@pytest.mark.parametrize("how", ["W0", "X0", "s0"])
def test_uniform_logits_closed_form(V, how):
    X, W, y = rand_case(1, 5, 16, V)
    s = 1.3
    if how == "W0":
        W[:] = 0
    elif how == "X0":
        X[:] = 0
    else:
        s = 0.0
    lp, lse, ent = oracle.forward(X, W, y, scale=s)
    np.testing.assert_allclose(lp, -math.log(V), atol=1e-12)
    np.testing.assert_allclose(lse, math.log(V), atol=1e-12)
    np.testing.assert_allclose(ent, math.log(V), atol=1e-12)


def test_single_class():
    X, W, y = rand_case(2, 6, 8, 1, ws=2.0)
    y[:] = 0
    s = 0.7
    lp, lse, ent = oracle.forward(X, W, y, scale=s)
    np.testing.assert_allclose(lp, 0.0, atol=1e-12)
    np.testing.assert_allclose(ent, 0.0, atol=1e-12)
    np.testing.assert_allclose(lse, s * (X @ W[0]), rtol=1e-13, atol=1e-12)


def test_two_classes_is_logistic():
    # With V = 2, logprob is the log-sigmoid of the logit margin and the entropy
    # is the binary entropy of the sigmoid: textbook logistic regression.
    X, W, y = rand_case(3, 32, 12, 2, ws=1.0)
    s = 1.7
    lp, lse, ent = oracle.forward(X, W, y, scale=s)
    for i in range(32):
        d = s * float(X[i] @ (W[y[i]] - W[1 - y[i]]))
        want_lp = -math.log1p(math.exp(-d)) if d > 0 else d - math.log1p(math.exp(d))
        p = 1.0 / (1.0 + math.exp(-d))
        want_ent = -(p * math.log(p) + (1 - p) * math.log(1 - p))
        assert abs(lp[i] - want_lp) < 1e-12
        assert abs(ent[i] - want_ent) < 1e-12


# ------------------------------------------------------------------ invariants

def test_probabilities_sum_to_one():
    M, H, V = 3, 10, 37
    X, W, _ = rand_case(4, M, H, V, ws=1.5)
    total = np.zeros(M)
    for j in range(V):
        lp, _, _ = oracle.forward(X, W, np.full(M, j), compute_entropy=False)
        total += np.exp(lp)
    np.testing.assert_allclose(total, 1.0, atol=1e-13)


def test_entropy_bounds_and_logprob_sign():
    for seed, ws in ((5, 0.1), (6, 1.0), (7, 10.0)):
        X, W, y = rand_case(seed, 40, 16, 97, ws=ws)
        lp, lse, ent = oracle.forward(X, W, y)
        assert np.all(ent >= -1e-12) and np.all(ent <= math.log(97) + 1e-12)
        assert np.all(lp <= 1e-12)


def test_shift_invariance():
    X, W, y = rand_case(8, 20, 9, 50)
    s, c = 0.8, 3.25
    lp0, lse0, ent0 = oracle.forward(X, W, y, scale=s)
    X1 = np.concatenate([X, np.ones((20, 1))], axis=1)
    W1 = np.concatenate([W, np.full((50, 1), c)], axis=1)
    lp1, lse1, ent1 = oracle.forward(X1, W1, y, scale=s)
    np.testing.assert_allclose(lse1 - lse0, s * c, atol=1e-12)
    np.testing.assert_allclose(lp1, lp0, atol=1e-12)
    np.testing.assert_allclose(ent1, ent0, atol=1e-12)


def test_strongly_negative_rows_stay_finite():
    # Every logit near -1e4: a sum-exp without the max shift would underflow to
    # zero and give -inf/NaN.  The SkyRL page's correctness fix starts the LSE
    # from the true row maximum; the results must equal the unshifted ones.
    X, W, y = rand_case(9, 16, 8, 64)
    lp0, lse0, ent0 = oracle.forward(X, W, y)
    X1 = np.concatenate([X, np.ones((16, 1))], axis=1)
    W1 = np.concatenate([W, np.full((64, 1), -1e4)], axis=1)
    lp1, lse1, ent1 = oracle.forward(X1, W1, y)
    assert np.all(np.isfinite(lp1)) and np.all(np.isfinite(ent1)) and np.all(np.isfinite(lse1))
    np.testing.assert_allclose(lse1, lse0 - 1e4, atol=1e-9)
    np.testing.assert_allclose(lp1, lp0, atol=1e-9)
    np.testing.assert_allclose(ent1, ent0, atol=1e-9)


def test_vocab_permutation_invariance():
    X, W, y = rand_case(10, 12, 7, 31)
    perm = rng(11).permutation(31)
    inv = np.argsort(perm)
    lp0, lse0, ent0 = oracle.forward(X, W, y)
    lp1, lse1, ent1 = oracle.forward(X, W[perm], inv[y])
    np.testing.assert_allclose(lp1, lp0, atol=1e-12)
    np.testing.assert_allclose(lse1, lse0, atol=1e-12)
    np.testing.assert_allclose(ent1, ent0, atol=1e-12)


def test_one_hot_dominant_row():
    V = 20
    X = np.array([[1.0]])
    W = np.zeros((V, 1))
    W[4, 0] = 200.0
    lp, lse, ent = oracle.forward(X, W, np.array([4]))
    assert abs(lp[0]) < 1e-70 and abs(ent[0]) < 1e-70 and abs(lse[0] - 200.0) < 1e-12
    lp, _, _ = oracle.forward(X, W, np.array([3]))
    np.testing.assert_allclose(lp[0], -200.0, atol=1e-9)


def test_brute_force_pure_python():
    # Naive log-softmax without any max shift, written with Python floats and
    # explicit loops (no numpy, no C): logits of moderate size so exp() is safe.
    M, H, V = 4, 5, 9
    X, W, y = rand_case(12, M, H, V, ws=0.6)
    s = 1.25
    y[2] = -100
    lp, lse, ent = oracle.forward(X, W, y, scale=s)
    for i in range(M):
        z = []
        for j in range(V):
            acc = 0.0
            for k in range(H):
                acc += float(X[i, k]) * float(W[j, k])
            z.append(s * acc)
        total = sum(math.exp(v) for v in z)
        want_lse = math.log(total)
        probs = [math.exp(v) / total for v in z]
        want_ent = -sum(p * math.log(p) for p in probs)
        assert abs(lse[i] - want_lse) < 1e-12
        if y[i] == -100:
            assert lp[i] == 0.0 and ent[i] == 0.0
        else:
            assert abs(lp[i] - math.log(probs[y[i]])) < 1e-12
            assert abs(ent[i] - want_ent) < 1e-12


def test_bf16_entry_matches_widened_f64():
    X, W, y = rand_case(13, 9, 24, 40)
    Xb, Wb = to_bf16_bits(X), to_bf16_bits(W)
    # numpy's own widening, independent of the C conversion
    Xw = (Xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Ww = (Wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    a = oracle.forward(Xb, Wb, y, scale=0.9)
    b = oracle.forward(Xw, Ww, y, scale=0.9)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)
    ga, gb = rng(14).normal(size=9), rng(15).normal(size=9)
    da = oracle.backward(Xb, Wb, y, ga, gb, scale=0.9)
    db = oracle.backward(Xw, Ww, y, ga, gb, scale=0.9)
    for u, v in zip(da, db):
        np.testing.assert_array_equal(u, v)


def test_ignored_and_bad_targets():
    X, W, y = rand_case(16, 6, 8, 10)
    y[1] = -100
    y[3] = 10  # out of range, not ignore_index
    with pytest.raises(oracle.OracleError):
        oracle.forward(X, W, y)
    lp, lse, ent = oracle.forward(X, W, y, allow_bad_target=True)
    assert lp[1] == 0.0 and ent[1] == 0.0 and np.isfinite(lse[1])
    assert math.isnan(lp[3])
    # a custom ignore_index
    y2 = y.copy()
    y2[3] = 7
    y2[1] = 5
    lp2, _, ent2 = oracle.forward(X, W, y2, ignore_index=5)
    assert lp2[1] == 0.0 and ent2[1] == 0.0


def test_row_subset_matches_full():
    X, W, y = rand_case(17, 30, 6, 25)
    full = oracle.forward(X, W, y)
    rows = np.array([29, 0, 13, 13, 7])
    sub = oracle.forward(X, W, y, rows=rows)
    for f, s in zip(full, sub):
        np.testing.assert_array_equal(f[rows], s)


# -------------------------------------------------------------------- backward

def _loss(X, W, y, g_lp, g_ent, s, ent_on):
    lp, _, ent = oracle.forward(X, W, y, scale=s, compute_entropy=ent_on)
    total = float(np.dot(g_lp, lp))
    if ent_on:
        total += float(np.dot(g_ent, ent))
    return total


@pytest.mark.parametrize("ent_on", [True, False])
def test_backward_matches_finite_differences(ent_on):
    M, H, V = 5, 6, 11
    X, W, y = rand_case(18, M, H, V, ws=0.8)
    y[3] = -100
    s = 1.4
    g_lp = rng(19).normal(size=M)
    g_ent = rng(20).normal(size=M)
    dX, dW = oracle.backward(X, W, y, g_lp, g_ent, scale=s, compute_entropy=ent_on)
    eps = 1e-6
    num_dX = np.zeros_like(X)
    for i in range(M):
        for k in range(H):
            Xp, Xm = X.copy(), X.copy()
            Xp[i, k] += eps
            Xm[i, k] -= eps
            num_dX[i, k] = (_loss(Xp, W, y, g_lp, g_ent, s, ent_on)
                            - _loss(Xm, W, y, g_lp, g_ent, s, ent_on)) / (2 * eps)
    num_dW = np.zeros_like(W)
    for j in range(V):
        for k in range(H):
            Wp, Wm = W.copy(), W.copy()
            Wp[j, k] += eps
            Wm[j, k] -= eps
            num_dW[j, k] = (_loss(X, Wp, y, g_lp, g_ent, s, ent_on)
                            - _loss(X, Wm, y, g_lp, g_ent, s, ent_on)) / (2 * eps)
    np.testing.assert_allclose(dX, num_dX, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dW, num_dW, rtol=1e-6, atol=1e-8)
    assert np.all(dX[3] == 0.0)


def test_backward_invariants():
    M, H, V = 12, 8, 33
    X, W, y = rand_case(21, M, H, V)
    y[[2, 7]] = -100
    g_lp = rng(22).normal(size=M)
    g_ent = rng(23).normal(size=M)
    dX, dW = oracle.backward(X, W, y, g_lp, g_ent, scale=0.6)
    # every dZ row sums to zero, so the columns of dW sum to zero
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-12)
    assert np.all(dX[[2, 7]] == 0.0)
    # zero upstream gradients give zero gradients
    z1, z2 = oracle.backward(X, W, y, np.zeros(M), np.zeros(M))
    assert not z1.any() and not z2.any()
    z1, z2 = oracle.backward(X, W, y, None, None)
    assert not z1.any() and not z2.any()
    # entropy gradient vanishes at uniform logits
    e1, e2 = oracle.backward(X, np.zeros_like(W), y, np.zeros(M), np.ones(M))
    np.testing.assert_allclose(e1, 0.0, atol=1e-15)
    np.testing.assert_allclose(e2, 0.0, atol=1e-15)


def test_backward_row_subset_and_linearity():
    M, H, V = 10, 5, 17
    X, W, y = rand_case(24, M, H, V)
    g_lp = rng(25).normal(size=M)
    g_ent = rng(26).normal(size=M)
    rows = np.array([1, 4, 8])
    dx_s, dw_s = oracle.backward(X, W, y, g_lp, g_ent, rows=rows)
    mask = np.zeros(M)
    mask[rows] = 1
    dx_f, dw_f = oracle.backward(X, W, y, g_lp * mask, g_ent * mask)
    np.testing.assert_allclose(dx_s, dx_f[rows], atol=1e-14)
    np.testing.assert_allclose(dw_s, dw_f, atol=1e-14)


def test_round_dz_bf16_is_small_perturbation():
    M, H, V = 8, 16, 64
    X, W, y = rand_case(27, M, H, V)
    g = rng(28).normal(size=M)
    dx0, dw0 = oracle.backward(X, W, y, g, g)
    dx1, dw1 = oracle.backward(X, W, y, g, g, round_dz_bf16=True)
    rel = np.linalg.norm(dw1 - dw0) / np.linalg.norm(dw0)
    assert 0 < rel < 2 ** -8
    rel = np.linalg.norm(dx1 - dx0) / np.linalg.norm(dx0)
    assert 0 < rel < 2 ** -8


# ------------------------------------------------- bf16 rounding of dZ, bit for bit

def _f32(bits):
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


@pytest.mark.parametrize("bits,want", [
    (0x3F800000, 0x3F80),  # 1.0, exact
    (0x3F808000, 0x3F80),  # tie, the lower neighbour is even: stays
    (0x3F818000, 0x3F82),  # tie, the lower neighbour is odd: rounds up to even
    (0x3F808001, 0x3F81),  # just above a tie: up
    (0x3F807FFF, 0x3F80),  # just below a tie: down
    (0xBF808000, 0xBF80),  # negative tie to even (magnitude rounds down)
    (0xBF818000, 0xBF82),  # negative tie to even (magnitude rounds up)
    (0xBF80C000, 0xBF81),  # negative, above the tie in magnitude
    (0x7F7F8000, 0x7F80),  # tie between the largest finite bf16 (odd) and +inf: +inf
    (0x7F7FFFFF, 0x7F80),  # the largest binary32 overflows to +inf
    (0x7F7F7FFF, 0x7F7F),  # below that tie: the largest finite bf16
    (0xFF7FFFFF, 0xFF80),  # ... and to -inf
    (0x7F800000, 0x7F80),  # +inf
    (0xFF800000, 0xFF80),  # -inf
    (0x00000000, 0x0000),  # +0
    (0x80000000, 0x8000),  # -0
    (0x00008000, 0x0000),  # subnormal tie to even (zero)
    (0x00018000, 0x0002),  # subnormal tie to even (up)
    (0x007FFFFF, 0x0080),  # largest subnormal rounds up to the smallest normal
])
def test_oracle_bf16_rounding_exact_bits(bits, want):
    """Round to nearest, ties to even (IEEE 754 roundTiesToEven applied at the
    bf16 precision: 8 significand bits); the expected patterns follow from
    that rule by hand."""
    got = int(oracle.round_bf16(np.array([_f32(bits)]))[0])
    assert got == want, f"{bits:#010x}: got {got:#06x}, want {want:#06x}"


@pytest.mark.parametrize("bits", [0x7FC00000, 0x7F800001, 0xFFC00001, 0x7FBFFFFF])
def test_oracle_bf16_rounding_keeps_nan(bits):
    """A NaN stays a NaN (a quiet one): a signalling NaN whose payload sits in
    the low half must not turn into an infinity."""
    got = int(oracle.round_bf16(np.array([_f32(bits)]))[0])
    assert (got & 0x7F80) == 0x7F80 and (got & 0x007F) != 0, f"{bits:#010x} -> {got:#06x}"
    assert (got & 0x8000) == (bits >> 16 & 0x8000)


def test_oracle_bf16_rounding_matches_torch_on_random_patterns():
    """torch's float32 -> bfloat16 conversion is round-to-nearest-even; on a
    million random non-NaN bit patterns (every exponent, both signs) and on
    every tie pattern of a few exponents the oracle agrees bit for bit."""
    import torch
    r = rng(99)
    bits = r.integers(0, 2**32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    ties = ((np.arange(0, 2**16, dtype=np.uint32) << 16) | 0x8000)
    bits = np.concatenate([bits, ties, ties - 1, ties + 1])
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(f)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} mismatches, first {f.view(np.uint32)[bad[0]]:#010x}"


def test_round_dz_bf16_rounds_each_dz_entry_before_the_contractions():
    """With H = 1 and X = 1, dW[j] is dZ[0, j] itself, so the rounding mode
    shows up unmixed: dW[j] = bf16(fp32(dZ_j)) with dZ from the closed form of
    a two-class row (logistic): p_1 = 1 / (1 + e^{z_0 - z_1})."""
    import torch
    s, g = 1.0, 1.0
    X = np.ones((1, 1))
    for z0, z1 in ((0.3, -1.7), (2.0, 2.0 + 1e-3), (-0.123456, 0.5)):
        W = np.array([[z0], [z1]])
        y = np.array([0])
        p1 = 1.0 / (1.0 + math.exp(z0 - z1))
        dz = np.array([s * g * (1.0 - (1.0 - p1)), s * g * (0.0 - p1)])  # onehot - p
        want = torch.from_numpy(dz.astype(np.float32)).to(torch.bfloat16).double().numpy()
        _, dw = oracle.backward(X, W, y, np.array([g]), None, compute_entropy=False, scale=s,
                                round_dz_bf16=True)
        np.testing.assert_array_equal(dw[:, 0], want)
        _, dw0 = oracle.backward(X, W, y, np.array([g]), None, compute_entropy=False, scale=s)
        np.testing.assert_allclose(dw0[:, 0], dz, rtol=1e-15, atol=1e-17)


# ------------------------------------------- dW on selected vocabulary rows

@pytest.mark.parametrize("rnd", [False, True])
def test_backward_dw_cols_equals_the_full_backward_rows(rnd):
    """The sampled-vocabulary dW (every row's gradient live) equals the rows
    of the full backward's dW, which the finite-difference pins above tie to
    the forward; also with an ignored row, s != 1 and entropy on."""
    M, H, V = 13, 7, 41
    X, W, y = rand_case(40, M, H, V)
    y[[3, 9]] = -100
    g_lp = rng(41).normal(size=M)
    g_ent = rng(42).normal(size=M)
    cols = np.array([0, 5, 17, 40, 17])
    _, dw = oracle.backward(X, W, y, g_lp, g_ent, scale=0.8, round_dz_bf16=rnd)
    got = oracle.backward_dw_cols(X, W, y, g_lp, g_ent, cols, scale=0.8, round_dz_bf16=rnd)
    np.testing.assert_allclose(got, dw[cols], rtol=1e-13, atol=1e-15)
    # bf16 inputs take the same path as their exact fp64 widening
    Xb, Wb = to_bf16_bits(X), to_bf16_bits(W)
    got_b = oracle.backward_dw_cols(Xb, Wb, y, g_lp, None, cols, compute_entropy=False)
    _, dw_b = oracle.backward(oracle.bf16_bits_to_f64(Xb), oracle.bf16_bits_to_f64(Wb), y, g_lp,
                              None, compute_entropy=False)
    np.testing.assert_allclose(got_b, dw_b[cols], rtol=1e-13, atol=1e-15)


def test_backward_dw_cols_forward_outputs_equal_the_forward():
    """The per-row forward outputs the dW-columns entry returns are those of
    the pinned forward, bit for bit (same definitions, same logit rows)."""
    M, H, V = 11, 6, 29
    X, W, y = rand_case(43, M, H, V)
    y[4] = -100
    g = rng(44).normal(size=M)
    for ent in (True, False):
        _, lp, lse, en = oracle.backward_dw_cols(X, W, y, g, g, [1, 2], scale=1.7,
                                                 compute_entropy=ent, with_forward=True)
        f_lp, f_lse, f_en = oracle.forward(X, W, y, scale=1.7, compute_entropy=ent)
        np.testing.assert_array_equal(lp, f_lp)
        np.testing.assert_array_equal(lse, f_lse)
        if ent:
            np.testing.assert_array_equal(en, f_en)
        else:
            assert en is None
