"""Pins for the oracle's index projections and dense indexer warm-up (CPU).

"Sparse Attention · Part II": section 3.2's detachment equation
(Q_idx = stopgrad(X) W_q^idx, K_idx = stopgrad(X) W_k^idx) and section
3.1's dense warm-up loss, in MSA's per-group form (section 3.2 follows the
warm-up with the same KL restricted to the selected blocks).  Each pin checks
the oracle against something other than itself: one-hot inputs, the
adjoint identity of a linear map, the block-sparse KL with every visible
block selected (a different formulation: blocks, selection and token sets),
scipy's relative entropy, a built teacher == student case, and central
finite differences through the projections.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
from block_sparse_gqa_causal_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits


def rnd_bf16(rng, shape):
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))


def widen(a):
    return bf16_bits_to_f32(a).astype(np.float64)


def test_projection_of_one_hot_rows_is_the_weight_rows():
    """X with a single 1 in column m of row t gives row m of W_q (split into
    the groups' index queries) and row m of W_k: catches a transposed
    weight or a wrong group stride."""
    rng = np.random.default_rng(0)
    T, Dm, Hkv, di = 7, 12, 3, 4
    one = f32_to_bf16_bits(np.float32(1.0))
    X = np.zeros((T, Dm), dtype=np.uint16)
    cols = rng.choice(Dm, size=T, replace=True)
    X[np.arange(T), cols] = one
    Wq, Wk = rnd_bf16(rng, (Dm, Hkv * di)), rnd_bf16(rng, (Dm, di))
    qi, ki = oracle.index_proj(X, Wq, Wk, Hkv, di)
    np.testing.assert_array_equal(qi, widen(Wq)[cols])
    np.testing.assert_array_equal(ki, widen(Wk)[cols])


def test_projection_is_linear_in_x():
    rng = np.random.default_rng(1)
    T, Dm, Hkv, di = 9, 10, 2, 5
    X1, X2 = rng.standard_normal((T, Dm)), rng.standard_normal((T, Dm))
    Wq, Wk = rng.standard_normal((Dm, Hkv * di)), rng.standard_normal((Dm, di))
    a, b = 0.7, -1.9
    q1, k1 = oracle.index_proj(X1, Wq, Wk, Hkv, di)
    q2, k2 = oracle.index_proj(X2, Wq, Wk, Hkv, di)
    q3, k3 = oracle.index_proj(a * X1 + b * X2, Wq, Wk, Hkv, di)
    np.testing.assert_allclose(q3, a * q1 + b * q2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(k3, a * k1 + b * k2, rtol=1e-12, atol=1e-12)


def test_weight_gradient_satisfies_the_adjoint_identity():
    """<dY, X W> = <X^T dY, W> for random W, separately for the query and key
    projections: the weight gradient is the adjoint of the forward map."""
    rng = np.random.default_rng(2)
    T, Dm, Hkv, di = 11, 6, 2, 3
    X = rng.standard_normal((T, Dm))
    Wq, Wk = rng.standard_normal((Dm, Hkv * di)), rng.standard_normal((Dm, di))
    dq, dk = rng.standard_normal((T, Hkv * di)), rng.standard_normal((T, di))
    qi, ki = oracle.index_proj(X, Wq, Wk, Hkv, di)
    dWq, dWk = oracle.index_proj_bwd(X, dq, dk, Hkv, di)
    assert np.sum(dq * qi) == pytest.approx(np.sum(dWq * Wq), rel=1e-12)
    assert np.sum(dk * ki) == pytest.approx(np.sum(dWk * Wk), rel=1e-12)
    assert dWq.shape == (Dm, Hkv * di) and dWk.shape == (Dm, di)


def _dense_case(rng, B=1, N=200, Hq=4, Hkv=2, d=16, di=16, block=32):
    sh = oracle.Shape(B=B, Nq=N, Nk=N, Hq=Hq, Hkv=Hkv, d=d, d_idx=di, topk=(N + block - 1) // block, block=block)
    q = rnd_bf16(rng, (B, N, Hq, d))
    k = rnd_bf16(rng, (B, N, Hkv, d))
    qi = rnd_bf16(rng, (B, N, Hkv, di))
    ki = rnd_bf16(rng, (B, N, di))
    return sh, q, k, qi, ki


def test_warmup_kl_equals_block_sparse_kl_with_every_block_selected():
    """With k >= the number of blocks every visible block is selected, so the
    block-sparse KL (blocks, selection, token sets) is the dense warm-up KL."""
    rng = np.random.default_rng(3)
    sh, q, k, qi, ki = _dense_case(rng, B=2, N=150)
    lse_w, kl_w = oracle.warmup_kl(sh, q, k, qi, ki)
    sel = oracle.select(sh, oracle.block_scores(sh, qi, ki))
    lse_s, kl_s = oracle.kl(sh, q, k, qi, ki, sel)
    np.testing.assert_allclose(kl_w, kl_s, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse_w, lse_s, rtol=1e-12, atol=1e-12)


def test_warmup_kl_matches_scipy_relative_entropy_over_the_prefix():
    rng = np.random.default_rng(4)
    sh, q, k, qi, ki = _dense_case(rng, N=90)
    lse_w, kl_w = oracle.warmup_kl(sh, q, k, qi, ki)
    assert np.all(kl_w >= -1e-15)
    G = sh.Hq // sh.Hkv
    qf, kf, qif, kif = widen(q)[0], widen(k)[0], widen(qi)[0], widen(ki)[0]
    causal = np.tril(np.ones((sh.Nq, sh.Nk), dtype=bool))
    for r in range(sh.Hkv):
        pt = 0.0
        for g in range(G):
            lg = qf[:, r * G + g] @ kf[:, r].T / math.sqrt(sh.d)
            pt = pt + scipy.special.softmax(np.where(causal, lg, -np.inf), axis=-1) / G
        s = np.where(causal, qif[:, r] @ kif.T / math.sqrt(sh.d_idx), -np.inf)
        want = scipy.special.rel_entr(pt, scipy.special.softmax(s, axis=-1)).sum(-1)
        np.testing.assert_allclose(kl_w[:, r], want, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(lse_w[:, r], scipy.special.logsumexp(s, axis=-1), rtol=1e-12)


def test_warmup_kl_is_zero_when_teacher_equals_student():
    rng = np.random.default_rng(5)
    N = 70
    sh = oracle.Shape(B=1, Nq=N, Nk=N, Hq=3, Hkv=1, d=8, d_idx=8, topk=3, block=32)
    qi = rnd_bf16(rng, (1, N, 1, 8))
    ki = rnd_bf16(rng, (1, N, 8))
    q = np.repeat(qi, 3, axis=2)
    k = ki[:, :, None, :].copy()
    _, kl_w = oracle.warmup_kl(sh, q, k, qi, ki)
    assert np.max(np.abs(kl_w)) < 1e-12


def _f64_warmup_case(seed=6):
    rng = np.random.default_rng(seed)
    T, Dm, Hq, Hkv, d, di = 40, 12, 4, 2, 8, 8
    sh = oracle.Shape(B=1, Nq=T, Nk=T, Hq=Hq, Hkv=Hkv, d=d, d_idx=di, topk=3, block=16)
    X = rng.standard_normal((T, Dm))
    Wq, Wk = rng.standard_normal((Dm, Hkv * di)) * 0.4, rng.standard_normal((Dm, di)) * 0.4
    q, k = rng.standard_normal((1, T, Hq, d)), rng.standard_normal((1, T, Hkv, d))
    return sh, X, Wq, Wk, q, k


def _warm_loss(sh, X, Wq, Wk, q, k, coef):
    qi, ki = oracle.index_proj(X, Wq, Wk, sh.Hkv, sh.d_idx)
    _, kl_w = oracle.warmup_kl(sh, q, k, qi.reshape(1, sh.Nq, sh.Hkv, sh.d_idx), ki.reshape(1, sh.Nk, sh.d_idx))
    return oracle.kl_loss(sh, kl_w, coef)


def test_warmup_gradient_matches_finite_differences_in_the_index_inputs():
    sh, X, Wq, Wk, q, k = _f64_warmup_case()
    coef = 0.9
    qi, ki = oracle.index_proj(X, Wq, Wk, sh.Hkv, sh.d_idx)
    qi, ki = qi.reshape(1, sh.Nq, sh.Hkv, sh.d_idx), ki.reshape(1, sh.Nk, sh.d_idx)
    dqi, dki = oracle.warmup_grad(sh, q, k, qi, ki, coef)

    def loss(qi_, ki_):
        return oracle.kl_loss(sh, oracle.warmup_kl(sh, q, k, qi_, ki_)[1], coef)

    rng = np.random.default_rng(7)
    h = 1e-5
    for name, x, g, f in (("q_idx", qi, dqi, lambda a: loss(a, ki)), ("k_idx", ki, dki, lambda a: loss(qi, a))):
        for flat in rng.choice(x.size, size=25, replace=False):
            xp, xm = x.copy(), x.copy()
            xp.flat[flat] += h
            xm.flat[flat] -= h
            fd = (f(xp) - f(xm)) / (2 * h)
            assert abs(fd - g.flat[flat]) <= 1e-8 + 1e-5 * abs(fd), (name, flat, fd, g.flat[flat])


def test_weight_gradient_of_the_warmup_loss_matches_finite_differences_in_w():
    """d L_warm / dW through the detached projections: the warm-up gradient in
    the index inputs chained by the projection's weight gradient equals
    central differences of the loss in the weights."""
    sh, X, Wq, Wk, q, k = _f64_warmup_case(seed=8)
    coef = 1.3
    qi, ki = oracle.index_proj(X, Wq, Wk, sh.Hkv, sh.d_idx)
    dqi, dki = oracle.warmup_grad(sh, q, k, qi.reshape(1, sh.Nq, sh.Hkv, sh.d_idx),
                                  ki.reshape(1, sh.Nk, sh.d_idx), coef)
    dWq, dWk = oracle.index_proj_bwd(X, dqi, dki, sh.Hkv, sh.d_idx)
    rng = np.random.default_rng(9)
    h = 1e-5
    for name, W, g in (("Wq", Wq, dWq), ("Wk", Wk, dWk)):
        for flat in rng.choice(W.size, size=20, replace=False):
            Wp, Wm = W.copy(), W.copy()
            Wp.flat[flat] += h
            Wm.flat[flat] -= h
            if name == "Wq":
                fd = (_warm_loss(sh, X, Wp, Wk, q, k, coef) - _warm_loss(sh, X, Wm, Wk, q, k, coef)) / (2 * h)
            else:
                fd = (_warm_loss(sh, X, Wq, Wp, q, k, coef) - _warm_loss(sh, X, Wq, Wm, q, k, coef)) / (2 * h)
            assert abs(fd - g.flat[flat]) <= 1e-8 + 1e-5 * abs(fd), (name, flat, fd, g.flat[flat])


def test_warmup_gradient_sees_the_teacher_only_through_its_probabilities():
    """The teacher is detached: the gradient the warm-up sends into the index
    inputs is unchanged when q and k (the teacher's inputs) are rescaled so
    that the main logits, hence the teacher, stay the same."""
    sh, X, Wq, Wk, q, k = _f64_warmup_case(seed=10)
    qi, ki = oracle.index_proj(X, Wq, Wk, sh.Hkv, sh.d_idx)
    qi, ki = qi.reshape(1, sh.Nq, sh.Hkv, sh.d_idx), ki.reshape(1, sh.Nk, sh.d_idx)
    g1 = oracle.warmup_grad(sh, q, k, qi, ki, 1.0)
    # scale q by 2 and k by 1/2: the main logits, hence the teacher, are unchanged
    g2 = oracle.warmup_grad(sh, 2.0 * q, 0.5 * k, qi, ki, 1.0)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)
