"""Pins for the CPU oracle: each test checks the oracle against something
other than itself (brute force, a textbook or library routine, an
invariant the method fixes, or finite differences).  CPU only.

The method: "Sparse Attention · Part II", section 3.2 (MiniMax's MSA).
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


def make(rng, sh: oracle.Shape, nq_rows=None):
    q = rnd_bf16(rng, (sh.B, sh.Nq, sh.Hq, sh.d))
    k = rnd_bf16(rng, (sh.B, sh.Nk, sh.Hkv, sh.d))
    v = rnd_bf16(rng, (sh.B, sh.Nk, sh.Hkv, sh.d))
    qi = rnd_bf16(rng, (sh.B, sh.Nq, sh.Hkv, sh.d_idx))
    ki = rnd_bf16(rng, (sh.B, sh.Nk, sh.d_idx))
    do = rnd_bf16(rng, (sh.B, sh.Nq, sh.Hq, sh.d))
    return q, k, v, qi, ki, do


def positions(sh):
    return sh.q_offset + np.arange(sh.Nq)


# ----------------------------------------------------------------- numpy refs
def np_token_scores(sh, qi, ki):
    """[B, Hkv, Nq, Nk] fp64 index scores, -inf where not causally visible."""
    s = np.einsum("bird,bjd->brij", widen(qi), widen(ki)[:, : sh.Nk]) * (1.0 / math.sqrt(sh.d_idx))
    vis = np.arange(sh.Nk)[None, :] <= positions(sh)[:, None]
    return np.where(vis[None, None], s, -np.inf)


def np_block_mask(sh, sel_full):
    """allowed[b, r, i, j]: j visible and its block selected."""
    blk = np.arange(sh.Nk) // sh.block
    chosen = (sel_full[..., None] == blk[None, None, None, None, :]).any(axis=3)  # [B,Hkv,Nq,Nk]
    vis = np.arange(sh.Nk)[None, :] <= positions(sh)[:, None]
    return chosen & vis[None, None]


def np_attention(sh, q, k, v, allowed):
    """Dense softmax attention with a boolean mask [B,Hkv,Nq,Nk]; O, LSE."""
    G = sh.Hq // sh.Hkv
    qf, kf, vf = widen(q), widen(k), widen(v)
    o = np.zeros((sh.B, sh.Nq, sh.Hq, sh.d))
    lse = np.zeros((sh.B, sh.Nq, sh.Hq))
    for h in range(sh.Hq):
        r = h // G
        lg = np.einsum("bid,bjd->bij", qf[:, :, h], kf[:, :, r]) / math.sqrt(sh.d)
        lg = np.where(allowed[:, r], lg, -np.inf)
        lse[:, :, h] = scipy.special.logsumexp(lg, axis=-1)
        p = scipy.special.softmax(lg, axis=-1)
        o[:, :, h] = np.einsum("bij,bjd->bid", p, vf[:, :, r])
    return o, lse


# ------------------------------------------------------------------ a1 / a2
@pytest.mark.parametrize("q_offset,nq,nk", [(0, 300, 300), (0, 256, 256), (509, 3, 512)])
def test_block_scores_match_bruteforce(q_offset, nq, nk):
    rng = np.random.default_rng(11)
    sh = oracle.Shape(B=2, Nq=nq, Nk=nk, Hq=4, Hkv=2, d=8, d_idx=16, topk=3, block=32, q_offset=q_offset)
    _, _, _, qi, ki, _ = make(rng, sh)
    got = oracle.block_scores(sh, qi, ki)                       # [B*Nq, Hkv, nb]
    s = np_token_scores(sh, qi, ki)                               # [B,Hkv,Nq,Nk]
    pad = sh.nb * sh.block - sh.Nk
    s = np.concatenate([s, np.full(s.shape[:-1] + (pad,), -np.inf)], axis=-1)
    want = s.reshape(s.shape[:-1] + (sh.nb, sh.block)).max(-1).astype(np.float32)
    want = want.transpose(0, 2, 1, 3).reshape(sh.B * sh.Nq, sh.Hkv, sh.nb)
    fin = np.isfinite(want)
    assert np.array_equal(fin, np.isfinite(got))
    np.testing.assert_allclose(got[fin], want[fin], rtol=1e-6, atol=1e-6)


# ----------------------------------------------------------------------- a3
def bruteforce_select(sh, bs_rows, rows):
    out = np.full((len(rows), sh.Hkv, sh.topk), -1, dtype=np.int32)
    for t, row in enumerate(rows):
        pos = sh.q_offset + row % sh.Nq
        c0 = pos // sh.block
        for r in range(sh.Hkv):
            if c0 + 1 <= sh.topk:
                ch = list(range(c0 + 1))
            else:
                order = sorted(range(c0), key=lambda c: (-float(bs_rows[t, r, c]), c))
                ch = sorted(order[: sh.topk - 1] + [c0])
            out[t, r, : len(ch)] = ch
    return out


@pytest.mark.parametrize("levels", [None, 3])
def test_select_matches_full_sort_and_invariants(levels):
    rng = np.random.default_rng(5)
    sh = oracle.Shape(B=2, Nq=200, Nk=200, Hq=2, Hkv=2, d=8, d_idx=8, topk=4, block=8)
    bs = rng.standard_normal((sh.B * sh.Nq, sh.Hkv, sh.nb)).astype(np.float32)
    if levels:  # many exact ties: the lower block index must win
        bs = np.floor(bs * levels).astype(np.float32)
    rows = np.arange(sh.B * sh.Nq)
    got = oracle.select(sh, bs, rows)
    assert np.array_equal(got, bruteforce_select(sh, bs, rows))
    for t, row in enumerate(rows):
        c0 = (row % sh.Nq) // sh.block
        for r in range(sh.Hkv):
            s = got[t, r]
            valid = s[s >= 0]
            assert c0 in valid                                   # local block always kept
            assert len(valid) == min(sh.topk, c0 + 1)
            assert np.all(valid <= c0) and np.all(np.diff(valid) > 0)
            assert np.all(s[len(valid):] == -1)


def test_select_prefers_lower_index_on_ties():
    sh = oracle.Shape(B=1, Nq=1, Nk=80, Hq=1, Hkv=1, d=8, d_idx=8, topk=3, block=8, q_offset=79)
    bs = np.zeros((1, 1, sh.nb), dtype=np.float32)
    bs[0, 0, [2, 5, 7]] = 1.0      # three-way tie for 2 free slots
    got = oracle.select(sh, bs, np.array([0]))
    assert got[0, 0].tolist() == [2, 5, 9]


# ----------------------------------------------------------------------- a4
def test_fwd_with_every_block_is_dense_causal_gqa():
    rng = np.random.default_rng(7)
    sh = oracle.Shape(B=2, Nq=96, Nk=96, Hq=6, Hkv=2, d=16, d_idx=8, topk=8, block=16)  # nb = 6 <= k
    q, k, v, qi, ki, _ = make(rng, sh)
    bs = oracle.block_scores(sh, qi, ki)
    sel_rows = oracle.select(sh, bs)
    o, lse = oracle.sparse_fwd(sh, q, k, v, sel_rows)
    vis = np.arange(sh.Nk)[None, :] <= positions(sh)[:, None]
    o_ref, lse_ref = np_attention(sh, q, k, v, np.broadcast_to(vis, (sh.B, sh.Hkv, sh.Nq, sh.Nk)))
    np.testing.assert_allclose(o.reshape(o_ref.shape), o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(lse_ref.shape), lse_ref, rtol=1e-12, atol=1e-12)


def _sparse_case(seed=3, q_offset=0, nq=160, nk=160):
    rng = np.random.default_rng(seed)
    sh = oracle.Shape(B=2, Nq=nq, Nk=nk, Hq=4, Hkv=2, d=16, d_idx=16, topk=3, block=16, q_offset=q_offset)
    q, k, v, qi, ki, do = make(rng, sh)
    bs = oracle.block_scores(sh, qi, ki)
    sel_rows = oracle.select(sh, bs)
    return sh, (q, k, v, qi, ki, do), sel_rows


@pytest.mark.parametrize("q_offset,nq,nk", [(0, 160, 160), (150, 10, 160)])
def test_fwd_equals_dense_attention_under_block_mask(q_offset, nq, nk):
    sh, (q, k, v, qi, ki, _), sel_rows = _sparse_case(q_offset=q_offset, nq=nq, nk=nk)
    o, lse = oracle.sparse_fwd(sh, q, k, v, sel_rows)
    allowed = np_block_mask(sh, oracle.sel_full_from_rows(sh, sel_rows))
    o_ref, lse_ref = np_attention(sh, q, k, v, allowed)
    np.testing.assert_allclose(o.reshape(o_ref.shape), o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(lse_ref.shape), lse_ref, rtol=1e-12, atol=1e-12)


def test_fwd_within_renormalisation_error_bound():
    """||o - o_sparse|| <= 2 B delta, delta = dense softmax mass dropped,
    B = max value norm (section 2 of the same page)."""
    sh, (q, k, v, qi, ki, _), sel_rows = _sparse_case(seed=9)
    o, _ = oracle.sparse_fwd(sh, q, k, v, sel_rows)
    o = o.reshape(sh.B, sh.Nq, sh.Hq, sh.d)
    vis = np.arange(sh.Nk)[None, :] <= positions(sh)[:, None]
    o_dense, lse_dense = np_attention(sh, q, k, v, np.broadcast_to(vis, (sh.B, sh.Hkv, sh.Nq, sh.Nk)))
    allowed = np_block_mask(sh, oracle.sel_full_from_rows(sh, sel_rows))
    G = sh.Hq // sh.Hkv
    qf, kf, vf = widen(q), widen(k), widen(v)
    for h in range(sh.Hq):
        r = h // G
        lg = np.einsum("bid,bjd->bij", qf[:, :, h], kf[:, :, r]) / math.sqrt(sh.d)
        p = np.where(vis[None], np.exp(lg - lse_dense[:, :, h, None]), 0.0)
        delta = np.where(allowed[:, r], 0.0, p).sum(-1)
        bound = 2 * np.linalg.norm(vf[:, :, r], axis=-1).max(axis=1)[:, None] * delta
        err = np.linalg.norm(o[:, :, h] - o_dense[:, :, h], axis=-1)
        assert np.all(err <= bound + 1e-12)


# ----------------------------------------------------------------------- a5
def test_kl_nonnegative_and_matches_scipy_relative_entropy():
    sh, (q, k, v, qi, ki, _), sel_rows = _sparse_case(seed=4)
    lse_idx, klr = oracle.kl(sh, q, k, qi, ki, sel_rows)
    assert np.all(klr >= -1e-15)
    allowed = np_block_mask(sh, oracle.sel_full_from_rows(sh, sel_rows))
    G = sh.Hq // sh.Hkv
    qf, kf = widen(q), widen(k)
    s = np_token_scores(sh, qi, ki)
    for r in range(sh.Hkv):
        pt = 0.0
        for g in range(G):
            lg = np.einsum("bid,bjd->bij", qf[:, :, r * G + g], kf[:, :, r]) / math.sqrt(sh.d)
            pt = pt + scipy.special.softmax(np.where(allowed[:, r], lg, -np.inf), axis=-1) / G
        sr = np.where(allowed[:, r], s[:, r], -np.inf)
        ps = scipy.special.softmax(sr, axis=-1)
        want = scipy.special.rel_entr(pt, ps).sum(-1)               # [B, Nq]
        np.testing.assert_allclose(klr[:, r].reshape(sh.B, sh.Nq), want, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(lse_idx[:, r].reshape(sh.B, sh.Nq), scipy.special.logsumexp(sr, axis=-1),
                                   rtol=1e-12, atol=1e-12)


def test_kl_is_zero_when_teacher_equals_student():
    rng = np.random.default_rng(8)
    sh = oracle.Shape(B=1, Nq=64, Nk=64, Hq=3, Hkv=1, d=16, d_idx=16, topk=2, block=16)
    qi = rnd_bf16(rng, (1, sh.Nq, 1, 16))
    ki = rnd_bf16(rng, (1, sh.Nk, 16))
    q = np.repeat(qi, 3, axis=2)        # every head's query is the index query
    k = ki[:, :, None, :].copy()        # the main key is the index key
    sel_rows = oracle.select(sh, oracle.block_scores(sh, qi, ki))
    _, klr = oracle.kl(sh, q, k, qi, ki, sel_rows)
    assert np.max(np.abs(klr)) < 1e-12


# ----------------------------------------------------------------------- a6
def _f64_case(seed=21):
    rng = np.random.default_rng(seed)
    sh = oracle.Shape(B=1, Nq=48, Nk=48, Hq=4, Hkv=2, d=8, d_idx=8, topk=2, block=8)
    arrs = [rng.standard_normal(s) for s in ((1, 48, 4, 8), (1, 48, 2, 8), (1, 48, 2, 8), (1, 48, 2, 8),
                                             (1, 48, 8), (1, 48, 4, 8))]
    q, k, v, qi, ki, do = arrs
    bs = oracle.block_scores(sh, qi, ki)
    sel_rows = oracle.select(sh, bs)
    return sh, q, k, v, qi, ki, do, sel_rows


def test_bwd_matches_central_finite_differences():
    sh, q, k, v, qi, ki, do, sel_rows = _f64_case()
    sel_full = oracle.sel_full_from_rows(sh, sel_rows)
    coef = 0.7
    dq, dqi = oracle.bwd_rows(sh, q, k, v, do, qi, ki, sel_full, coef)
    dk, dv, dki = oracle.bwd_keys(sh, q, k, v, do, qi, ki, sel_full, coef)

    def main_loss(q_, k_, v_):
        o, _ = oracle.sparse_fwd(sh, q_, k_, v_, sel_rows)
        return float(np.sum(o * do.reshape(o.shape)))

    def kl_loss(qi_, ki_):
        _, klr = oracle.kl(sh, q, k, qi_, ki_, sel_rows)
        return oracle.kl_loss(sh, klr, coef)

    rng = np.random.default_rng(1)
    h = 1e-5
    checks = [("q", q, dq.reshape(q.shape), lambda a: main_loss(a, k, v)),
              ("k", k, dk, lambda a: main_loss(q, a, v)),
              ("v", v, dv, lambda a: main_loss(q, k, a)),
              ("q_idx", qi, dqi.reshape(qi.shape), lambda a: kl_loss(a, ki)),
              ("k_idx", ki, dki, lambda a: kl_loss(qi, a))]
    for name, x, g, f in checks:
        for flat in rng.choice(x.size, size=25, replace=False):
            xp, xm = x.copy(), x.copy()
            xp.flat[flat] += h
            xm.flat[flat] -= h
            fd = (f(xp) - f(xm)) / (2 * h)
            assert abs(fd - g.flat[flat]) <= 1e-6 + 1e-5 * abs(fd), (name, flat, fd, g.flat[flat])


def test_bwd_detachment_invariants():
    sh, q, k, v, qi, ki, do, sel_rows = _f64_case(seed=22)
    sel_full = oracle.sel_full_from_rows(sh, sel_rows)
    dq1, dqi1 = oracle.bwd_rows(sh, q, k, v, do, qi, ki, sel_full, 1.0)
    dq2, dqi2 = oracle.bwd_rows(sh, q, k, v, 3 * do, qi, ki, sel_full, 0.0)
    k1 = oracle.bwd_keys(sh, q, k, v, do, qi, ki, sel_full, 1.0)
    k2 = oracle.bwd_keys(sh, q, k, v, do, qi, ki, sel_full, 5.0)
    np.testing.assert_allclose(3 * dq1, dq2, rtol=1e-12, atol=1e-14)   # main grads ignore kl_coef
    assert np.all(dqi2 == 0)                                             # index grads ignore dO
    np.testing.assert_allclose(k1[0], k2[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(k1[1], k2[1], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(5 * k1[2], k2[2], rtol=1e-12, atol=1e-14)


def test_bwd_matches_torch_autograd_on_masked_dense_attention():
    torch = pytest.importorskip("torch")
    sh, q, k, v, qi, ki, do, sel_rows = _f64_case(seed=23)
    sel_full = oracle.sel_full_from_rows(sh, sel_rows)
    coef = 1.3
    dq, dqi = oracle.bwd_rows(sh, q, k, v, do, qi, ki, sel_full, coef)
    dk, dv, dki = oracle.bwd_keys(sh, q, k, v, do, qi, ki, sel_full, coef)

    allowed = torch.from_numpy(np_block_mask(sh, sel_full))            # [B,Hkv,Nq,Nk]
    G = sh.Hq // sh.Hkv
    T = {n: torch.tensor(a, dtype=torch.float64, requires_grad=True) for n, a in
         (("q", q), ("k", k), ("v", v), ("qi", qi), ("ki", ki))}
    kk = T["k"].repeat_interleave(G, dim=2)                               # [B,Nk,Hq,d]
    vv = T["v"].repeat_interleave(G, dim=2)
    lg = torch.einsum("bihd,bjhd->bhij", T["q"], kk) / math.sqrt(sh.d)
    mask = allowed.repeat_interleave(G, dim=1)
    p = torch.softmax(lg.masked_fill(~mask, float("-inf")), dim=-1)
    o = torch.einsum("bhij,bjhd->bihd", p, vv)
    loss_main = (o * torch.from_numpy(do)).sum()
    s = torch.einsum("bird,bjd->brij", T["qi"], T["ki"]) / math.sqrt(sh.d_idx)
    logps = torch.log_softmax(s.masked_fill(~allowed, float("-inf")), dim=-1)
    pt = p.detach().reshape(sh.B, sh.Hkv, G, sh.Nq, sh.Nk).mean(2)
    kl = torch.where(pt > 0, pt * (torch.log(pt.clamp_min(1e-300)) - logps), torch.zeros_like(pt)).sum(-1)
    loss = loss_main + coef * kl.sum() / (sh.B * sh.Nq * sh.Hkv)
    loss.backward()
    np.testing.assert_allclose(dq.reshape(q.shape), T["q"].grad.numpy(), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dk, T["k"].grad.numpy(), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dv, T["v"].grad.numpy(), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dqi.reshape(qi.shape), T["qi"].grad.numpy(), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dki, T["ki"].grad.numpy(), rtol=1e-9, atol=1e-12)


def test_bwd_keys_subset_equals_rows_of_full():
    sh, (q, k, v, qi, ki, do), sel_rows = _sparse_case(seed=6)
    sel_full = oracle.sel_full_from_rows(sh, sel_rows)
    full = oracle.bwd_keys(sh, q, k, v, do, qi, ki, sel_full)
    sub_blocks = np.array([0, 4, 9])
    sub = oracle.bwd_keys(sh, q, k, v, do, qi, ki, sel_full, kblocks=sub_blocks)
    idx = (sub_blocks[:, None] * sh.block + np.arange(sh.block)[None]).reshape(-1)
    for a, b in zip(full, sub):
        np.testing.assert_allclose(a[:, idx], b, rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------ input recipe
def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 1.0 + 2**-9], dtype=np.float32)
    assert f32_to_bf16_bits(x).tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F80]


def _golden(name):
    import os
    vals = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, val = line.split(":", 1)
            vals[key.strip()] = val.strip()
    return vals


def test_block_mask_worked_example():
    """The block-mask word printed for the first query block of section 4.3's
    figure: key tiles 0, 3, 6 active -> 01001001 = 73, walk visits 0, 3, 6."""
    g = _golden("block_mask_example.txt")
    nb = int(g["num_key_blocks"])
    active = [int(x) for x in g["active_blocks"].split()]
    sh = oracle.Shape(B=1, Nq=128, Nk=nb * 128, Hq=1, Hkv=1, d=16, d_idx=16, topk=2, q_offset=(nb - 1) * 128)
    sel = np.full((1, 1, 128, 2), -1, dtype=np.int32)
    sel[0, 0, 0] = [active[0], active[1]]          # two queries of the tile share the three blocks
    sel[0, 0, 77] = [active[2], -1]
    sel[0, 0, 5] = [active[1], -1]
    m = oracle.block_mask(sh, sel)
    assert m.shape == (1, 1, 1, 1)
    assert int(m[0, 0, 0, 0]) == int(g["word"])
    assert format(int(m[0, 0, 0, 0]) & 0xFF, "08b") == g["low_byte_binary"]
    walk = oracle.mask_walk(m[0, 0, 0])
    assert walk.tolist() == active and len(walk) == int(g["popcount"])


def test_block_mask_is_the_tile_union_and_walk_visits_it_in_order():
    """Brute force on random selections: per (b, group, 128-row tile), the walk
    of the mask words is the sorted union of the tile's selected blocks;
    padding (-1) and ids >= nb set nothing, so the last word's unused bits
    stay zero; an empty word is visited zero times."""
    rng = np.random.default_rng(8)
    for B, Nq, nk_blocks, Hkv, k in [(1, 300, 40, 2, 4), (2, 129, 64, 1, 3), (1, 1, 97, 3, 16)]:
        sh = oracle.Shape(B=B, Nq=Nq, Nk=nk_blocks * 128 - 5, Hq=Hkv, Hkv=Hkv, d=16, d_idx=16, topk=k)
        nb = sh.nb
        sel = rng.integers(-1, nb, size=(B, Hkv, Nq, k)).astype(np.int32)
        sel[..., 0] = np.where(rng.random((B, Hkv, Nq)) < 0.1, nb + 3, sel[..., 0])   # out of range: ignored
        m = oracle.block_mask(sh, sel)
        T, W = (Nq + 127) // 128, (nb + 31) // 32
        assert m.shape == (B, Hkv, T, W)
        for b in range(B):
            for r in range(Hkv):
                for t in range(T):
                    ids = sel[b, r, 128 * t:128 * (t + 1)].reshape(-1)
                    union = sorted({int(c) for c in ids if 0 <= c < nb})
                    assert oracle.mask_walk(m[b, r, t]).tolist() == union
                    if nb % 32:
                        assert int(m[b, r, t, W - 1]) >> (nb % 32) == 0
    assert oracle.mask_walk(np.zeros(3, dtype=np.uint32)).tolist() == []
