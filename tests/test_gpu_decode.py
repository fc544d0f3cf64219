"""GPU parity of the decode path: one new query per sequence attends to a
KV / K_idx cache through the same two entry points (Nq = 1, q_offset = pos,
Nk = pos + 1, kv_rows = cache capacity).  The cache here holds 64K tokens
(512 blocks, so selection ranks 511 earlier blocks and the index kernel
splits the key range across CTAs); the last blocks are partial, as in the
1M-token decode workload."""
import numpy as np
import pytest

import oracle
from msa_testutil import assert_close, bf16_to_np, check_selection, to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def decode_case():
    from block_sparse_gqa_causal_gb300.inputs import make_inputs
    from block_sparse_gqa_causal_gb300.workloads import DECODE_1M
    w = DECODE_1M.scaled(name="decode_64k", B=2, N=65536, Hq=16, Hkv=4, decode_steps=200, seed=11)
    return w, make_inputs(w)


@pytest.mark.parametrize("step", [0, 57, 199])
def test_decode_step_parity(decode_case, step):
    import torch
    from block_sparse_gqa_causal_gb300 import api
    from block_sparse_gqa_causal_gb300.inputs import decode_position
    w, x = decode_case
    pos = decode_position(w, step)
    q = np.ascontiguousarray(x["q"][:, step:step + 1])
    qi = np.ascontiguousarray(x["q_idx"][:, step:step + 1])
    sh = api.Shape(B=w.B, Nq=1, Nk=pos + 1, Hq=w.Hq, Hkv=w.Hkv, d=w.d, d_idx=w.d_idx, topk=w.topk, q_offset=pos,
                   kv_rows=w.N)
    t = {n: to_torch(a) for n, a in (("q", q), ("q_idx", qi), ("k", x["k"]), ("v", x["v"]), ("k_idx", x["k_idx"]))}
    sel, bs = api.index_select(sh, t["q_idx"], t["k_idx"], return_scores=True)
    o, lse = api.sparse_attn_fwd(sh, t["q"], t["k"], t["v"], sel)
    torch.cuda.synchronize()

    osh = oracle.Shape(B=w.B, Nq=1, Nk=pos + 1, Hq=w.Hq, Hkv=w.Hkv, d=w.d, d_idx=w.d_idx, topk=w.topk, q_offset=pos,
                       kv_rows=w.N)
    rows = np.arange(w.B)
    bs_o = oracle.block_scores(osh, qi, x["k_idx"], rows)
    bs_g = bs.cpu().numpy().reshape(w.B, w.Hkv, -1)
    vis = np.isfinite(bs_o)
    assert_close(bs_g[vis], bs_o[vis], "block scores", max_abs=2e-3, rel_l2=1e-4)
    sel_np = sel.cpu().numpy()
    sel_o = oracle.select(osh, bs_o, rows)
    sel_g = sel_np[:, :, 0, :]
    exact, tol = check_selection(w.topk, 128, pos, 1, rows, sel_g, sel_o, bs_o)
    assert exact >= 1
    o_ref, lse_ref = oracle.sparse_fwd(osh, q, x["k"], x["v"], sel_g, rows)
    assert_close(bf16_to_np(o).reshape(o_ref.shape), o_ref, "o", bf16_out=True)
    assert_close(lse.cpu().numpy().reshape(lse_ref.shape), lse_ref, "lse", max_abs=1e-3, rel_l2=1e-5)


def test_decode_long_cache_split_selection():
    """A cache of 2,088 blocks with two (query, group) rows: the selection runs
    one CTA per row (segments spread over its warps, then merged) and the
    forward splits each row's chunks over several CTAs (split-KV)."""
    import torch
    from block_sparse_gqa_causal_gb300 import api
    from block_sparse_gqa_causal_gb300.inputs import f32_to_bf16_bits
    B, Hq, Hkv, d, k = 1, 4, 2, 64, 16
    cap = 2088 * 128
    pos = cap - 37                                   # the last block is partial
    rng = np.random.default_rng(23)
    bf = lambda shape: f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))
    x = {"q": bf((B, 1, Hq, d)), "q_idx": bf((B, 1, Hkv, d)), "k": bf((B, cap, Hkv, d)), "v": bf((B, cap, Hkv, d)),
         "k_idx": bf((B, cap, d))}
    sh = api.Shape(B=B, Nq=1, Nk=pos + 1, Hq=Hq, Hkv=Hkv, d=d, d_idx=d, topk=k, q_offset=pos, kv_rows=cap)
    t = {n: to_torch(a) for n, a in x.items()}
    sel, bs = api.index_select(sh, t["q_idx"], t["k_idx"], return_scores=True)
    o, lse = api.sparse_attn_fwd(sh, t["q"], t["k"], t["v"], sel)
    torch.cuda.synchronize()
    osh = oracle.Shape(B=B, Nq=1, Nk=pos + 1, Hq=Hq, Hkv=Hkv, d=d, d_idx=d, topk=k, q_offset=pos, kv_rows=cap)
    rows = np.arange(B)
    bs_o = oracle.block_scores(osh, x["q_idx"], x["k_idx"], rows)
    bs_g = bs.cpu().numpy().reshape(B, Hkv, -1)
    vis = np.isfinite(bs_o)
    assert_close(bs_g[vis], bs_o[vis], "block scores", max_abs=2e-3, rel_l2=1e-4)
    sel_g = sel.cpu().numpy()[:, :, 0, :]
    sel_o = oracle.select(osh, bs_o, rows)
    exact, tol = check_selection(k, 128, pos, 1, rows, sel_g, sel_o, bs_o)
    assert exact >= 1
    o_ref, lse_ref = oracle.sparse_fwd(osh, x["q"], x["k"], x["v"], sel_g, rows)
    assert_close(bf16_to_np(o).reshape(o_ref.shape), o_ref, "o", bf16_out=True)
    assert_close(lse.cpu().numpy().reshape(lse_ref.shape), lse_ref, "lse", max_abs=1e-3, rel_l2=1e-5)


@pytest.mark.parametrize("step", [0, 57, 199])
def test_decode_split_fused_selection_matches_scores_path(decode_case, step):
    """Without block scores asked for, a decode row's blocks are ranked in the
    score kernel's epilogue, each CTA keeping its slice's 16 best, and a merge
    kernel picks the row's selection.  It must equal the selection made from
    the stored scores (same fp32 scores, same tie rule) and the oracle's."""
    import torch
    from block_sparse_gqa_causal_gb300 import api
    from block_sparse_gqa_causal_gb300.inputs import decode_position
    w, x = decode_case
    pos = decode_position(w, step)
    qi = np.ascontiguousarray(x["q_idx"][:, step:step + 1])
    sh = api.Shape(B=w.B, Nq=1, Nk=pos + 1, Hq=w.Hq, Hkv=w.Hkv, d=w.d, d_idx=w.d_idx, topk=w.topk, q_offset=pos,
                   kv_rows=w.N)
    tqi, tki = to_torch(qi), to_torch(x["k_idx"])
    sel_f = api.index_select(sh, tqi, tki)
    sel_s, _ = api.index_select(sh, tqi, tki, return_scores=True)
    torch.cuda.synchronize()
    assert np.array_equal(sel_f.cpu().numpy(), sel_s.cpu().numpy())
    osh = oracle.Shape(B=w.B, Nq=1, Nk=pos + 1, Hq=w.Hq, Hkv=w.Hkv, d=w.d, d_idx=w.d_idx, topk=w.topk, q_offset=pos,
                       kv_rows=w.N)
    rows = np.arange(w.B)
    bs_o = oracle.block_scores(osh, qi, x["k_idx"], rows)
    sel_o = oracle.select(osh, bs_o, rows)
    exact, tol = check_selection(w.topk, 128, pos, 1, rows, sel_f.cpu().numpy()[:, :, 0, :], sel_o, bs_o)
    assert exact >= 1


def test_decode_split_fused_selection_ties_go_to_lower_blocks():
    """Every K_idx row equal: all block scores tie exactly, across the CTAs'
    slices too, so the selection is blocks 0..k-2 plus the local block."""
    import torch
    from block_sparse_gqa_causal_gb300 import api
    from block_sparse_gqa_causal_gb300.inputs import f32_to_bf16_bits
    B, Hkv, d, k = 2, 2, 64, 16
    cap = 700 * 128
    rng = np.random.default_rng(5)
    qi = f32_to_bf16_bits(rng.standard_normal((B, 1, Hkv, d)).astype(np.float32))
    row = f32_to_bf16_bits(rng.standard_normal((1, 1, d)).astype(np.float32))
    ki = np.ascontiguousarray(np.broadcast_to(row, (B, cap, d)))
    for pos in (cap - 1, cap - 200, 31 * 128 + 5):
        sh = api.Shape(B=B, Nq=1, Nk=pos + 1, Hq=Hkv, Hkv=Hkv, d=d, d_idx=d, topk=k, q_offset=pos, kv_rows=cap)
        sel = api.index_select(sh, to_torch(qi), to_torch(ki))
        torch.cuda.synchronize()
        want = np.array(list(range(k - 1)) + [pos // 128], dtype=np.int32)
        assert np.array_equal(sel.cpu().numpy().reshape(B * Hkv, k), np.broadcast_to(want, (B * Hkv, k)))


@pytest.mark.slow
def test_decode_1m_split_fused_selection_matches_scores_path():
    """The benchmark's decode shape (4 sequences, 1,048,576-token caches, 8
    groups) at its last step: the split-fused selection equals the one made
    from the stored scores, and every row is a valid selection."""
    import torch
    from block_sparse_gqa_causal_gb300 import api
    from block_sparse_gqa_causal_gb300.inputs import f32_to_bf16_bits
    B, Hkv, d, k, cap = 4, 8, 128, 16, 1048576
    pos = cap - 1
    g = torch.Generator(device="cuda").manual_seed(17)
    qi = torch.randn(B, 1, Hkv, d, device="cuda", generator=g).bfloat16()
    ki = torch.randn(B, cap, d, device="cuda", generator=g).bfloat16()
    sh = api.Shape(B=B, Nq=1, Nk=pos + 1, Hq=64, Hkv=Hkv, d=d, d_idx=d, topk=k, q_offset=pos, kv_rows=cap)
    sel_f = api.index_select(sh, qi, ki)
    sel_s, _ = api.index_select(sh, qi, ki, return_scores=True)
    torch.cuda.synchronize()
    s = sel_f.cpu().numpy().reshape(B * Hkv, k)
    assert np.array_equal(s, sel_s.cpu().numpy().reshape(B * Hkv, k))
    assert np.all(s[:, -1] == pos // 128) and np.all(np.diff(s, axis=1) > 0) and np.all(s >= 0)


@pytest.mark.parametrize("B,Nq,Nk,q_offset,Hkv,k", [(1, 3000, 3000, 0, 8, 16), (2, 1, 200000, 199999, 4, 16),
                                                     (1, 40, 70000, 69960, 2, 8), (1, 256, 202802, 202546, 2, 16)])
def test_split_selection_ignores_stale_workspace(B, Nq, Nk, q_offset, Hkv, k):
    """Rows split across CTAs with the scores not asked for (per-slice
    candidates, then the merge), run in a workspace filled with garbage first:
    the selection must equal the scores path's.  A row tile skips the slices
    past all its blocks, which then hold stale memory: in the last case the
    final slice (24 blocks wide) holds only block 1584, which the first tile's
    rows (local blocks 1582, 1583) never see."""
    import torch
    from block_sparse_gqa_causal_gb300 import api
    g = torch.Generator(device="cuda").manual_seed(Nq + Nk)
    sh = api.Shape(B=B, Nq=Nq, Nk=Nk, Hq=Hkv, Hkv=Hkv, d=128, d_idx=128, topk=k, q_offset=q_offset)
    qi = torch.randn(B, Nq, Hkv, 128, device="cuda", generator=g).bfloat16()
    ki = torch.randn(B, Nk, 128, device="cuda", generator=g).bfloat16()
    want, _ = api.index_select(sh, qi, ki, return_scores=True)
    for fill in (0xFF, 0x7F, 0x3C):
        ws = api.new_workspace(sh, api.OP_INDEX_SELECT)
        ws.fill_(fill)
        ws[:256] = 0                                   # the status word starts clear
        got = api.index_select(sh, qi, ki, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(got, want), fill


def test_kv_append_writes_exactly_the_new_rows():
    """msa_kv_append: the new tokens' K, V and K_idx rows land at cache rows
    q_offset .. q_offset+Nq-1 of every batch entry, bit for bit; every other
    row is untouched; a pair given as None is skipped."""
    import torch
    from block_sparse_gqa_causal_gb300 import api
    rng = np.random.default_rng(11)
    B, cap, Hkv, d, di = 3, 1000, 2, 64, 128
    mk = lambda shape: torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16).cuda()
    for Nq, qo, skip_v in ((1, 999, False), (5, 300, False), (2, 0, True)):
        k, v, ki = mk((B, cap, Hkv, d)), mk((B, cap, Hkv, d)), mk((B, cap, di))
        k0, v0, ki0 = k.clone(), v.clone(), ki.clone()
        kn, vn, kin = mk((B, Nq, Hkv, d)), mk((B, Nq, Hkv, d)), mk((B, Nq, di))
        sh = api.Shape(B=B, Nq=Nq, Nk=qo + Nq, Hq=4 * Hkv, Hkv=Hkv, d=d, d_idx=di, topk=4, q_offset=qo, kv_rows=cap)
        api.kv_append(sh, kn, None if skip_v else vn, kin, k, None if skip_v else v, ki)
        torch.cuda.synchronize()
        want_k, want_v, want_ki = k0.clone(), v0.clone(), ki0.clone()
        want_k[:, qo:qo + Nq] = kn
        if not skip_v:
            want_v[:, qo:qo + Nq] = vn
        want_ki[:, qo:qo + Nq] = kin
        for got, want in ((k, want_k), (v, want_v), (ki, want_ki)):
            assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_decode_steps_through_the_cache_append():
    """A decode loop as a caller runs it, at a head layout no other decode case
    uses (G = 4, d = d_idx = 64, batch 2): each step appends the new token's K,
    V and K_idx rows to caches that end at the previous token
    (msa_kv_append), selects and attends for its query, and is checked against
    the oracle on caches holding every token so far -- steps that stay inside
    a block and one that opens a new block."""
    import torch
    from block_sparse_gqa_causal_gb300 import api
    from block_sparse_gqa_causal_gb300.inputs import f32_to_bf16_bits
    rng = np.random.default_rng(23)
    bf = lambda shape: f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))
    B, Hq, Hkv, d, di, k, cap = 2, 8, 2, 64, 64, 8, 8192
    pos0 = 6013                                       # steps at 6013 .. 6017 cross into block 47 at 6016
    kx, vx, kix = bf((B, cap, Hkv, d)), bf((B, cap, Hkv, d)), bf((B, cap, di))
    kc, vc, kic = to_torch(kx.copy()), to_torch(vx.copy()), to_torch(kix.copy())
    kc[:, pos0:].zero_()
    vc[:, pos0:].zero_()
    kic[:, pos0:].zero_()
    for s in range(5):
        pos = pos0 + s
        q, qi = bf((B, 1, Hq, d)), bf((B, 1, Hkv, di))
        sh = api.Shape(B=B, Nq=1, Nk=pos + 1, Hq=Hq, Hkv=Hkv, d=d, d_idx=di, topk=k, q_offset=pos, kv_rows=cap)
        api.kv_append(sh, to_torch(np.ascontiguousarray(kx[:, pos:pos + 1])), to_torch(np.ascontiguousarray(vx[:, pos:pos + 1])),
                      to_torch(np.ascontiguousarray(kix[:, pos:pos + 1])), kc, vc, kic)
        sel = api.index_select(sh, to_torch(qi), kic)
        o, lse = api.sparse_attn_fwd(sh, to_torch(q), kc, vc, sel)
        torch.cuda.synchronize()
        osh = oracle.Shape(B=B, Nq=1, Nk=pos + 1, Hq=Hq, Hkv=Hkv, d=d, d_idx=di, topk=k, q_offset=pos, kv_rows=cap)
        rows = np.arange(B)
        bs_o = oracle.block_scores(osh, qi, kix, rows)
        sel_o = oracle.select(osh, bs_o, rows)
        sel_g = sel.cpu().numpy()[:, :, 0, :]
        check_selection(k, 128, pos, 1, rows, sel_g, sel_o, bs_o)
        assert np.all(sel_g[:, :, -1] == pos // 128), "the local block is last and always selected"
        o_ref, lse_ref = oracle.sparse_fwd(osh, q, kx, vx, sel_g, rows)
        assert_close(bf16_to_np(o).reshape(o_ref.shape), o_ref, f"o (step {s})", bf16_out=True)
        assert_close(lse.cpu().numpy().reshape(lse_ref.shape), lse_ref, f"lse (step {s})", max_abs=1e-3, rel_l2=1e-5)
