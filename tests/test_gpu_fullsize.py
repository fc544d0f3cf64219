"""Parity at the benchmark's full size, in the launch configuration bench.py
times: train_n128k (B=1, N=131,072, Hq=64, Hkv=8, d=d_idx=128, k=16, the
bench's seeded inputs), run as the bench runs it: one msa_train_step call --
selection fused into the index kernel with no stored scores, one inverse
index, the key-major forward, the lse_idx-only KL pass, the fused backward
that returns the KL loss.

The oracle recomputes sampled outputs one row (or one key block) at a time:
the selection, O and LSE, lse_idx, the KL of each sampled row, dq and dq_idx
of the sampled rows, dK, dV and dK_idx of a few key blocks (an early heavy
one, a middle one, the last one).  Over every row the test checks what holds
at any size: each selection is valid (ascending, distinct, ends with the
local block, only visible blocks), outputs and gradients are finite, the KL
rows are non-negative and the loss is kl_coef times their mean.
"""
import numpy as np
import pytest

import oracle
from msa_testutil import assert_close, bf16_to_np, check_selection

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

KL_COEF = 1.0


@pytest.fixture(scope="module")
def step():
    import torch
    from block_sparse_gqa_causal_gb300 import api
    from block_sparse_gqa_causal_gb300.inputs import make_inputs
    from block_sparse_gqa_causal_gb300.workloads import BY_NAME
    w = BY_NAME["train_n128k"]
    x = make_inputs(w, with_grad=True)
    dev = torch.device("cuda", 0)
    names = ["q", "k", "v", "q_idx", "k_idx", "d_o"]
    d = {n: torch.from_numpy(x[n].view(np.int16)).view(torch.bfloat16).to(dev) for n in names}
    sh = api.Shape(B=w.B, Nq=w.N, Nk=w.N, Hq=w.Hq, Hkv=w.Hkv, d=w.d, d_idx=w.d_idx, topk=w.topk)
    # the bench's step
    out = api.train_step(sh, d["q"], d["k"], d["v"], d["q_idx"], d["k_idx"], d["d_o"], KL_COEF)
    torch.cuda.synchronize()
    res = {"sel": out["sel"].cpu().numpy(), "o": bf16_to_np(out["o"]), "lse": out["lse"].cpu().numpy(),
           "lse_idx": out["lse_idx"].cpu().numpy(), "kl_rows": out["kl_rows"].cpu().numpy(),
           "kl_loss": float(out["kl_loss"].item()),
           "grads": [bf16_to_np(out[n]) for n in ("dq", "dk", "dv", "dq_idx", "dk_idx")]}
    osh = oracle.Shape(B=w.B, Nq=w.N, Nk=w.N, Hq=w.Hq, Hkv=w.Hkv, d=w.d, d_idx=w.d_idx, topk=w.topk)
    rng = np.random.default_rng(2024)
    fixed = [0, 1, 127, 128, 129, 2047, 2048, 2049, 65535, 65536, w.N - 129, w.N - 1]
    rows = np.unique(np.concatenate([fixed, rng.choice(w.N, size=12, replace=False)]))
    return w, x, osh, res, rows


def test_selection_sampled_and_valid_everywhere(step):
    w, x, osh, res, rows = step
    bs_o = oracle.block_scores(osh, x["q_idx"], x["k_idx"], rows)
    sel_o = oracle.select(osh, bs_o, rows)
    sel_g = oracle.sel_rows_from_full(osh, res["sel"], rows)
    exact, tol = check_selection(w.topk, 128, 0, w.N, rows, sel_g, sel_o, bs_o)
    assert exact >= len(rows) * w.Hkv // 2
    # every row: ascending distinct ids ending with the local block, all visible
    s = res["sel"][0]                                                   # [Hkv, N, k]
    c0 = (np.arange(w.N) // 128)[None, :]
    valid = s >= 0
    assert np.all(s.max(axis=-1) == c0)                                  # the local block is the largest id
    ok_order = np.where(valid[..., 1:] & valid[..., :-1], np.diff(s, axis=-1) > 0, True)
    assert np.all(ok_order)
    assert np.all(np.where(valid, s <= c0[..., None], True))
    n_valid = valid.sum(axis=-1)
    assert np.all(n_valid == np.minimum(w.topk, c0 + 1))


def test_forward_sampled(step):
    w, x, osh, res, rows = step
    sel_rows = oracle.sel_rows_from_full(osh, res["sel"], rows)
    o_ref, lse_ref = oracle.sparse_fwd(osh, x["q"], x["k"], x["v"], sel_rows, rows)
    o_g = res["o"].reshape(w.N, w.Hq, w.d)[rows]
    assert_close(o_g, o_ref, "o (sampled rows)", bf16_out=True)
    lse_g = res["lse"][0][:, rows].T
    assert_close(lse_g, lse_ref, "lse (sampled rows)", max_abs=1e-3, rel_l2=1e-5)
    assert np.all(np.isfinite(res["o"])) and np.all(np.isfinite(res["lse"]))


def test_kl_sampled_and_loss(step):
    w, x, osh, res, rows = step
    sel_rows = oracle.sel_rows_from_full(osh, res["sel"], rows)
    lse_idx_ref, kl_ref = oracle.kl(osh, x["q"], x["k"], x["q_idx"], x["k_idx"], sel_rows, rows)
    assert_close(res["lse_idx"][0][:, rows].T, lse_idx_ref, "lse_idx (sampled rows)", max_abs=1e-3, rel_l2=1e-5)
    assert_close(res["kl_rows"][0][:, rows].T, kl_ref, "kl_rows (sampled rows)")
    kl_all = res["kl_rows"].astype(np.float64)
    assert np.all(np.isfinite(kl_all)) and np.all(kl_all > -1e-3)
    want = KL_COEF * kl_all.sum() / (w.B * w.N * w.Hkv)
    assert abs(res["kl_loss"] - want) <= 1e-4 * abs(want) + 1e-7


def test_gradients_sampled(step):
    w, x, osh, res, rows = step
    g_dq, g_dk, g_dv, g_dqi, g_dki = res["grads"]
    for g in res["grads"]:
        assert np.all(np.isfinite(g))
    args = (osh, x["q"], x["k"], x["v"], x["d_o"], x["q_idx"], x["k_idx"], res["sel"], KL_COEF)
    dq, dqi = oracle.bwd_rows(*args, rows=rows)
    assert_close(g_dq.reshape(w.N, w.Hq, w.d)[rows], dq, "dq (sampled rows)", bf16_out=True)
    assert_close(g_dqi.reshape(w.N, w.Hkv, w.d_idx)[rows], dqi, "dq_idx (sampled rows)", bf16_out=True)
    kblocks = np.array([64, 700, w.N // 128 - 1])
    dk, dv, dki = oracle.bwd_keys(*args, kblocks=kblocks)
    keys = (kblocks[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)
    assert_close(g_dk[:, keys], dk, "dk (sampled blocks)", bf16_out=True)
    assert_close(g_dv[:, keys], dv, "dv (sampled blocks)", bf16_out=True)
    assert_close(g_dki[:, keys], dki, "dk_idx (sampled blocks)", bf16_out=True)
