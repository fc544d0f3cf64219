"""GPU parity of the index projections and the dense indexer warm-up.

"Sparse Attention · Part II": section 3.2's detachment equation
(Q_idx = stopgrad(X) W_q^idx, K_idx = stopgrad(X) W_k^idx; the KL trains the
two projections and sends nothing into X) and section 3.1's dense warm-up
loss in MSA's per-group form.  Through the C-ABI: msa_index_proj_fwd,
msa_index_proj_bwd and msa_warmup_kl against the CPU oracle's index_proj,
index_proj_bwd, warmup_kl and warmup_grad, on synthetic weights (the pages
give none).  Tolerances as elsewhere: max-abs 2e-2 beyond a bf16 output's
own rounding and relative L2 1e-2; lse within 1e-3.
"""
import math

import numpy as np
import pytest

import oracle
from msa_testutil import assert_close, bf16_to_np, to_torch

pytestmark = pytest.mark.gpu


def _bf(rng, shape, scale=1.0):
    from block_sparse_gqa_causal_gb300.inputs import f32_to_bf16_bits
    return f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


@pytest.mark.parametrize("T,Dm,Hkv,di", [(1000, 512, 2, 128), (300, 136, 3, 64), (129, 1024, 8, 128)])
def test_index_projection_forward(T, Dm, Hkv, di):
    import torch
    from block_sparse_gqa_causal_gb300 import api
    rng = np.random.default_rng(T + Dm)
    X = _bf(rng, (T, Dm))
    Wq, Wk = _bf(rng, (Dm, Hkv * di), 1 / math.sqrt(Dm)), _bf(rng, (Dm, di), 1 / math.sqrt(Dm))
    sh = api.ProjShape(T=T, Dm=Dm, Hkv=Hkv, d_idx=di)
    qi, ki = api.index_proj_fwd(sh, to_torch(X), to_torch(Wq), to_torch(Wk))
    torch.cuda.synchronize()
    qo, ko = oracle.index_proj(X, Wq, Wk, Hkv, di)
    assert_close(bf16_to_np(qi).reshape(qo.shape), qo, "q_idx = X W_q", bf16_out=True)
    assert_close(bf16_to_np(ki), ko, "k_idx = X W_k", bf16_out=True)


@pytest.mark.parametrize("T,Dm,Hkv,di", [(1000, 512, 2, 128), (300, 136, 3, 64), (20000, 256, 2, 128)])
def test_index_projection_weight_gradient(T, Dm, Hkv, di):
    """dW = X^T dY in fp32; the 20,000-token case splits the token sum over
    many CTAs (parts added in a fixed order: the same bits on a second call)."""
    import torch
    from block_sparse_gqa_causal_gb300 import api
    rng = np.random.default_rng(T * 3 + Dm)
    X = _bf(rng, (T, Dm))
    dq, dk = _bf(rng, (T, Hkv, di)), _bf(rng, (T, di))
    sh = api.ProjShape(T=T, Dm=Dm, Hkv=Hkv, d_idx=di)
    dwq, dwk = api.index_proj_bwd(sh, to_torch(X), to_torch(dq), to_torch(dk))
    dwq2, dwk2 = api.index_proj_bwd(sh, to_torch(X), to_torch(dq), to_torch(dk))
    torch.cuda.synchronize()
    assert torch.equal(dwq, dwq2) and torch.equal(dwk, dwk2)
    wq_o, wk_o = oracle.index_proj_bwd(X, dq, dk, Hkv, di)
    # fp32 results of exact bf16 products: the error is accumulation rounding only
    scale = math.sqrt(T)
    assert_close(dwq.cpu().numpy().astype(np.float64) / scale, wq_o / scale, "dW_q = X^T dq_idx")
    assert_close(dwk.cpu().numpy().astype(np.float64) / scale, wk_o / scale, "dW_k = X^T dk_idx")


WARM = [  # name, B, N, Hq, Hkv, d, d_idx
    ("n2048_g8", 1, 2048, 16, 2, 128, 128),
    ("b2_n1000_g4_ragged", 2, 1000, 8, 2, 128, 128),
    ("n4096_32_blocks", 1, 4096, 8, 1, 128, 128),
    ("n1500_g8_d64", 1, 1500, 16, 2, 64, 64),
]


def _warm_inputs(name, B, N, Hq, Hkv, d=128, di=128, seed=0):
    rng = np.random.default_rng(seed)
    x = {"q": _bf(rng, (B, N, Hq, d)), "k": _bf(rng, (B, N, Hkv, d)), "v": _bf(rng, (B, N, Hkv, d)),
         "q_idx": _bf(rng, (B, N, Hkv, di)), "k_idx": _bf(rng, (B, N, di))}
    return x


@pytest.mark.parametrize("case", WARM, ids=[c[0] for c in WARM])
def test_warmup_kl_and_gradients(case):
    import torch
    from block_sparse_gqa_causal_gb300 import api
    name, B, N, Hq, Hkv, d, di = case
    x = _warm_inputs(*case, seed=N + Hq)
    coef = float(B * N * Hkv)                           # gradients of order one
    sh = api.Shape(B=B, Nq=N, Nk=N, Hq=Hq, Hkv=Hkv, d=d, d_idx=di, topk=1)
    t = {n: to_torch(a) for n, a in x.items()}
    out = api.warmup_kl(sh, t["q"], t["k"], t["v"], t["q_idx"], t["k_idx"], coef)
    again = api.warmup_kl(sh, t["q"], t["k"], t["v"], t["q_idx"], t["k_idx"], coef)
    torch.cuda.synchronize()
    for n in out:
        assert torch.equal(out[n], again[n]), n          # deterministic
    nb = (N + 127) // 128
    osh = oracle.Shape(B=B, Nq=N, Nk=N, Hq=Hq, Hkv=Hkv, d=d, d_idx=di, topk=nb)
    lse_idx_o, kl_o = oracle.warmup_kl(osh, x["q"], x["k"], x["q_idx"], x["k_idx"])
    to_rows = lambda a: a.cpu().numpy().transpose(0, 2, 1).reshape(B * N, Hkv)
    assert_close(to_rows(out["lse_idx"]), lse_idx_o, "warm-up lse_idx", max_abs=1e-3, rel_l2=1e-5)
    assert_close(to_rows(out["kl_rows"]), kl_o, "warm-up kl_rows")
    want = coef * kl_o.sum() / (B * N * Hkv)
    assert abs(float(out["kl_loss"].item()) - want) <= 1e-4 * abs(want) + 1e-6
    # the dense main attention's lse: the teacher's normaliser
    every = np.array([[list(range(min(nb, i // 128 + 1))) + [-1] * (nb - min(nb, i // 128 + 1))
                       for i in range(N)]], dtype=np.int32)
    sel_rows = np.ascontiguousarray(np.repeat(np.tile(every[0], (B, 1, 1)).reshape(B * N, 1, nb), Hkv, axis=1))
    _, lse_o = oracle.sparse_fwd(osh, x["q"], x["k"], x["v"], sel_rows)
    assert_close(out["lse"].cpu().numpy().transpose(0, 2, 1).reshape(B * N, Hq), lse_o, "dense lse", max_abs=1e-3,
                 rel_l2=1e-5)
    dqi_o, dki_o = oracle.warmup_grad(osh, x["q"], x["k"], x["q_idx"], x["k_idx"], coef)
    assert_close(bf16_to_np(out["dq_idx"]), dqi_o, "warm-up dq_idx", bf16_out=True)
    assert_close(bf16_to_np(out["dk_idx"]), dki_o, "warm-up dk_idx", bf16_out=True)


def test_warmup_equals_the_sparse_kl_with_every_block_selected():
    """With topk >= the number of blocks the selection keeps every visible
    block, so msa_kl_fwd's rows and msa_sparse_attn_fwd's lse are the warm-up's."""
    import torch
    from block_sparse_gqa_causal_gb300 import api
    B, N, Hq, Hkv = 1, 1536, 16, 2
    x = _warm_inputs("s", B, N, Hq, Hkv, seed=77)
    t = {n: to_torch(a) for n, a in x.items()}
    nb = N // 128
    sh = api.Shape(B=B, Nq=N, Nk=N, Hq=Hq, Hkv=Hkv, d=128, d_idx=128, topk=nb)
    w = api.warmup_kl(sh, t["q"], t["k"], t["v"], t["q_idx"], t["k_idx"], 1.0)
    sel = api.index_select(sh, t["q_idx"], t["k_idx"])
    o, lse = api.sparse_attn_fwd(sh, t["q"], t["k"], t["v"], sel)
    loss, lse_idx, kl_rows = api.kl_fwd(sh, t["q"], t["k"], t["q_idx"], t["k_idx"], sel, lse, 1.0)
    torch.cuda.synchronize()
    assert_close(w["lse"].cpu().numpy(), lse.cpu().numpy(), "lse (warm-up vs sparse, every block)", max_abs=1e-5,
                 rel_l2=1e-6)
    assert_close(w["kl_rows"].cpu().numpy(), kl_rows.cpu().numpy(), "kl rows (warm-up vs sparse)", max_abs=1e-5,
                 rel_l2=1e-5)
    assert abs(float(w["kl_loss"].item()) - float(loss.item())) <= 1e-5 * abs(float(loss.item()))


def test_projection_warmup_and_weight_gradient_chain():
    """X -> (msa_index_proj_fwd) q_idx, k_idx -> (msa_warmup_kl) dq_idx,
    dk_idx -> (msa_index_proj_bwd) dW_q, dW_k: each stage against the oracle
    on the library's own inputs for that stage, and the weight gradient
    against the oracle's chain from the same bf16 index inputs."""
    import torch
    from block_sparse_gqa_causal_gb300 import api
    B, N, Hq, Hkv, Dm = 1, 1024, 8, 2, 256
    rng = np.random.default_rng(5)
    X = _bf(rng, (B * N, Dm))
    Wq, Wk = _bf(rng, (Dm, Hkv * 128), 1 / math.sqrt(Dm)), _bf(rng, (Dm, 128), 1 / math.sqrt(Dm))
    q, k, v = _bf(rng, (B, N, Hq, 128)), _bf(rng, (B, N, Hkv, 128)), _bf(rng, (B, N, Hkv, 128))
    psh = api.ProjShape(T=B * N, Dm=Dm, Hkv=Hkv, d_idx=128)
    tX = to_torch(X)
    qi, ki = api.index_proj_fwd(psh, tX, to_torch(Wq), to_torch(Wk))
    coef = float(B * N * Hkv)
    sh = api.Shape(B=B, Nq=N, Nk=N, Hq=Hq, Hkv=Hkv, d=128, d_idx=128, topk=1)
    w = api.warmup_kl(sh, to_torch(q), to_torch(k), to_torch(v), qi.view(B, N, Hkv, 128), ki.view(B, N, 128), coef)
    dwq, dwk = api.index_proj_bwd(psh, tX, w["dq_idx"].view(B * N, Hkv, 128), w["dk_idx"].view(B * N, 128))
    torch.cuda.synchronize()
    # the chain in the oracle from the library's bf16 index inputs
    qi_b = qi.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B, N, Hkv, 128)
    ki_b = ki.view(torch.int16).cpu().numpy().view(np.uint16).reshape(B, N, 128)
    osh = oracle.Shape(B=B, Nq=N, Nk=N, Hq=Hq, Hkv=Hkv, d=128, d_idx=128, topk=N // 128)
    dqi_o, dki_o = oracle.warmup_grad(osh, q, k, qi_b, ki_b, coef)
    Xf = bf16_to_np(tX)
    wq_o, wk_o = oracle.index_proj_bwd(Xf, dqi_o.reshape(B * N, Hkv * 128), dki_o.reshape(B * N, 128), Hkv, 128)
    assert_close(dwq.cpu().numpy().astype(np.float64), wq_o, "dW_q of the warm-up loss")
    assert_close(dwk.cpu().numpy().astype(np.float64), wk_o, "dW_k of the warm-up loss")
