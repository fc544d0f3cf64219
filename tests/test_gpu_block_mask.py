"""GPU parity of msa_block_mask (section 4.3 of "Sparse Attention · Part
II": the selection of each 128-query tile as one bit per key block, 32 per
word, and the traversal that lists the active blocks) against the oracle,
bit for bit: on the section's worked example, on random selections at
ragged sizes (tiles cut short, the last word partly unused, ids to ignore)
and on a real selection made by msa_index_select."""
import numpy as np
import pytest

import oracle
from msa_testutil import to_torch

pytestmark = pytest.mark.gpu


def _run(sh, sel_np):
    import torch
    from block_sparse_gqa_causal_gb300 import api
    # the mask depends on B, Nq, Nk, Hkv and topk only; head dims the library supports
    ash = api.Shape(B=sh.B, Nq=sh.Nq, Nk=sh.Nk, Hq=sh.Hq, Hkv=sh.Hkv, d=64, d_idx=64, topk=sh.topk,
                    q_offset=sh.q_offset)
    mask, cnt, blk = api.block_mask(ash, torch.from_numpy(sel_np).cuda(), counts=True, blocks=True)
    torch.cuda.synchronize()
    return mask.cpu().numpy().view(np.uint32), cnt.cpu().numpy(), blk.cpu().numpy()


def _check(sh, sel_np):
    mask, cnt, blk = _run(sh, sel_np)
    want = oracle.block_mask(sh, sel_np)
    assert np.array_equal(mask, want)
    nb = sh.nb
    for idx in np.ndindex(*want.shape[:3]):
        walk = oracle.mask_walk(want[idx])
        assert cnt[idx] == len(walk)
        assert np.array_equal(blk[idx][:len(walk)], walk)
        assert np.all(blk[idx][len(walk):nb] == -1)


def test_block_mask_worked_example():
    sh = oracle.Shape(B=1, Nq=128, Nk=8 * 128, Hq=1, Hkv=1, d=16, d_idx=16, topk=2, q_offset=7 * 128)
    sel = np.full((1, 1, 128, 2), -1, dtype=np.int32)
    sel[0, 0, 0] = [0, 3]
    sel[0, 0, 77] = [6, -1]
    sel[0, 0, 5] = [3, -1]
    mask, cnt, blk = _run(sh, sel)
    assert int(mask[0, 0, 0, 0]) == 73 and int(cnt[0, 0, 0]) == 3
    assert blk[0, 0, 0].tolist() == [0, 3, 6, -1, -1, -1, -1, -1]


@pytest.mark.parametrize("B,Nq,nkb,Hkv,k", [(1, 300, 40, 2, 4), (2, 129, 64, 1, 3), (3, 1, 97, 3, 16),
                                            (1, 1000, 1000, 2, 32)])
def test_block_mask_random_selections(B, Nq, nkb, Hkv, k):
    rng = np.random.default_rng(Nq + nkb)
    sh = oracle.Shape(B=B, Nq=Nq, Nk=nkb * 128 - 7, Hq=Hkv, Hkv=Hkv, d=16, d_idx=16, topk=k)
    sel = rng.integers(-1, sh.nb, size=(B, Hkv, Nq, k)).astype(np.int32)
    sel[..., 0] = np.where(rng.random((B, Hkv, Nq)) < 0.1, sh.nb + 5, sel[..., 0])   # ignored
    _check(sh, sel)


def test_block_mask_of_a_real_selection():
    import torch
    from block_sparse_gqa_causal_gb300 import api
    from block_sparse_gqa_causal_gb300.inputs import make_inputs
    from block_sparse_gqa_causal_gb300.workloads import BY_NAME
    w = BY_NAME["fwd_n8k_b2"]
    x = make_inputs(w)
    ash = api.Shape(B=w.B, Nq=w.N, Nk=w.N, Hq=w.Hq, Hkv=w.Hkv, d=w.d, d_idx=w.d_idx, topk=w.topk)
    sel = api.index_select(ash, to_torch(x["q_idx"]), to_torch(x["k_idx"]))
    torch.cuda.synchronize()
    sh = oracle.Shape(B=w.B, Nq=w.N, Nk=w.N, Hq=w.Hq, Hkv=w.Hkv, d=w.d, d_idx=w.d_idx, topk=w.topk)
    _check(sh, sel.cpu().numpy())
