"""msa_index_select_noalloc: index selection for callers that cannot allocate.

Callers such as a serving process with a frozen memory pool, or a plugin
that only receives raw device pointers, cannot provide a workspace.  This
entry point runs the same selection as msa_index_select with its scratch in
a static device array inside the library.  The test calls it through the
C-ABI on two consecutive calls and checks each result against the
workspace-based msa_index_select (block indices are integers: bit-exact).
It lives in its own file, collected last, and passes alone or after the
rest of the suite (the first call on a device performs the one-time
address lookup).
"""
import ctypes

import pytest

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    from block_sparse_gqa_causal_gb300 import api
    L = api.lib()
    fn = L.msa_index_select_noalloc
    fn.argtypes = [ctypes.POINTER(api._CShape), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


CASES = [
    # prefill, topk <= 16: the top-k runs in the score kernel, no scratch used
    ("fused_small", dict(B=2, Nq=1000, Nk=1000, Hq=8, Hkv=2, d=64, d_idx=64, topk=4)),
    ("fused_g8", dict(B=1, Nq=3000, Nk=3000, Hq=32, Hkv=8, d=128, d_idx=128, topk=16)),
    # a 32K prefill: its fused selection needs no scratch, so the 64 MiB limit does not apply
    ("fused_32k", dict(B=1, Nq=32768, Nk=32768, Hq=32, Hkv=8, d=128, d_idx=128, topk=16)),
    # decode: a row's blocks split across CTAs, per-slice candidates in the array, then a merge
    ("split_decode", dict(B=2, Nq=1, Nk=200000, Hq=4, Hkv=4, d=128, d_idx=128, topk=16, q_offset=199999)),
    # topk > 16: block scores in the array, then the separate top-k kernel (warp per row)
    ("scores_k24", dict(B=1, Nq=2000, Nk=2000, Hq=2, Hkv=2, d=64, d_idx=64, topk=24)),
    # topk > 16 with a long decode row (a CTA per row in the top-k kernel)
    ("scores_k24_decode", dict(B=2, Nq=1, Nk=300000, Hq=2, Hkv=2, d=64, d_idx=64, topk=24, q_offset=299999)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_noalloc_select_matches_workspace_entry_point_on_two_calls(name, kw):
    import torch
    from block_sparse_gqa_causal_gb300 import api
    fn = _noalloc_fn()
    stream = torch.cuda.current_stream()
    sh = api.Shape(**kw)
    for call in range(2):
        g = torch.Generator(device="cuda").manual_seed(1000 * call + sh.Nk + sh.topk)
        qi = torch.randn(sh.B, sh.Nq, sh.Hkv, sh.d_idx, device="cuda", generator=g).bfloat16()
        ki = torch.randn(sh.B, sh.Nk, sh.d_idx, device="cuda", generator=g).bfloat16()
        want = api.index_select(sh, qi, ki)
        got = torch.full_like(want, -7)
        rc = fn(ctypes.byref(sh.c()), qi.data_ptr(), ki.data_ptr(), got.data_ptr(), stream.cuda_stream)
        assert rc == 0, api.lib().msa_last_error()
        torch.cuda.synchronize()
        assert torch.equal(got, want), (name, call)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from block_sparse_gqa_causal_gb300 import api
    fn = _noalloc_fn()
    # topk > 16 keeps the block scores: 32768 x 8 groups x 256 blocks x 4 bytes = 256 MiB > 64 MiB
    sh = api.Shape(B=1, Nq=32768, Nk=32768, Hq=32, Hkv=8, d=128, d_idx=128, topk=24)
    rc = fn(ctypes.byref(sh.c()), None, None, None, None)
    assert rc == 3
    assert b"64 MiB" in api.lib().msa_last_error()
