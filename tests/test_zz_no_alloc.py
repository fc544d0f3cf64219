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


def test_noalloc_select_matches_workspace_entry_point_on_two_calls():
    import torch
    from block_sparse_gqa_causal_gb300 import api
    fn = _noalloc_fn()
    stream = torch.cuda.current_stream()
    cases = [
        (api.Shape(B=2, Nq=1000, Nk=1000, Hq=8, Hkv=2, d=64, d_idx=64, topk=4), 1),
        (api.Shape(B=1, Nq=3000, Nk=3000, Hq=32, Hkv=8, d=128, d_idx=128, topk=16), 2),
    ]
    for sh, seed in cases:
        g = torch.Generator(device="cuda").manual_seed(seed)
        qi = torch.randn(sh.B, sh.Nq, sh.Hkv, sh.d_idx, device="cuda", generator=g).bfloat16()
        ki = torch.randn(sh.B, sh.Nk, sh.d_idx, device="cuda", generator=g).bfloat16()
        want = api.index_select(sh, qi, ki)
        got = torch.full_like(want, -7)
        rc = fn(ctypes.byref(sh.c()), qi.data_ptr(), ki.data_ptr(), got.data_ptr(), stream.cuda_stream)
        assert rc == 0, api.lib().msa_last_error()
        torch.cuda.synchronize()
        assert torch.equal(got, want)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from block_sparse_gqa_causal_gb300 import api
    fn = _noalloc_fn()
    # 32768 x 8 groups x 256 blocks x 4 bytes = 256 MiB of block scores > 64 MiB
    sh = api.Shape(B=1, Nq=32768, Nk=32768, Hq=32, Hkv=8, d=128, d_idx=128, topk=16)
    rc = fn(ctypes.byref(sh.c()), None, None, None, None)
    assert rc == 3
    assert b"64 MiB" in api.lib().msa_last_error()
