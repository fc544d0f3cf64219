"""The C-ABI library builds, loads and exports every symbol include/msa.h
declares; host-side validation works without a GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libmsa():
    from block_sparse_gqa_causal_gb300 import build
    build.build()
    from block_sparse_gqa_causal_gb300 import api
    return api.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("msa_index_select", "msa_sparse_attn_fwd", "msa_kl_fwd", "msa_fused_bwd", "msa_workspace_size",
              "msa_last_error", "msa_check_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(libmsa):
    for n in declared_symbols():
        assert hasattr(libmsa, n), n


def test_version_and_workspace_sizes(libmsa):
    from block_sparse_gqa_causal_gb300 import api
    assert "sm_103a" in api.version()
    sh = api.Shape(B=1, Nq=131072, Nk=131072, Hq=64, Hkv=8, d=128, d_idx=128, topk=16)
    # topk <= 16 in prefill: the top-k runs inside the score kernel, so only the status word
    assert api.workspace_size(sh, api.OP_INDEX_SELECT) == 256
    # topk > 16: block scores B*Nq*Hkv*nb fp32 + status word
    sh24 = api.Shape(B=1, Nq=131072, Nk=131072, Hq=64, Hkv=8, d=128, d_idx=128, topk=24)
    assert api.workspace_size(sh24, api.OP_INDEX_SELECT) == 131072 * 8 * 1024 * 4 + 256
    # key-major forward: bf16 partial outputs per (query, head, selected block) + their (max, sum)
    assert api.workspace_size(sh, api.OP_SPARSE_ATTN_FWD) >= 131072 * 64 * 16 * (128 * 2 + 8)
    dec = api.Shape(B=4, Nq=1, Nk=1 << 20, Hq=64, Hkv=8, d=128, d_idx=128, topk=16, q_offset=(1 << 20) - 1)
    # decode: 32 (b, i, r) rows cannot fill the GPU, so each row's chunks are split over several CTAs
    # (at most 32 shares) whose fp32 partial outputs and (max, sum) are merged afterwards
    dec_ws = api.workspace_size(dec, api.OP_SPARSE_ATTN_FWD)
    assert 256 + 4 * 64 * 2 * (128 * 4 + 8) <= dec_ws <= 256 + 4 * 64 * 32 * (128 * 4 + 8) + 256
    assert api.workspace_size(sh, api.OP_KL_FWD) >= 131072 * 8 * 4


@pytest.mark.parametrize("field,value,code", [
    ("block", 64, 2), ("d", 96, 2), ("topk", 33, 2), ("Hkv", 3, 1), ("Nq", 0, 1), ("q_offset", 5, 1),
    ("Hq", 48, 2),
])
def test_invalid_shapes_are_rejected_before_any_launch(libmsa, field, value, code):
    from block_sparse_gqa_causal_gb300 import api
    sh = api.Shape(B=1, Nq=256, Nk=256, Hq=8, Hkv=2, d=64, d_idx=64, topk=4)
    setattr(sh, field, value)
    if field == "Hq":
        sh.Hkv = 3      # G = 16
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: validation fails first
    sel = ctypes.c_void_p(1 << 21)
    rc = libmsa.msa_index_select(ctypes.byref(sh.c()), fake, fake, sel, None, fake, 1 << 30, None)
    assert rc == code, (field, rc, libmsa.msa_last_error())
    assert libmsa.msa_last_error().decode()


def test_null_and_misaligned_pointers_are_rejected(libmsa):
    from block_sparse_gqa_causal_gb300 import api
    sh = api.Shape(B=1, Nq=256, Nk=256, Hq=8, Hkv=2, d=64, d_idx=64, topk=4)
    good = ctypes.c_void_p(1 << 20)
    rc = libmsa.msa_sparse_attn_fwd(ctypes.byref(sh.c()), None, good, good, good, good, good, good, 256, None)
    assert rc == 1 and b"q is NULL" in libmsa.msa_last_error()
    bad = ctypes.c_void_p((1 << 20) + 2)
    rc = libmsa.msa_sparse_attn_fwd(ctypes.byref(sh.c()), bad, good, good, good, good, good, good, 256, None)
    assert rc == 1 and b"aligned" in libmsa.msa_last_error()
    rc = libmsa.msa_sparse_attn_fwd(ctypes.byref(sh.c()), good, good, good, good, good, good, good, 16, None)
    assert rc == 3   # workspace too small


def test_block_mask_rejects_bad_arguments_before_any_launch(libmsa):
    from block_sparse_gqa_causal_gb300 import api
    sh = api.Shape(B=1, Nq=256, Nk=256, Hq=8, Hkv=2, d=64, d_idx=64, topk=4)
    good = ctypes.c_void_p(1 << 20)
    rc = libmsa.msa_block_mask(ctypes.byref(sh.c()), None, good, None, None, None)
    assert rc == 1 and b"non-NULL" in libmsa.msa_last_error()
    rc = libmsa.msa_block_mask(ctypes.byref(sh.c()), good, ctypes.c_void_p((1 << 20) + 2), None, None, None)
    assert rc == 1 and b"aligned" in libmsa.msa_last_error()
    big = api.Shape(B=1, Nq=1, Nk=700000 * 128, Hq=8, Hkv=2, d=64, d_idx=64, topk=4, q_offset=700000 * 128 - 1)
    rc = libmsa.msa_block_mask(ctypes.byref(big.c()), good, good, None, None, None)
    assert rc == 2 and b"655,328" in libmsa.msa_last_error()


def test_kv_append_rejects_bad_arguments_before_any_launch(libmsa):
    from block_sparse_gqa_causal_gb300 import api
    sh = api.Shape(B=2, Nq=1, Nk=501, Hq=8, Hkv=2, d=64, d_idx=128, topk=4, q_offset=500, kv_rows=1000)
    good = ctypes.c_void_p(1 << 20)
    # a half-given pair
    rc = libmsa.msa_kv_append(ctypes.byref(sh.c()), good, None, None, None, None, None, None)
    assert rc == 1 and b"both or neither" in libmsa.msa_last_error()
    rc = libmsa.msa_kv_append(ctypes.byref(sh.c()), None, None, None, None, None, None, None)
    assert rc == 1 and b"nothing to append" in libmsa.msa_last_error()
    bad = ctypes.c_void_p((1 << 20) + 8)
    rc = libmsa.msa_kv_append(ctypes.byref(sh.c()), good, good, good, good, good, bad, None)
    assert rc == 1 and b"aligned" in libmsa.msa_last_error()
    # the new rows must lie inside the cache: q_offset + Nq <= Nk <= kv_rows
    over = api.Shape(B=2, Nq=2, Nk=501, Hq=8, Hkv=2, d=64, d_idx=128, topk=4, q_offset=500, kv_rows=1000)
    rc = libmsa.msa_kv_append(ctypes.byref(over.c()), good, good, good, good, good, good, None)
    assert rc == 1 and b"exceeds Nk" in libmsa.msa_last_error()
    small = api.Shape(B=2, Nq=1, Nk=501, Hq=8, Hkv=2, d=64, d_idx=128, topk=4, q_offset=500, kv_rows=400)
    rc = libmsa.msa_kv_append(ctypes.byref(small.c()), good, good, good, good, good, good, None)
    assert rc == 1 and b"kv_rows" in libmsa.msa_last_error()


def test_bwd_rejects_non_training_layout(libmsa):
    from block_sparse_gqa_causal_gb300 import api
    sh = api.Shape(B=1, Nq=3, Nk=256, Hq=8, Hkv=2, d=64, d_idx=64, topk=4, q_offset=253)
    g = ctypes.c_void_p(1 << 20)
    rc = libmsa.msa_fused_bwd(ctypes.byref(sh.c()), g, g, g, g, g, g, g, g, g, g, ctypes.c_float(1.0),
                              g, g, g, g, g, g, 1 << 30, None)
    assert rc == 2


def test_train_step_staged_rejects_bad_arguments_before_any_launch(libmsa):
    """The staged training step validates like msa_train_step: a non-training
    layout, a NULL input and a short workspace are refused on the host (the
    event pointers are never touched on these paths)."""
    from block_sparse_gqa_causal_gb300 import api
    g = ctypes.c_void_p(1 << 20)
    ev = ctypes.c_void_p(1 << 12)
    f = ctypes.c_float(1.0)
    chunked = api.Shape(B=1, Nq=3, Nk=256, Hq=8, Hkv=2, d=64, d_idx=64, topk=4, q_offset=253)
    rc = libmsa.msa_train_step_staged(ctypes.byref(chunked.c()), g, g, g, g, g, g, f, g, g, g, g, None, g, g, g, g, g,
                                      g, ev, ev, ev, g, 1 << 30, None)
    assert rc == 2 and b"train_step" in libmsa.msa_last_error()
    sh = api.Shape(B=1, Nq=256, Nk=256, Hq=8, Hkv=2, d=64, d_idx=64, topk=4)
    rc = libmsa.msa_train_step_staged(ctypes.byref(sh.c()), None, g, g, g, g, g, f, g, g, g, g, None, g, g, g, g, g,
                                      g, ev, ev, ev, g, 1 << 30, None)
    assert rc == 1 and b"q is NULL" in libmsa.msa_last_error()
    rc = libmsa.msa_train_step_staged(ctypes.byref(sh.c()), g, g, g, g, g, g, f, g, g, g, g, None, g, g, g, g, g,
                                      g, None, None, None, g, 256, None)
    assert rc == 3


def test_product_path_has_no_oracle_or_fallback():
    """The library binding never imports the oracle and has no CPU path."""
    pkg = os.path.join(ROOT, "block_sparse_gqa_causal_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "msa_oracle" not in text, f


@pytest.mark.parametrize("d,di", [(128, 128), (64, 64), (128, 64)])
def test_backward_workspace_holds_no_distribution(libmsa, d, di):
    """The fused backward's workspace (the tensor-core path, at every head
    dim) is D, one fp32 dK_idx share per group, the inverse index and the
    per-slot dQ / dq_idx partial rows -- nothing per (slot, key): the teacher
    is rebuilt on chip and never stored.  With the KL loss, four floats per
    slot more."""
    from block_sparse_gqa_causal_gb300 import api
    B, N, Hq, Hkv, k = 1, 131072, 64, 8, 16
    sh = api.Shape(B=B, Nq=N, Nk=N, Hq=Hq, Hkv=Hkv, d=d, d_idx=di, topk=k)
    a = lambda x: (x + 255) // 256 * 256
    nb = N // 128
    nct = (N + 511) // 512
    index = 2 * a((B * Hkv * nb + 1) * 4) + a(2 * B * Hkv * nct * nb * 4) + a(B * Hkv * N * k * 4)
    slots = B * N * k
    want = (256 + a(B * Hq * N * 4) + a(B * Hkv * N * di * 4) + index + a(slots * Hq * d * 2)
            + a(slots * Hkv * di * 2))
    assert api.workspace_size(sh, api.OP_FUSED_BWD) == want
    assert api.workspace_size(sh, api.OP_FUSED_BWD_KL) == want + a(B * Hkv * N * 4) + a(slots * Hkv * 16)


def test_training_step_phases_share_one_workspace_region(libmsa):
    """msa_train_step keeps the inverse index and D for the whole step and
    overlays the phases' own buffers in one region -- the forward's partial
    rows, the KL index pass's partials, the backward's dK_idx shares, partial
    rows and KL terms -- since each phase's partials are combined before the
    next phase writes: at 128K the region is the larger of the forward's and
    the backward's buffers, not their sum."""
    from block_sparse_gqa_causal_gb300 import api
    B, N, Hq, Hkv, d, di, k = 1, 131072, 64, 8, 128, 128, 16
    sh = api.Shape(B=B, Nq=N, Nk=N, Hq=Hq, Hkv=Hkv, d=d, d_idx=di, topk=k)
    a = lambda x: (x + 255) // 256 * 256
    nb = N // 128
    nct = (N + 511) // 512
    index = 2 * a((B * Hkv * nb + 1) * 4) + a(2 * B * Hkv * nct * nb * 4) + a(B * Hkv * N * k * 4)
    rows, slots = B * N * Hq * k, B * N * k
    fwd = a(rows * d * 2) + a(rows * 8)
    bwd = a(B * Hkv * N * di * 4) + a(slots * Hq * d * 2) + a(slots * Hkv * di * 2) + a(B * Hkv * N * 4) \
        + a(slots * Hkv * 16)
    want = 256 + index + a(B * Hq * N * 4) + max(fwd, bwd)
    assert api.workspace_size(sh, api.OP_TRAIN_STEP) == want
    assert want < 40e9      # the forward's 35.4 GB of partial rows and the backward's 39.5 GB are never live together


def test_warmup_and_projection_calls_validate_on_the_host(libmsa):
    """The dense warm-up needs a training sequence of at most 32 blocks; the
    projections need d_idx in {64, 128} and Dm a multiple of 8; bad pointers
    and short workspaces are refused before any launch."""
    from block_sparse_gqa_causal_gb300 import api
    g = ctypes.c_void_p(1 << 20)
    f = ctypes.c_float(1.0)
    for kw in (dict(Nq=8192, Nk=8192), dict(Nq=3, Nk=256, q_offset=253)):
        base = dict(B=1, Nq=1024, Nk=1024, Hq=8, Hkv=2, d=128, d_idx=128, topk=1)
        base.update(kw)
        sh = api.Shape(**base)
        assert api.lib().msa_workspace_size(ctypes.byref(sh.c()), api.OP_WARMUP_KL) == 0
        assert b"at most 32 blocks" in libmsa.msa_last_error()
        rc = libmsa.msa_warmup_kl(ctypes.byref(sh.c()), g, g, g, g, g, f, g, g, g, g, g, g, g, 1 << 40, None)
        assert rc == 2, (kw, libmsa.msa_last_error())
    sh = api.Shape(B=1, Nq=1024, Nk=1024, Hq=8, Hkv=2, d=128, d_idx=128, topk=1)
    assert api.workspace_size(sh, api.OP_WARMUP_KL) > 0
    rc = libmsa.msa_warmup_kl(ctypes.byref(sh.c()), None, g, g, g, g, f, g, g, g, g, g, g, g, 1 << 40, None)
    assert rc == 1 and b"q is NULL" in libmsa.msa_last_error()
    rc = libmsa.msa_warmup_kl(ctypes.byref(sh.c()), g, g, g, g, g, f, g, g, g, g, g, g, g, 256, None)
    assert rc == 3
    for T, Dm, Hkv, di, code in ((100, 256, 2, 96, 2), (100, 250, 2, 128, 2), (0, 256, 2, 128, 1)):
        ps = api.ProjShape(T=T, Dm=Dm, Hkv=Hkv, d_idx=di)
        rc = libmsa.msa_index_proj_fwd(ctypes.byref(ps.c()), g, g, g, g, g, g, 1 << 20, None)
        assert rc == code, (T, Dm, di, libmsa.msa_last_error())
    ps = api.ProjShape(T=20000, Dm=256, Hkv=2, d_idx=128)
    need = libmsa.msa_index_proj_workspace_size(ctypes.byref(ps.c()))
    assert need >= 256 + 256 * 384 * 4                  # at least one fp32 partial of [Dm][Hkv*d_idx + d_idx]
    rc = libmsa.msa_index_proj_bwd(ctypes.byref(ps.c()), g, g, g, g, g, g, 256, None)
    assert rc == 3
