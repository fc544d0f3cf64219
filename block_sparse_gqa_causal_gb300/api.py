"""Thin Python binding of libmsa.so (C-ABI in include/msa.h).

Argument marshalling only: it checks dtypes and layouts, allocates outputs
and workspaces with torch (device memory), and passes raw pointers and the
current CUDA stream to the library.  Every step of the computation runs in
the library's kernels; there is no fallback.  If libmsa.so has not been
built, the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

OP_INDEX_SELECT, OP_SPARSE_ATTN_FWD, OP_KL_FWD, OP_FUSED_BWD, OP_FUSED_BWD_KL, OP_TRAIN_STEP = 0, 1, 2, 3, 4, 5
OP_WARMUP_KL = 6
STATUS = {0: "MSA_OK", 1: "MSA_ERR_INVALID_ARGUMENT", 2: "MSA_ERR_UNSUPPORTED", 3: "MSA_ERR_WORKSPACE",
          4: "MSA_ERR_CUDA", 5: "MSA_ERR_TIMEOUT", 6: "MSA_ERR_DEVICE"}
EXPORTS = ("msa_workspace_size", "msa_index_select", "msa_sparse_attn_fwd", "msa_kl_fwd", "msa_fused_bwd",
           "msa_fused_bwd_kl", "msa_train_step", "msa_train_step_staged", "msa_block_mask", "msa_warmup_kl",
           "msa_index_proj_workspace_size", "msa_index_proj_fwd", "msa_index_proj_bwd", "msa_kv_append",
           "msa_last_error", "msa_check_device_status", "msa_version", "msa_launch_count")


class MsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class _CProjShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("T", "Dm", "Hkv", "d_idx")]


@dataclass
class ProjShape:
    """msa_proj_shape: T tokens of Dm features projected to Hkv index queries
    and one index key of d_idx features each."""
    T: int
    Dm: int
    Hkv: int
    d_idx: int

    def c(self) -> _CProjShape:
        return _CProjShape(self.T, self.Dm, self.Hkv, self.d_idx)


class _CShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("B", "Nq", "Nk", "q_offset", "Hq", "Hkv", "d", "d_idx", "block", "topk")] + [
        ("kv_rows", ctypes.c_longlong), ("scale", ctypes.c_float), ("scale_idx", ctypes.c_float)]


@dataclass
class Shape:
    """msa_shape: see include/msa.h for the meaning of each field."""
    B: int
    Nq: int
    Nk: int
    Hq: int
    Hkv: int
    d: int
    d_idx: int
    topk: int
    block: int = 128
    q_offset: int = 0
    kv_rows: int = 0
    scale: float = 0.0
    scale_idx: float = 0.0

    @property
    def nb(self) -> int:
        return (self.Nk + self.block - 1) // self.block

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def rows_kv(self) -> int:
        return self.kv_rows or self.Nk

    def c(self) -> _CShape:
        return _CShape(self.B, self.Nq, self.Nk, self.q_offset, self.Hq, self.Hkv, self.d, self.d_idx, self.block,
                       self.topk, self.kv_rows, self.scale, self.scale_idx)


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libmsa.so (fails loudly if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            P, S = ctypes.c_void_p, ctypes.POINTER(_CShape)
            sz, f = ctypes.c_size_t, ctypes.c_float
            L.msa_workspace_size.argtypes = [S, ctypes.c_int]
            L.msa_workspace_size.restype = sz
            L.msa_index_select.argtypes = [S, P, P, P, P, P, sz, P]
            L.msa_sparse_attn_fwd.argtypes = [S, P, P, P, P, P, P, P, sz, P]
            L.msa_kl_fwd.argtypes = [S, P, P, P, P, P, P, f, P, P, P, P, sz, P]
            L.msa_fused_bwd.argtypes = [S, P, P, P, P, P, P, P, P, P, P, f, P, P, P, P, P, P, sz, P]
            L.msa_fused_bwd_kl.argtypes = [S, P, P, P, P, P, P, P, P, P, P, f, P, P, P, P, P, P, P, P, sz, P]
            L.msa_train_step.argtypes = [S, P, P, P, P, P, P, f, P, P, P, P, P, P, P, P, P, P, P, P, sz, P]
            L.msa_train_step_staged.argtypes = [S, P, P, P, P, P, P, f, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P,
                                                sz, P]
            L.msa_check_device_status.argtypes = [P, P]
            L.msa_block_mask.argtypes = [S, P, P, P, P, P]
            L.msa_kv_append.argtypes = [S, P, P, P, P, P, P, P]
            L.msa_warmup_kl.argtypes = [S, P, P, P, P, P, f, P, P, P, P, P, P, P, sz, P]
            PS = ctypes.POINTER(_CProjShape)
            L.msa_index_proj_workspace_size.argtypes = [PS]
            L.msa_index_proj_workspace_size.restype = sz
            L.msa_index_proj_fwd.argtypes = [PS, P, P, P, P, P, P, sz, P]
            L.msa_index_proj_bwd.argtypes = [PS, P, P, P, P, P, P, sz, P]
            L.msa_selftest_wait_timeout.argtypes = [P, ctypes.c_uint, P]
            for fn in ("msa_index_select", "msa_sparse_attn_fwd", "msa_kl_fwd", "msa_fused_bwd", "msa_fused_bwd_kl",
                       "msa_train_step", "msa_train_step_staged", "msa_check_device_status", "msa_block_mask",
                       "msa_warmup_kl", "msa_index_proj_fwd", "msa_index_proj_bwd", "msa_selftest_wait_timeout",
                       "msa_kv_append"):
                getattr(L, fn).restype = ctypes.c_int
            L.msa_last_error.restype = ctypes.c_char_p
            L.msa_version.restype = ctypes.c_char_p
            L.msa_launch_count.restype = ctypes.c_ulonglong
            L.msa_kernel_timing.argtypes = [ctypes.c_int]
            L.msa_kernel_timing.restype = ctypes.c_int
            L.msa_kernel_timing_report.argtypes = [ctypes.c_char_p, sz]
            L.msa_kernel_timing_report.restype = sz
            _lib = L
        return _lib


def _check(code: int) -> None:
    if code != 0:
        raise MsaError(code, lib().msa_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, shape, dtype) -> None:
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: need a contiguous CUDA {dtype} tensor of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)} contiguous={t.is_contiguous()} cuda={t.is_cuda}")


def workspace_size(shape: Shape, op: int) -> int:
    n = lib().msa_workspace_size(ctypes.byref(shape.c()), op)
    if n == 0:
        _check(1)
    return int(n)


def new_workspace(shape: Shape, op: int, device=None) -> torch.Tensor:
    """A workspace with its 256-byte status word zeroed."""
    n = workspace_size(shape, op)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    ws[:256].zero_()
    return ws


def _ws(ws, shape, op, device):
    if ws is None:
        ws = new_workspace(shape, op, device)
    return ws


def index_select(shape: Shape, q_idx, k_idx, *, sel_idx=None, block_scores=None, return_scores=False,
                 workspace=None, stream=None):
    """msa_index_select.  Returns sel_idx [B,Hkv,Nq,topk] int32 (and the block
    scores [B,Nq,Hkv,nb] fp32 when asked for)."""
    s = shape
    _need(q_idx, "q_idx", (s.B, s.Nq, s.Hkv, s.d_idx), torch.bfloat16)
    _need(k_idx, "k_idx", (s.B, s.rows_kv, s.d_idx), torch.bfloat16)
    dev = q_idx.device
    if sel_idx is None:
        sel_idx = torch.empty((s.B, s.Hkv, s.Nq, s.topk), dtype=torch.int32, device=dev)
    if return_scores and block_scores is None:
        block_scores = torch.empty((s.B, s.Nq, s.Hkv, s.nb), dtype=torch.float32, device=dev)
    ws = _ws(workspace, s, OP_INDEX_SELECT, dev)
    _check(lib().msa_index_select(ctypes.byref(s.c()), _ptr(q_idx), _ptr(k_idx), _ptr(sel_idx), _ptr(block_scores),
                                  _ptr(ws), ws.numel(), _stream(stream)))
    return (sel_idx, block_scores) if return_scores else sel_idx


def sparse_attn_fwd(shape: Shape, q, k, v, sel_idx, *, o=None, lse=None, workspace=None, stream=None):
    """msa_sparse_attn_fwd.  Returns (o [B,Nq,Hq,d] bf16, lse [B,Hq,Nq] fp32)."""
    s = shape
    _need(q, "q", (s.B, s.Nq, s.Hq, s.d), torch.bfloat16)
    _need(k, "k", (s.B, s.rows_kv, s.Hkv, s.d), torch.bfloat16)
    _need(v, "v", (s.B, s.rows_kv, s.Hkv, s.d), torch.bfloat16)
    _need(sel_idx, "sel_idx", (s.B, s.Hkv, s.Nq, s.topk), torch.int32)
    dev = q.device
    o = torch.empty((s.B, s.Nq, s.Hq, s.d), dtype=torch.bfloat16, device=dev) if o is None else o
    lse = torch.empty((s.B, s.Hq, s.Nq), dtype=torch.float32, device=dev) if lse is None else lse
    ws = _ws(workspace, s, OP_SPARSE_ATTN_FWD, dev)
    _check(lib().msa_sparse_attn_fwd(ctypes.byref(s.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(sel_idx), _ptr(o),
                                     _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))
    return o, lse


def kl_fwd(shape: Shape, q, k, q_idx, k_idx, sel_idx, lse, kl_coef: float = 1.0, *, lse_idx=None, kl_rows=None,
           kl_loss=None, want_rows=True, lse_only=False, workspace=None, stream=None):
    """msa_kl_fwd.  Returns (kl_loss scalar tensor, lse_idx [B,Hkv,Nq], kl_rows [B,Hkv,Nq] or None).
    lse_only: compute lse_idx alone (kl_loss and kl_rows are None); the
    training step's form, whose loss then comes from fused_bwd(..., with_kl=True)."""
    s = shape
    _need(q, "q", (s.B, s.Nq, s.Hq, s.d), torch.bfloat16)
    _need(k, "k", (s.B, s.rows_kv, s.Hkv, s.d), torch.bfloat16)
    _need(q_idx, "q_idx", (s.B, s.Nq, s.Hkv, s.d_idx), torch.bfloat16)
    _need(k_idx, "k_idx", (s.B, s.rows_kv, s.d_idx), torch.bfloat16)
    _need(sel_idx, "sel_idx", (s.B, s.Hkv, s.Nq, s.topk), torch.int32)
    _need(lse, "lse", (s.B, s.Hq, s.Nq), torch.float32)
    dev = q.device
    lse_idx = torch.empty((s.B, s.Hkv, s.Nq), dtype=torch.float32, device=dev) if lse_idx is None else lse_idx
    if lse_only:
        kl_rows = kl_loss = None
    else:
        if want_rows and kl_rows is None:
            kl_rows = torch.empty((s.B, s.Hkv, s.Nq), dtype=torch.float32, device=dev)
        kl_loss = torch.empty((), dtype=torch.float32, device=dev) if kl_loss is None else kl_loss
    ws = _ws(workspace, s, OP_KL_FWD, dev)
    _check(lib().msa_kl_fwd(ctypes.byref(s.c()), _ptr(q), _ptr(k), _ptr(q_idx), _ptr(k_idx), _ptr(sel_idx),
                            _ptr(lse), ctypes.c_float(kl_coef), _ptr(lse_idx), _ptr(kl_rows), _ptr(kl_loss),
                            _ptr(ws), ws.numel(), _stream(stream)))
    return kl_loss, lse_idx, kl_rows


def fused_bwd(shape: Shape, q, k, v, o, d_o, lse, q_idx, k_idx, sel_idx, lse_idx, kl_coef: float = 1.0, *,
              grads=None, with_kl=False, kl_rows=None, kl_loss=None, workspace=None, stream=None):
    """msa_fused_bwd.  Returns (dq, dk, dv, dq_idx, dk_idx) bf16.
    with_kl: msa_fused_bwd_kl, which also gives the step's KL loss; returns
    (dq, dk, dv, dq_idx, dk_idx, kl_loss, kl_rows), kl_rows None unless a
    [B,Hkv,Nq] fp32 tensor is passed for it."""
    s = shape
    for t, n, shp in ((q, "q", (s.B, s.Nq, s.Hq, s.d)), (o, "o", (s.B, s.Nq, s.Hq, s.d)),
                      (d_o, "d_o", (s.B, s.Nq, s.Hq, s.d)), (k, "k", (s.B, s.Nk, s.Hkv, s.d)),
                      (v, "v", (s.B, s.Nk, s.Hkv, s.d)), (q_idx, "q_idx", (s.B, s.Nq, s.Hkv, s.d_idx)),
                      (k_idx, "k_idx", (s.B, s.Nk, s.d_idx))):
        _need(t, n, shp, torch.bfloat16)
    _need(lse, "lse", (s.B, s.Hq, s.Nq), torch.float32)
    _need(lse_idx, "lse_idx", (s.B, s.Hkv, s.Nq), torch.float32)
    _need(sel_idx, "sel_idx", (s.B, s.Hkv, s.Nq, s.topk), torch.int32)
    if grads is None:
        grads = tuple(torch.empty_like(t) for t in (q, k, v, q_idx, k_idx))
    dq, dk, dv, dqi, dki = grads
    if with_kl:
        kl_loss = torch.empty((), dtype=torch.float32, device=q.device) if kl_loss is None else kl_loss
        if kl_rows is not None:
            _need(kl_rows, "kl_rows", (s.B, s.Hkv, s.Nq), torch.float32)
        ws = _ws(workspace, s, OP_FUSED_BWD_KL, q.device)
        _check(lib().msa_fused_bwd_kl(ctypes.byref(s.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(d_o), _ptr(lse),
                                      _ptr(q_idx), _ptr(k_idx), _ptr(sel_idx), _ptr(lse_idx), ctypes.c_float(kl_coef),
                                      _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dqi), _ptr(dki), _ptr(kl_rows), _ptr(kl_loss),
                                      _ptr(ws), ws.numel(), _stream(stream)))
        return dq, dk, dv, dqi, dki, kl_loss, kl_rows
    ws = _ws(workspace, s, OP_FUSED_BWD, q.device)
    _check(lib().msa_fused_bwd(ctypes.byref(s.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(d_o), _ptr(lse),
                               _ptr(q_idx), _ptr(k_idx), _ptr(sel_idx), _ptr(lse_idx), ctypes.c_float(kl_coef),
                               _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dqi), _ptr(dki), _ptr(ws), ws.numel(),
                               _stream(stream)))
    return dq, dk, dv, dqi, dki


def train_step(shape: Shape, q, k, v, q_idx, k_idx, d_o, kl_coef: float = 1.0, *, out=None, workspace=None,
               stream=None, input_ready=None):
    """msa_train_step: selection, forward, lse_idx, fused backward with the KL loss in one call.
    Returns a dict with sel, o, lse, lse_idx, kl_rows, kl_loss, dq, dk, dv, dq_idx, dk_idx
    (pass `out`, a dict of preallocated tensors with those keys, to reuse buffers).
    input_ready: three torch.cuda.Events (or None each), recorded after the writes
    of (q_idx, k_idx), (q, k, v) and d_o: msa_train_step_staged, whose stream waits
    on each just before the first phase reading those inputs."""
    s = shape
    for t, n, shp in ((q, "q", (s.B, s.Nq, s.Hq, s.d)), (d_o, "d_o", (s.B, s.Nq, s.Hq, s.d)),
                      (k, "k", (s.B, s.Nk, s.Hkv, s.d)), (v, "v", (s.B, s.Nk, s.Hkv, s.d)),
                      (q_idx, "q_idx", (s.B, s.Nq, s.Hkv, s.d_idx)), (k_idx, "k_idx", (s.B, s.Nk, s.d_idx))):
        _need(t, n, shp, torch.bfloat16)
    dev = q.device
    if out is None:
        out = {"sel": torch.empty((s.B, s.Hkv, s.Nq, s.topk), dtype=torch.int32, device=dev),
               "o": torch.empty_like(q), "lse": torch.empty((s.B, s.Hq, s.Nq), dtype=torch.float32, device=dev),
               "lse_idx": torch.empty((s.B, s.Hkv, s.Nq), dtype=torch.float32, device=dev),
               "kl_rows": torch.empty((s.B, s.Hkv, s.Nq), dtype=torch.float32, device=dev),
               "kl_loss": torch.empty((), dtype=torch.float32, device=dev),
               "dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
               "dq_idx": torch.empty_like(q_idx), "dk_idx": torch.empty_like(k_idx)}
    ws = _ws(workspace, s, OP_TRAIN_STEP, dev)
    args = [ctypes.byref(s.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx), _ptr(d_o),
            ctypes.c_float(kl_coef), _ptr(out["sel"]), _ptr(out["o"]), _ptr(out["lse"]), _ptr(out["lse_idx"]),
            _ptr(out.get("kl_rows")), _ptr(out["kl_loss"]), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
            _ptr(out["dq_idx"]), _ptr(out["dk_idx"])]
    if input_ready is None:
        _check(lib().msa_train_step(*args, _ptr(ws), ws.numel(), _stream(stream)))
    else:
        evs = [None if ev is None else ctypes.c_void_p(ev.cuda_event) for ev in input_ready]
        _check(lib().msa_train_step_staged(*args, *evs, _ptr(ws), ws.numel(), _stream(stream)))
    return out


def block_mask(shape: Shape, sel_idx, *, counts=False, blocks=False, stream=None):
    """msa_block_mask.  Returns the mask words [B, Hkv, ceil(Nq/128),
    ceil(nb/32)] as int32 (the uint32 bit patterns), plus the per-tile
    active-block counts [B, Hkv, T] and the ascending active-block lists
    [B, Hkv, T, nb] (-1 padded) when asked for."""
    s = shape
    _need(sel_idx, "sel_idx", (s.B, s.Hkv, s.Nq, s.topk), torch.int32)
    T, W = (s.Nq + 127) // 128, (s.nb + 31) // 32
    dev = sel_idx.device
    mask = torch.empty((s.B, s.Hkv, T, W), dtype=torch.int32, device=dev)
    cnt = torch.empty((s.B, s.Hkv, T), dtype=torch.int32, device=dev) if counts else None
    blk = torch.empty((s.B, s.Hkv, T, s.nb), dtype=torch.int32, device=dev) if blocks else None
    _check(lib().msa_block_mask(ctypes.byref(s.c()), _ptr(sel_idx), _ptr(mask), _ptr(cnt), _ptr(blk),
                                _stream(stream)))
    out = (mask,) + ((cnt,) if counts else ()) + ((blk,) if blocks else ())
    return out[0] if len(out) == 1 else out


def kv_append(shape: Shape, k_new, v_new, k_idx_new, k, v, k_idx, *, stream=None) -> None:
    """msa_kv_append: the Nq new tokens' K, V [B, Nq, Hkv, d] and K_idx
    [B, Nq, d_idx] rows into the caches k, v [B, kv_rows, Hkv, d] and k_idx
    [B, kv_rows, d_idx] at rows q_offset .. q_offset+Nq-1 (a pair given as
    None, None is skipped)."""
    s = shape
    for new, cache, row in ((k_new, k, (s.Hkv, s.d)), (v_new, v, (s.Hkv, s.d)), (k_idx_new, k_idx, (s.d_idx,))):
        if new is not None:
            _need(new, "new rows", (s.B, s.Nq) + row, torch.bfloat16)
        if cache is not None:
            _need(cache, "cache", (s.B, s.rows_kv) + row, torch.bfloat16)
    _check(lib().msa_kv_append(ctypes.byref(s.c()), _ptr(k_new), _ptr(v_new), _ptr(k_idx_new), _ptr(k), _ptr(v),
                               _ptr(k_idx), _stream(stream)))


def check_device_status(workspace, stream=None) -> None:
    """msa_check_device_status: raises MsaError on a recorded device-side error."""
    _check(lib().msa_check_device_status(_ptr(workspace), _stream(stream)))


def kernel_timing(enable: bool) -> bool:
    """msa_kernel_timing: bracket each library kernel with CUDA events on its
    stream while enabled (clears earlier records); returns the previous setting."""
    return bool(lib().msa_kernel_timing(1 if enable else 0))


def kernel_times() -> dict:
    """msa_kernel_timing_report: {kernel name: (launches, total ms)} of the
    launches recorded since timing was last switched."""
    L = lib()
    need = int(L.msa_kernel_timing_report(None, 0))
    buf = ctypes.create_string_buffer(need)
    L.msa_kernel_timing_report(buf, need)
    out = {}
    for line in buf.value.decode().splitlines():
        name, n, ms = line.split()
        out[name] = (int(n), float(ms))
    return out


def launch_count() -> int:
    """Kernels launched through the library by this process so far."""
    return int(lib().msa_launch_count())


def version() -> str:
    return lib().msa_version().decode()


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def warmup_kl(shape: Shape, q, k, v, q_idx, k_idx, kl_coef: float = 1.0, *, out=None, workspace=None, stream=None):
    """msa_warmup_kl: the dense indexer warm-up loss and its gradient in the
    index inputs.  Returns a dict with lse [B,Hq,Nq], lse_idx, kl_rows
    [B,Hkv,Nq], kl_loss (scalar), dq_idx, dk_idx (bf16)."""
    s = shape
    for t, n, shp in ((q, "q", (s.B, s.Nq, s.Hq, s.d)), (k, "k", (s.B, s.Nk, s.Hkv, s.d)),
                      (v, "v", (s.B, s.Nk, s.Hkv, s.d)), (q_idx, "q_idx", (s.B, s.Nq, s.Hkv, s.d_idx)),
                      (k_idx, "k_idx", (s.B, s.Nk, s.d_idx))):
        _need(t, n, shp, torch.bfloat16)
    dev = q.device
    if out is None:
        f32 = dict(dtype=torch.float32, device=dev)
        out = {"lse": torch.empty((s.B, s.Hq, s.Nq), **f32), "lse_idx": torch.empty((s.B, s.Hkv, s.Nq), **f32),
               "kl_rows": torch.empty((s.B, s.Hkv, s.Nq), **f32), "kl_loss": torch.empty((), **f32),
               "dq_idx": torch.empty_like(q_idx), "dk_idx": torch.empty_like(k_idx)}
    ws = _ws(workspace, s, OP_WARMUP_KL, dev)
    _check(lib().msa_warmup_kl(ctypes.byref(s.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(q_idx), _ptr(k_idx),
                               ctypes.c_float(kl_coef), _ptr(out["lse"]), _ptr(out["lse_idx"]), _ptr(out["kl_rows"]),
                               _ptr(out["kl_loss"]), _ptr(out["dq_idx"]), _ptr(out["dk_idx"]), _ptr(ws), ws.numel(),
                               _stream(stream)))
    return out


def proj_workspace(shape: ProjShape, device=None) -> torch.Tensor:
    n = lib().msa_index_proj_workspace_size(ctypes.byref(shape.c()))
    if n == 0:
        _check(1)
    ws = torch.empty(int(n), dtype=torch.uint8, device=device or "cuda")
    ws[:256].zero_()
    return ws


def index_proj_fwd(shape: ProjShape, x, wq_idx, wk_idx, *, q_idx=None, k_idx=None, workspace=None, stream=None):
    """msa_index_proj_fwd: q_idx [T, Hkv, d_idx], k_idx [T, d_idx] (bf16) of x [T, Dm]."""
    s = shape
    _need(x, "x", (s.T, s.Dm), torch.bfloat16)
    _need(wq_idx, "wq_idx", (s.Dm, s.Hkv * s.d_idx), torch.bfloat16)
    _need(wk_idx, "wk_idx", (s.Dm, s.d_idx), torch.bfloat16)
    dev = x.device
    q_idx = torch.empty((s.T, s.Hkv, s.d_idx), dtype=torch.bfloat16, device=dev) if q_idx is None else q_idx
    k_idx = torch.empty((s.T, s.d_idx), dtype=torch.bfloat16, device=dev) if k_idx is None else k_idx
    ws = proj_workspace(s, dev) if workspace is None else workspace
    _check(lib().msa_index_proj_fwd(ctypes.byref(s.c()), _ptr(x), _ptr(wq_idx), _ptr(wk_idx), _ptr(q_idx),
                                    _ptr(k_idx), _ptr(ws), ws.numel(), _stream(stream)))
    return q_idx, k_idx


def index_proj_bwd(shape: ProjShape, x, dq_idx, dk_idx, *, dwq=None, dwk=None, workspace=None, stream=None):
    """msa_index_proj_bwd: dwq [Dm, Hkv*d_idx], dwk [Dm, d_idx] (fp32); x gets no gradient."""
    s = shape
    _need(x, "x", (s.T, s.Dm), torch.bfloat16)
    _need(dq_idx, "dq_idx", (s.T, s.Hkv, s.d_idx), torch.bfloat16)
    _need(dk_idx, "dk_idx", (s.T, s.d_idx), torch.bfloat16)
    dev = x.device
    dwq = torch.empty((s.Dm, s.Hkv * s.d_idx), dtype=torch.float32, device=dev) if dwq is None else dwq
    dwk = torch.empty((s.Dm, s.d_idx), dtype=torch.float32, device=dev) if dwk is None else dwk
    ws = proj_workspace(s, dev) if workspace is None else workspace
    _check(lib().msa_index_proj_bwd(ctypes.byref(s.c()), _ptr(x), _ptr(dq_idx), _ptr(dk_idx), _ptr(dwq), _ptr(dwk),
                                    _ptr(ws), ws.numel(), _stream(stream)))
    return dwq, dwk


def selftest_wait_timeout(workspace, spin_limit: int = 4096, stream=None) -> None:
    """msa_selftest_wait_timeout: one thread's bounded wait on a barrier that
    nothing arrives on runs out and is recorded in the workspace's status word."""
    _check(lib().msa_selftest_wait_timeout(_ptr(workspace), int(spin_limit), _stream(stream)))
