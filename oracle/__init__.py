"""CPU oracle for the MSA hot path -- TEST INFRASTRUCTURE ONLY.

A plain fp64 C implementation (msa_oracle.c) of what the path computes,
written from "Sparse Attention · Part II", section 3.2 (MiniMax's MSA),
loaded through ctypes.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may use it; the library never does.  It shares no code
with the CUDA library.

Two builds of the same source: liboracle_bf16.so takes bf16 bit patterns
(uint16), liboracle_f64.so takes float64 inputs (finite-difference checks).

Also: the index projections of the detached hidden states (section 3.2's
detachment equation) with their weight gradient, and the dense indexer
warm-up loss (section 3.1) with its gradient in the index inputs.

Parity pins (tests/test_oracle.py): brute-force block max-pool and a full
sort for selection; the block-mask word of section 4.3's worked example
(tests/golden/) and set unions for the mask and its traversal; dense causal GQA attention when every visible block is
selected; dense attention under an explicit block mask; the renormalisation
error bound of section 2; KL >= 0, KL = 0 for a built teacher == student
case and KL against scipy's relative entropy; gradients against central
finite differences and against torch autograd on masked dense attention.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIBS = {"bf16": os.path.join(_HERE, "liboracle_bf16.so"), "f64": os.path.join(_HERE, "liboracle_f64.so")}
_lock = threading.Lock()
_loaded: dict = {}


def build(force: bool = False) -> None:
    """Compile both oracle variants with gcc + OpenMP (no GPU involved)."""
    for kind, out in _LIBS.items():
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
            continue
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-o", out + ".tmp", _SRC, "-lm"]
        if kind == "f64":
            cmd.insert(1, "-DORC_F64")
        subprocess.check_call(cmd)
        os.replace(out + ".tmp", out)


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("B", "Nq", "Nk", "q_offset", "Hq", "Hkv", "d", "d_idx", "block", "topk")] + [
        ("kv_rows", ctypes.c_longlong), ("scale", ctypes.c_double), ("scale_idx", ctypes.c_double)]


@dataclass
class Shape:
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
    kv_rows: int = 0          # rows per batch entry of k, v, k_idx (0 -> Nk)
    scale: float = 0.0        # 0 -> 1/sqrt(d)
    scale_idx: float = 0.0    # 0 -> 1/sqrt(d_idx)

    @property
    def nb(self) -> int:
        return (self.Nk + self.block - 1) // self.block

    def c(self) -> _Shape:
        return _Shape(self.B, self.Nq, self.Nk, self.q_offset, self.Hq, self.Hkv, self.d, self.d_idx, self.block,
                      self.topk, self.kv_rows, self.scale or 1.0 / math.sqrt(self.d),
                      self.scale_idx or 1.0 / math.sqrt(self.d_idx))


def _lib(kind: str):
    with _lock:
        if kind not in _loaded:
            build()
            lib = ctypes.CDLL(_LIBS[kind])
            P = ctypes.c_void_p
            S = ctypes.POINTER(_Shape)
            i, d = ctypes.c_int, ctypes.c_double
            lib.orc_block_scores.argtypes = [S, P, P, i, P, P]
            lib.orc_select.argtypes = [S, P, i, P, P]
            lib.orc_sparse_fwd.argtypes = [S, P, P, P, P, i, P, P, P]
            lib.orc_kl.argtypes = [S, P, P, P, P, P, i, P, P, P]
            lib.orc_bwd_rows.argtypes = [S, P, P, P, P, P, P, P, d, i, P, P, P]
            lib.orc_bwd_keys.argtypes = [S, P, P, P, P, P, P, P, d, i, P, P, P, P]
            lib.orc_block_mask.argtypes = [S, P, P]
            lib.orc_mask_walk.argtypes = [P, i, P]
            lib.orc_index_proj.argtypes = [i, i, i, i, P, P, P, P, P]
            lib.orc_index_proj_bwd.argtypes = [i, i, i, i, P, P, P, P, P]
            lib.orc_warmup_kl.argtypes = [S, P, P, P, P, i, P, P, P]
            lib.orc_warmup_grad.argtypes = [S, P, P, P, P, d, P, P]
            for f in ("orc_block_scores", "orc_select", "orc_sparse_fwd", "orc_kl", "orc_bwd_rows", "orc_bwd_keys",
                      "orc_block_mask", "orc_mask_walk", "orc_num_threads", "orc_index_proj", "orc_index_proj_bwd",
                      "orc_warmup_kl", "orc_warmup_grad"):
                getattr(lib, f).restype = ctypes.c_int
            _loaded[kind] = lib
        return _loaded[kind]


def _in(a: np.ndarray):
    """Pick the oracle variant from the input dtype and return a C pointer."""
    return a.ctypes.data_as(ctypes.c_void_p)


def _kind(*arrs) -> str:
    dt = {a.dtype for a in arrs}
    if dt == {np.dtype(np.uint16)}:
        return "bf16"
    if dt == {np.dtype(np.float64)}:
        return "f64"
    raise TypeError(f"oracle inputs must be all uint16 (bf16 bits) or all float64, got {dt}")


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _rows(shape: Shape, rows) -> np.ndarray:
    if rows is None:
        rows = np.arange(shape.B * shape.Nq)
    return _c(rows, np.int64)


def num_threads() -> int:
    return _lib("bf16").orc_num_threads()


def block_scores(shape: Shape, q_idx, k_idx, rows=None) -> np.ndarray:
    """fp32 block scores [n_rows, Hkv, nb]; invisible blocks are -inf."""
    rows = _rows(shape, rows)
    q_idx, k_idx = _c(q_idx, q_idx.dtype), _c(k_idx, k_idx.dtype)
    kind = _kind(q_idx, k_idx)
    out = np.empty((len(rows), shape.Hkv, shape.nb), dtype=np.float32)
    sh = shape.c()
    _lib(kind).orc_block_scores(ctypes.byref(sh), _in(q_idx), _in(k_idx), len(rows), _in(rows), _in(out))
    return out


def select(shape: Shape, bs, rows=None) -> np.ndarray:
    """Selected block ids [n_rows, Hkv, topk], ascending, -1 padded."""
    rows = _rows(shape, rows)
    bs = _c(bs, np.float32)
    out = np.empty((len(rows), shape.Hkv, shape.topk), dtype=np.int32)
    sh = shape.c()
    if _lib("bf16").orc_select(ctypes.byref(sh), _in(bs), len(rows), _in(rows), _in(out)) != 0:
        raise ValueError("topk above the oracle's limit of 64")
    return out


def block_mask(shape: Shape, sel_full) -> np.ndarray:
    """Block mask of a selection [B, Hkv, Nq, topk] (section 4.3): uint32
    words [B, Hkv, ceil(Nq/128), ceil(nb/32)], bit c%32 of word c/32 set when
    some query of the 128-row tile selected block c."""
    sel_full = _c(sel_full, np.int32)
    T, W = (shape.Nq + 127) // 128, (shape.nb + 31) // 32
    out = np.empty((shape.B, shape.Hkv, T, W), dtype=np.uint32)
    sh = shape.c()
    _lib("bf16").orc_block_mask(ctypes.byref(sh), _in(sel_full), _in(out))
    return out


def mask_walk(words) -> np.ndarray:
    """The active blocks of one tile's mask words, in visiting order."""
    words = _c(np.asarray(words, dtype=np.uint32).reshape(-1), np.uint32)
    out = np.empty(32 * max(1, len(words)), dtype=np.int32)
    n = _lib("bf16").orc_mask_walk(_in(words), len(words), _in(out))
    return out[:n].copy()


def sel_rows_from_full(shape: Shape, sel_full, rows) -> np.ndarray:
    """[B, Hkv, Nq, topk] -> [n_rows, Hkv, topk] for the listed row ids."""
    rows = _rows(shape, rows)
    b, i = rows // shape.Nq, rows % shape.Nq
    return _c(np.asarray(sel_full)[b, :, i, :], np.int32)


def sel_full_from_rows(shape: Shape, sel_rows) -> np.ndarray:
    """[B*Nq, Hkv, topk] (every row, in order) -> [B, Hkv, Nq, topk]."""
    a = np.asarray(sel_rows).reshape(shape.B, shape.Nq, shape.Hkv, shape.topk)
    return _c(a.transpose(0, 2, 1, 3), np.int32)


def sparse_fwd(shape: Shape, q, k, v, sel_rows, rows=None):
    """Main branch: O [n_rows, Hq, d] and LSE [n_rows, Hq] in float64."""
    rows = _rows(shape, rows)
    q, k, v = (_c(a, a.dtype) for a in (q, k, v))
    kind = _kind(q, k, v)
    sel_rows = _c(sel_rows, np.int32)
    o = np.empty((len(rows), shape.Hq, shape.d), dtype=np.float64)
    lse = np.empty((len(rows), shape.Hq), dtype=np.float64)
    sh = shape.c()
    _lib(kind).orc_sparse_fwd(ctypes.byref(sh), _in(q), _in(k), _in(v), _in(sel_rows), len(rows), _in(rows), _in(o),
                              _in(lse))
    return o, lse


def kl(shape: Shape, q, k, q_idx, k_idx, sel_rows, rows=None):
    """KL per (row, group) and the index log-sum-exp, float64 [n_rows, Hkv]."""
    rows = _rows(shape, rows)
    q, k, q_idx, k_idx = (_c(a, a.dtype) for a in (q, k, q_idx, k_idx))
    kind = _kind(q, k, q_idx, k_idx)
    sel_rows = _c(sel_rows, np.int32)
    lse_idx = np.empty((len(rows), shape.Hkv), dtype=np.float64)
    kl_rows = np.empty((len(rows), shape.Hkv), dtype=np.float64)
    sh = shape.c()
    _lib(kind).orc_kl(ctypes.byref(sh), _in(q), _in(k), _in(q_idx), _in(k_idx), _in(sel_rows), len(rows), _in(rows),
                      _in(lse_idx), _in(kl_rows))
    return lse_idx, kl_rows


def kl_loss(shape: Shape, kl_rows_all, kl_coef: float = 1.0) -> float:
    """The scalar L_KL from every row's KL: kl_coef / (B Nq Hkv) * sum."""
    return float(kl_coef * np.sum(kl_rows_all, dtype=np.float64) / (shape.B * shape.Nq * shape.Hkv))


def bwd_rows(shape: Shape, q, k, v, d_o, q_idx, k_idx, sel_full, kl_coef: float = 1.0, rows=None):
    """Query-side gradients for the listed rows: dq [n,Hq,d], dq_idx [n,Hkv,d_idx]."""
    rows = _rows(shape, rows)
    arrs = [_c(a, a.dtype) for a in (q, k, v, d_o, q_idx, k_idx)]
    kind = _kind(*arrs)
    sel_full = _c(sel_full, np.int32)
    dq = np.empty((len(rows), shape.Hq, shape.d), dtype=np.float64)
    dqi = np.empty((len(rows), shape.Hkv, shape.d_idx), dtype=np.float64)
    sh = shape.c()
    _lib(kind).orc_bwd_rows(ctypes.byref(sh), *[_in(a) for a in arrs], _in(sel_full), float(kl_coef), len(rows),
                            _in(rows), _in(dq), _in(dqi))
    return dq, dqi


def bwd_keys(shape: Shape, q, k, v, d_o, q_idx, k_idx, sel_full, kl_coef: float = 1.0, kblocks=None):
    """Key-side gradients for the listed key blocks:
    dk, dv [B, n_kb*block, Hkv, d], dk_idx [B, n_kb*block, d_idx]."""
    if kblocks is None:
        kblocks = np.arange(shape.nb)
    kblocks = _c(kblocks, np.int32)
    arrs = [_c(a, a.dtype) for a in (q, k, v, d_o, q_idx, k_idx)]
    kind = _kind(*arrs)
    sel_full = _c(sel_full, np.int32)
    n = len(kblocks) * shape.block
    dk = np.empty((shape.B, n, shape.Hkv, shape.d), dtype=np.float64)
    dv = np.empty_like(dk)
    dki = np.empty((shape.B, n, shape.d_idx), dtype=np.float64)
    sh = shape.c()
    rc = _lib(kind).orc_bwd_keys(ctypes.byref(sh), *[_in(a) for a in arrs], _in(sel_full), float(kl_coef),
                                 len(kblocks), _in(kblocks), _in(dk), _in(dv), _in(dki))
    if rc != 0:
        raise MemoryError("oracle could not allocate its partial buffers")
    return dk, dv, dki


def index_proj(X, Wq, Wk, Hkv: int, d_idx: int):
    """q_idx [T, Hkv*d_idx] and k_idx [T, d_idx] (float64) of X [T, Dm]."""
    X, Wq, Wk = (_c(a, a.dtype) for a in (X, Wq, Wk))
    kind = _kind(X, Wq, Wk)
    T, Dm = X.shape
    qi = np.empty((T, Hkv * d_idx), dtype=np.float64)
    ki = np.empty((T, d_idx), dtype=np.float64)
    _lib(kind).orc_index_proj(T, Dm, Hkv, d_idx, _in(X), _in(Wq), _in(Wk), _in(qi), _in(ki))
    return qi, ki


def index_proj_bwd(X, dq_idx, dk_idx, Hkv: int, d_idx: int):
    """dWq [Dm, Hkv*d_idx] and dWk [Dm, d_idx] (float64); no gradient into X."""
    X = _c(X, X.dtype)
    dq_idx = _c(np.asarray(dq_idx).reshape(X.shape[0], Hkv * d_idx), X.dtype)
    dk_idx = _c(np.asarray(dk_idx).reshape(X.shape[0], d_idx), X.dtype)
    kind = _kind(X, dq_idx, dk_idx)
    T, Dm = X.shape
    dWq = np.empty((Dm, Hkv * d_idx), dtype=np.float64)
    dWk = np.empty((Dm, d_idx), dtype=np.float64)
    _lib(kind).orc_index_proj_bwd(T, Dm, Hkv, d_idx, _in(X), _in(dq_idx), _in(dk_idx), _in(dWq), _in(dWk))
    return dWq, dWk


def warmup_kl(shape: Shape, q, k, q_idx, k_idx, rows=None):
    """Dense warm-up KL per (row, group) over the whole visible prefix, and
    the index log-sum-exp, float64 [n_rows, Hkv]."""
    rows = _rows(shape, rows)
    q, k, q_idx, k_idx = (_c(a, a.dtype) for a in (q, k, q_idx, k_idx))
    kind = _kind(q, k, q_idx, k_idx)
    lse_idx = np.empty((len(rows), shape.Hkv), dtype=np.float64)
    kl_rows = np.empty((len(rows), shape.Hkv), dtype=np.float64)
    sh = shape.c()
    _lib(kind).orc_warmup_kl(ctypes.byref(sh), _in(q), _in(k), _in(q_idx), _in(k_idx), len(rows), _in(rows),
                             _in(lse_idx), _in(kl_rows))
    return lse_idx, kl_rows


def warmup_grad(shape: Shape, q, k, q_idx, k_idx, kl_coef: float = 1.0):
    """Gradient of the dense warm-up loss kl_coef/(B Nq Hkv) * sum of rows in
    the index inputs: dq_idx [B, Nq, Hkv, d_idx], dk_idx [B, Nk, d_idx]."""
    q, k, q_idx, k_idx = (_c(a, a.dtype) for a in (q, k, q_idx, k_idx))
    kind = _kind(q, k, q_idx, k_idx)
    dqi = np.empty((shape.B, shape.Nq, shape.Hkv, shape.d_idx), dtype=np.float64)
    dki = np.empty((shape.B, shape.Nk, shape.d_idx), dtype=np.float64)
    sh = shape.c()
    _lib(kind).orc_warmup_grad(ctypes.byref(sh), _in(q), _in(k), _in(q_idx), _in(k_idx), float(kl_coef), _in(dqi),
                               _in(dki))
    return dqi, dki
