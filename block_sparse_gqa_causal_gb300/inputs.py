"""Seeded synthetic inputs for the MSA workloads (numpy only).

This module holds no arithmetic of the method: it draws N(0,1) tensors,
rounds them to bf16 and plants needle blocks.  Both the CUDA path's tests
and benchmark and the CPU oracle's tests take their inputs from here.

Recipe
  * Every tensor is drawn from numpy's default_rng as float32 N(0,1) in
    chunks of 2**22 elements; chunk c of tensor t uses
    SeedSequence(seed, spawn_key=(t, c)), so the values do not depend on
    which other tensors are drawn or on the thread count.  Tensor ids:
    q=0, k=1, v=2, q_idx=3, k_idx=4, d_o=5, needle choices=6.
  * float32 -> bf16 is round-to-nearest-even on the bit pattern; tensors are
    returned as uint16 arrays of bf16 bits.
  * Needles: for batch b and group r, u_r is the float32 mean over the
    sequence's query tokens of q_idx[b, :, r, :], scaled to unit L2 norm.
    Each group draws `needles_per_group` distinct blocks (rng of tensor id 6,
    chunk b), and every token of a drawn block gets k_idx += 0.5 * u_r,
    summed over groups in float32 and rounded to bf16 once.  Prefill draws
    from all blocks; decode draws from the blocks fully inside the prefilled
    cache.

Prefill layouts: q [B,N,Hq,d], k/v [B,N,Hkv,d], q_idx [B,N,Hkv,d_idx],
k_idx [B,N,d_idx], d_o like q.  Decode: q [B,S,Hq,d], q_idx [B,S,Hkv,d_idx]
for the S steps, k/v/k_idx caches with N (capacity) rows; step s queries at
position N - S + s.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .workloads import Workload

CHUNK = 1 << 22
TID = {"q": 0, "k": 1, "v": 2, "q_idx": 3, "k_idx": 4, "d_o": 5, "needle": 6}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _fill_chunk(out: np.ndarray, seed: int, tid: int, c: int) -> None:
    lo = c * CHUNK
    hi = min(out.size, lo + CHUNK)
    rng = np.random.default_rng(np.random.SeedSequence(seed, spawn_key=(tid, c)))
    out[lo:hi] = f32_to_bf16_bits(rng.standard_normal(hi - lo, dtype=np.float32))


def normal_bf16(shape, seed: int, tid: int, threads: int | None = None) -> np.ndarray:
    """N(0,1) tensor of the given shape as bf16 bits (uint16)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    nch = (n + CHUNK - 1) // CHUNK
    threads = threads or min(32, os.cpu_count() or 1)
    if nch <= 1 or threads <= 1:
        for c in range(nch):
            _fill_chunk(out, seed, tid, c)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda c: _fill_chunk(out, seed, tid, c), range(nch)))
    return out.reshape(shape)


def plant_needles(w: Workload, q_idx: np.ndarray, k_idx: np.ndarray, n_blocks_eligible: int) -> np.ndarray:
    """Add 0.5*u_r to every token of each group's drawn needle blocks (in place).
    Returns the drawn blocks, shape [B, Hkv, needles_per_group]."""
    n = w.needles_per_group
    drawn = np.zeros((w.B, w.Hkv, n), dtype=np.int64)
    for b in range(w.B):
        rng = np.random.default_rng(np.random.SeedSequence(w.seed, spawn_key=(TID["needle"], b)))
        delta = np.zeros((n_blocks_eligible, w.d_idx), dtype=np.float32)
        for r in range(w.Hkv):
            u = bf16_bits_to_f32(q_idx[b, :, r, :]).mean(axis=0, dtype=np.float32)
            u = (u / np.float32(np.linalg.norm(u))).astype(np.float32)
            blocks = rng.choice(n_blocks_eligible, size=n, replace=False)
            drawn[b, r] = blocks
            for blk in blocks:
                delta[blk] += np.float32(0.5) * u
        for blk in np.unique(drawn[b]):
            rows = slice(blk * w.block, (blk + 1) * w.block)
            k_idx[b, rows, :] = f32_to_bf16_bits(bf16_bits_to_f32(k_idx[b, rows, :]) + delta[blk][None, :])
    return drawn


def make_inputs(w: Workload, with_grad: bool | None = None, threads: int | None = None) -> dict:
    """All input tensors of a workload, as bf16 bit arrays, plus metadata."""
    with_grad = w.train if with_grad is None else with_grad
    nq = w.decode_steps if w.decode_steps else w.N
    out = {
        "q": normal_bf16((w.B, nq, w.Hq, w.d), w.seed, TID["q"], threads),
        "k": normal_bf16((w.B, w.N, w.Hkv, w.d), w.seed, TID["k"], threads),
        "v": normal_bf16((w.B, w.N, w.Hkv, w.d), w.seed, TID["v"], threads),
        "q_idx": normal_bf16((w.B, nq, w.Hkv, w.d_idx), w.seed, TID["q_idx"], threads),
        "k_idx": normal_bf16((w.B, w.N, w.d_idx), w.seed, TID["k_idx"], threads),
    }
    if with_grad:
        out["d_o"] = normal_bf16((w.B, nq, w.Hq, w.d), w.seed, TID["d_o"], threads)
    if w.needles_per_group:
        eligible = (w.N - w.decode_steps) // w.block if w.decode_steps else w.nb
        out["needles"] = plant_needles(w, out["q_idx"], out["k_idx"], eligible)
    return out


def decode_position(w: Workload, step: int) -> int:
    """Absolute position of the query of decode step `step`."""
    return w.N - w.decode_steps + step
