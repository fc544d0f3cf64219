"""The seeded input recipe (block_sparse_gqa_causal_gb300/inputs.py), pinned
on the CPU: values depend only on (seed, tensor, chunk) -- not on the thread
count, on which other tensors are drawn, or on the chunking of a larger
draw -- and the needle planting follows its statement: u_r the unit-norm fp32
mean of the group's index queries, 0.5 u_r added (summed over groups) to every
token of each drawn block, other tokens unchanged."""
import numpy as np
import pytest

from block_sparse_gqa_causal_gb300 import inputs
from block_sparse_gqa_causal_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits, make_inputs
from block_sparse_gqa_causal_gb300.workloads import TINY, FWD_8K, DECODE_1M


def test_draws_do_not_depend_on_threads_or_on_other_tensors():
    shape = (3, inputs.CHUNK // 1000 + 7, 1000)        # more than two chunks
    a = inputs.normal_bf16(shape, 5, 1, threads=1)
    b = inputs.normal_bf16(shape, 5, 1, threads=4)
    assert np.array_equal(a, b)
    # a tensor's first chunk is the same whatever the total size
    small = inputs.normal_bf16((1000,), 5, 1, threads=1)
    assert np.array_equal(small, a.reshape(-1)[:1000])
    # another tensor id or seed gives other values
    assert not np.array_equal(inputs.normal_bf16((1000,), 5, 2), small)
    assert not np.array_equal(inputs.normal_bf16((1000,), 6, 1), small)
    w = TINY
    x1, x2 = make_inputs(w, with_grad=False), make_inputs(w, with_grad=True)
    for n in ("q", "k", "v", "q_idx", "k_idx"):
        assert np.array_equal(x1[n], x2[n])


def test_draws_are_standard_normal():
    x = bf16_bits_to_f32(inputs.normal_bf16((1 << 20,), 3, 0)).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3


@pytest.mark.parametrize("w", [FWD_8K.scaled(name="needles_small", B=2, N=2048, Hq=8, Hkv=4),
                               DECODE_1M.scaled(name="needles_decode", B=2, N=4096, Hq=8, Hkv=4, decode_steps=200)],
                         ids=lambda w: w.name)
def test_needles_follow_the_recipe(w):
    x = make_inputs(w)
    base = make_inputs(w.scaled(needles_per_group=0))
    drawn = x["needles"]
    eligible = (w.N - w.decode_steps) // w.block if w.decode_steps else w.nb
    assert drawn.shape == (w.B, w.Hkv, w.needles_per_group)
    for b in range(w.B):
        delta = np.zeros((eligible, w.d_idx), dtype=np.float32)
        for r in range(w.Hkv):
            blocks = drawn[b, r]
            assert len(set(blocks.tolist())) == len(blocks) and blocks.min() >= 0 and blocks.max() < eligible
            u = bf16_bits_to_f32(x["q_idx"][b, :, r, :]).astype(np.float64).mean(axis=0)
            u = (u / np.linalg.norm(u)).astype(np.float32)
            for blk in blocks:
                delta[blk] += np.float32(0.5) * u
        planted = np.zeros(w.N, dtype=bool)
        for blk in np.unique(drawn[b]):
            rows = slice(blk * w.block, (blk + 1) * w.block)
            planted[rows] = True
            want = f32_to_bf16_bits(bf16_bits_to_f32(base["k_idx"][b, rows, :]) + delta[blk][None, :])
            # the recipe's fp32 mean may differ from this fp64 one in the last bit of u
            diff = np.abs(want.astype(np.int64) - x["k_idx"][b, rows, :].astype(np.int64))
            assert diff.max() <= 1
        assert np.array_equal(x["k_idx"][b, ~planted], base["k_idx"][b, ~planted])
    for n in ("q", "k", "v", "q_idx"):
        assert np.array_equal(x[n], base[n])
