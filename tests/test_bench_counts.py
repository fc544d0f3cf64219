"""The benchmark's arithmetic, pinned on the CPU: the closed-form useful-FLOP
counts behind its TFLOP/s metric against brute-force counts over explicit
selections, and the per-workload totals these closed forms give for the
training and prefill shapes (index 17.59, forward 8.46 TFLOP at 128K)."""
import numpy as np
import pytest

import bench
from block_sparse_gqa_causal_gb300.workloads import BY_NAME, TINY


def _brute_tokens(w, rng):
    """Visible tokens of an explicit selection per query row: the local block
    plus k-1 distinct earlier blocks drawn at random (all of them when the
    query sees at most k blocks); every earlier block is fully visible."""
    T = np.zeros(w.N, dtype=np.int64)
    for i in range(w.N):
        c0 = i // w.block
        earlier = np.arange(c0)
        chosen = earlier if c0 + 1 <= w.topk else rng.choice(earlier, size=w.topk - 1, replace=False)
        toks = 0
        for c in list(chosen) + [c0]:
            lo, hi = c * w.block, min((c + 1) * w.block, i + 1)   # keys j <= i of block c
            toks += max(0, hi - lo)
        T[i] = toks
    return T


@pytest.mark.parametrize("w", [TINY, TINY.scaled(name="ragged", N=1000, topk=3), TINY.scaled(name="k1", N=700, topk=1)],
                         ids=lambda w: w.name)
def test_tokens_per_row_matches_explicit_selections(w):
    rng = np.random.default_rng(1)
    pos = np.arange(w.N)
    assert np.array_equal(bench.tokens_per_row(w, pos), _brute_tokens(w, rng))


def test_useful_flops_match_brute_force_counts():
    w = TINY.scaled(name="tiny_train", N=900, train=True)
    rng = np.random.default_rng(2)
    T = _brute_tokens(w, rng).astype(np.float64)
    vis = np.arange(w.N) + 1.0                              # keys a query's index scores cover
    want = {"index": 2 * w.d_idx * w.Hkv * vis.sum(), "fwd": 4 * w.d * w.Hq * T.sum(),
            "kl": 2 * w.d_idx * w.Hkv * T.sum(), "bwd": (10 * w.d * w.Hq + 6 * w.d_idx * w.Hkv) * T.sum()}
    got = bench.useful_flops(w)
    for k, v in want.items():
        assert got[k] == pytest.approx(w.B * v, rel=1e-12), k


def test_workload_totals():
    f = bench.useful_flops(BY_NAME["train_n128k"])
    assert f["index"] / 1e12 == pytest.approx(17.592, abs=5e-4)
    assert f["fwd"] / 1e12 == pytest.approx(8.459, abs=5e-4)
    assert f["bwd"] / 1e12 == pytest.approx(22.73, abs=5e-3)
    f32k = bench.useful_flops(BY_NAME["train_n32k"])
    assert f32k["fwd"] / 1e12 == pytest.approx(1.033, abs=5e-4)
    assert f32k["index"] / 1e12 == pytest.approx(1.100, abs=5e-4)


def test_kernel_work_slot_counts():
    """Per-slot and per-bucket byte counts scale with the slot count the
    selection implies: every (query, group) row holds min(k, c0 + 1) blocks."""
    w = BY_NAME["train_n128k"]
    work = bench.kernel_work(w)
    pos = np.arange(w.N)
    slots = w.B * w.Hkv * float(np.sum(np.minimum(w.topk, pos // 128 + 1)))
    buckets = w.B * w.Hkv * w.nb
    G, d = w.G, w.d
    assert work["bwd_main_tc_kernel"]["bytes"] == pytest.approx(
        slots * (2 * G * d * 2 + G * d * 2 + 256 + 8 * G) + buckets * 4 * 128 * d * 2, rel=1e-12)
    assert work["sparse_fwd_tc_kernel"]["bytes"] / 1e9 == pytest.approx(69.82, abs=0.01)
    assert work["bwd_main_tc_kernel"]["bytes"] / 1e9 == pytest.approx(108.73, abs=0.01)
