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


def test_kernel_work_design_slot_counts():
    """The design's per-slot and per-bucket byte counts scale with the slot
    count the selection implies: every (query, group) row holds min(k, c0 + 1)
    blocks."""
    w = BY_NAME["train_n128k"]
    work = bench.kernel_work(w)
    pos = np.arange(w.N)
    slots = w.B * w.Hkv * float(np.sum(np.minimum(w.topk, pos // 128 + 1)))
    buckets = w.B * w.Hkv * w.nb
    G, d = w.G, w.d
    assert work["bwd_main_tc_kernel"]["design_bytes"] == pytest.approx(
        slots * (2 * G * d * 2 + G * d * 2 + 8 * G) + buckets * 4 * 128 * d * 2, rel=1e-12)
    assert work["sparse_fwd_tc_kernel"]["design_bytes"] / 1e9 == pytest.approx(69.82, abs=0.01)


def test_kernel_work_algorithmic_bytes():
    """Algorithmic bytes: each tensor the kernel's step reads, once, and each
    it writes, once.  The main backward at 128K: Q, dO, dQ (2.147 GB each), K,
    V, dK, dV (0.268 GB each), LSE and D (33.5 MB each), the selection (67 MB):
    7.65 GB, against 21.15 TFLOP -- tensor-bound at the measured peaks."""
    w = BY_NAME["train_n128k"]
    work = bench.kernel_work(w)
    q_b = 131072 * 64 * 128 * 2
    kv_b = 131072 * 8 * 128 * 2
    want = 3 * q_b + 4 * kv_b + 2 * 64 * 131072 * 4 + 8 * 131072 * 16 * 4
    assert work["bwd_main_tc_kernel"]["bytes"] == pytest.approx(want, rel=1e-12)
    assert work["bwd_main_tc_kernel"]["bytes"] / 1e9 == pytest.approx(7.65, abs=0.01)
    # forward: Q, K, V, selection in; O, LSE out
    assert work["sparse_fwd_tc_kernel"]["bytes"] == pytest.approx(
        2 * q_b + 2 * kv_b + 8 * 131072 * 16 * 4 + 64 * 131072 * 4, rel=1e-12)
    peaks = {"hbm_gbs": 6780.4, "bf16_tflops": 1923.3, "bf16_tflops_sustained": 1712.0, "source": "measured"}
    ktimes = {"bwd_main_tc_kernel": (5, 5 * 22.8)}
    r = bench.kernel_roofline("bwd_main_tc_kernel", ktimes, work, peaks, w)
    assert r["bound"] == "tensor"
    # timed inside the training step: against the sustained bf16 rate, the burst fraction beside it
    assert r["peak"] == 1712.0
    assert r["frac"] == pytest.approx(21.147e12 / 22.8e-3 / 1712.0e12, rel=2e-3)
    assert r["frac_of_burst"] == pytest.approx(21.147e12 / 22.8e-3 / 1923.3e12, rel=2e-3)
    assert r["hbm"]["frac"] == pytest.approx(want / 22.8e-3 / 6780.4e9, rel=2e-3)


def test_oracle_sample_flops_count_only_the_work_run():
    """The CPU baseline is credited with index, forward, KL index scores and
    the query-side backward of its sampled rows (6 d T per head + 4 d_idx T
    per group), not with the key-side gradients it does not run."""
    w = BY_NAME["train_n128k"]
    rows = np.array([0, 5000, 131071])
    T = bench.tokens_per_row(w, rows).astype(np.float64)
    f = bench.useful_flops(w.scaled(B=1), positions=rows)
    want = f["index"] + f["fwd"] + f["kl"] + float(np.sum((6 * w.d * w.Hq + 4 * w.d_idx * w.Hkv) * T))
    assert bench.oracle_flops(w, rows) == pytest.approx(want, rel=1e-12)
    assert bench.oracle_flops(w, rows) < sum(f.values())
