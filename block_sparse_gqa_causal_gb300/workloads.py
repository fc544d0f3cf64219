"""The five synthetic MSA workloads: shapes, seeds and structure.

Only sizes live here (no arithmetic of the method).  Shapes follow the
operating point of "Sparse Attention · Part II", section 3.2 (128-token
blocks, 16 selected blocks per query and group, one of them the local
block) and the GQA layout that section describes.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    N: int                 # prefill: query and key length; decode: cache capacity
    Hq: int
    Hkv: int
    d: int
    d_idx: int
    topk: int
    seed: int
    block: int = 128
    needles_per_group: int = 0
    train: bool = False    # draws dO and runs KL + backward
    kl: bool = False       # runs the KL forward
    decode_steps: int = 0  # >0: decode workload, one new query per step
    notes: str = field(default="", compare=False)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def nb(self) -> int:
        return (self.N + self.block - 1) // self.block

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload("tiny_fwd_kl_n1k", B=1, N=1024, Hq=8, Hkv=2, d=64, d_idx=64, topk=4, seed=0,
                kl=True, train=True,
                notes="8 blocks of 128, 4 q-heads per group, k=4 incl. local block")
FWD_8K = Workload("fwd_n8k_b2", B=2, N=8192, Hq=32, Hkv=8, d=128, d_idx=128, topk=16, seed=1,
                  needles_per_group=2, notes="2 planted needle blocks per group")
TRAIN_32K = Workload("train_n32k", B=1, N=32768, Hq=32, Hkv=8, d=128, d_idx=128, topk=16, seed=2,
                     kl=True, train=True, notes="forward + KL + fused backward from dO")
PREFILL_128K = Workload("prefill_n128k", B=1, N=131072, Hq=64, Hkv=8, d=128, d_idx=128, topk=16,
                        seed=3, needles_per_group=2, notes="1024 blocks, 8 q-heads per group")
DECODE_1M = Workload("decode_1m_b4", B=4, N=1048576, Hq=64, Hkv=8, d=128, d_idx=128, topk=16,
                     seed=4, needles_per_group=4, decode_steps=256,
                     notes="cache of 1,048,576 tokens, 256 decode steps")

ALL = (TINY, FWD_8K, TRAIN_32K, PREFILL_128K, DECODE_1M)
BY_NAME = {w.name: w for w in ALL}

# The training step at the 128K prefill shapes (forward + KL + backward);
# the timed workload of the benchmark.
TRAIN_128K = PREFILL_128K.scaled(name="train_n128k", kl=True, train=True,
                                 notes="prefill_n128k shapes with KL and fused backward")
BY_NAME[TRAIN_128K.name] = TRAIN_128K
# The same head layout at 8K tokens: the small case for detailed profiles
# (inputs still larger than L2, a few GB on the device).
TRAIN_8K_H64 = PREFILL_128K.scaled(name="train_n8k_h64", N=8192, seed=5, kl=True, train=True,
                                   notes="train_n128k head layout at 8,192 tokens")
BY_NAME[TRAIN_8K_H64.name] = TRAIN_8K_H64
