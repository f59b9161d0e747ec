"""Named workloads: the shapes, precision, retrieval noise and input scale of each case the
library is tested and measured on.  Sizes only; no arithmetic.

    B            sequences
    n_chunks     chunks of 64 tokens per sequence (L = 64 n_chunks)
    H, dh        heads and head dim of Q / K / V
    D            landmark dim
    topk         retrieved chunks per query chunk
    qkv_std      element std of the synthetic Q, K, V, dO (landmarks are N(0, 1))
    groups       retrieval groups (the second takes group 1's output as query landmarks)
    query_chunks query chunks per sequence (all of them, or one for decode)
    causal_offset candidates are chunks j < i + causal_offset (all past chunks at decode)
"""
from __future__ import annotations

from dataclasses import dataclass

CHUNK = 64


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    n_chunks: int
    H: int
    dh: int
    D: int
    topk: int
    dtype: str
    gumbel: bool
    qkv_std: float
    groups: int = 1
    query_chunks: int | None = None
    causal_offset: int = 0

    @property
    def L(self) -> int:
        return self.n_chunks * CHUNK

    @property
    def nQ(self) -> int:
        return self.query_chunks if self.query_chunks is not None else self.n_chunks


TINY_F32 = Workload("tiny fp32 parity case", B=1, n_chunks=16, H=4, dh=32, D=128, topk=4, dtype="f32", gumbel=False,
                    qkv_std=1.0)
TRAIN_128M = Workload("training step, 128M-model shape", B=4, n_chunks=256, H=12, dh=64, D=768, topk=8, dtype="bf16",
                      gumbel=True, qkv_std=0.125)
TRAIN_350M_G2 = Workload("training step, 350M-model shape, two retrieval groups", B=8, n_chunks=256, H=16, dh=64,
                         D=1024, topk=8, dtype="bf16", gumbel=True, qkv_std=0.125, groups=2)
PREFILL_1M = Workload("prefill of 1M tokens", B=1, n_chunks=16384, H=12, dh=64, D=768, topk=8, dtype="bf16",
                      gumbel=False, qkv_std=0.125)
DECODE_16M = Workload("decode at 16M context, one query chunk per sequence", B=16, n_chunks=262144, H=12, dh=64,
                      D=768, topk=8, dtype="bf16", gumbel=False, qkv_std=0.125, query_chunks=1,
                      causal_offset=262144)

ALL = (TINY_F32, TRAIN_128M, TRAIN_350M_G2, PREFILL_1M, DECODE_16M)
