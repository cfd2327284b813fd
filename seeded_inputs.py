"""Seeded synthetic inputs and workload shapes shared by the tests, the bench and the oracle's callers.

This module holds no arithmetic of the attention method: it only draws random numbers and names the
workload shapes. Both the CUDA path's tests and the CPU oracle receive the very same bytes from here.

Recipe (one draw each for Q, K and V, in that order):
  * ``torch.Generator('cpu').manual_seed(seed)``, ``torch.randn`` in fp32, i.e. N(0, 1) values;
  * bf16 workloads round those fp32 values to bf16 (round to nearest even, torch's ``.to``);
  * the default seed of workload ``i`` (0-based) is ``1000 + i + 1``.
Values are dense and unstructured, as in the pages' setting of causal self-attention over a long
sequence (USP review page, section "实验结果"; Context-Parallel page, Fig. 2).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention workload over a virtual Ulysses x Ring grid on one device."""
    name: str
    bs: int
    L: int
    hq: int
    hkv: int
    hd: int
    dtype: str          # "f32" or "bf16"
    ud: int             # Ulysses degree (head split)
    rd: int             # Ring degree (sequence split, zigzag)
    head_chunk: Optional[int] = None   # query heads per head group (UPipe-style chunking), None = all
    sample_rows: Optional[int] = None  # oracle rows per head for parity when full attention is too slow
    causal: bool = True

    @property
    def c(self) -> int:          # zigzag chunk length L / (2 rd)
        return self.L // (2 * self.rd)

    @property
    def Lr(self) -> int:         # ring-local sequence length L / rd
        return self.L // self.rd

    @property
    def Lu(self) -> int:         # tokens per virtual rank L / (rd ud)
        return self.L // (self.rd * self.ud)

    @property
    def causal_flops(self) -> float:
        """Causal-adjusted forward attention FLOPs: dense 4*bs*hq*L^2*hd, halved for the causal mask."""
        f = 4.0 * self.bs * self.hq * float(self.L) ** 2 * self.hd
        return f / 2 if self.causal else f

    def bytes_of(self, which: str) -> int:
        es = 4 if self.dtype == "f32" else 2
        h = self.hq if which in ("q", "o") else self.hkv
        return self.bs * self.L * h * self.hd * es


WORKLOADS = [
    Workload("tiny_mha_causal_L1024_h4_d64_f32_u1r4", 1, 1024, 4, 4, 64, "f32", ud=1, rd=4),
    Workload("mha_causal_L8192_h32_d128_bf16_u2r4", 1, 8192, 32, 32, 128, "bf16", ud=2, rd=4),
    Workload("gqa_causal_L32768_h32kv8_d128_bf16_u1r8", 1, 32768, 32, 8, 128, "bf16", ud=1, rd=8,
             sample_rows=256),
    Workload("mha_causal_L131072_h32_d128_bf16_u4r2", 1, 131072, 32, 32, 128, "bf16", ud=4, rd=2,
             sample_rows=256),
    Workload("gqa_causal_L262144_h32kv8_d128_bf16_u2r4_chunk8", 1, 262144, 32, 8, 128, "bf16", ud=2, rd=4,
             head_chunk=8, sample_rows=128),
    # MQA with more Ulysses ranks than KV heads: the all-to-all replicates the KV head on 4 ranks
    Workload("mqa_causal_L65536_h32kv1_d128_bf16_u4r2", 1, 65536, 32, 1, 128, "bf16", ud=4, rd=2,
             sample_rows=256),
]


def default_seed(index: int) -> int:
    return 1000 + index + 1


def make_qkv(bs: int, L: int, hq: int, hkv: int, hd: int, dtype: str, seed: int):
    """Q (bs,L,hq,hd), K and V (bs,L,hkv,hd) on the CPU, natural token order."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(bs, L, hq, hd, generator=g, dtype=torch.float32)
    k = torch.randn(bs, L, hkv, hd, generator=g, dtype=torch.float32)
    v = torch.randn(bs, L, hkv, hd, generator=g, dtype=torch.float32)
    if dtype == "bf16":
        q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    elif dtype != "f32":
        raise ValueError(f"unknown dtype {dtype}")
    return q, k, v


def make_workload_qkv(w: Workload, seed: int):
    return make_qkv(w.bs, w.L, w.hq, w.hkv, w.hd, w.dtype, seed)


def make_rows(L: int, c: int, n: int, seed: int):
    """Sorted sampled query rows: ``n`` uniform rows without replacement (seeded) plus forced rows
    0, L-1 and the first and last row of every zigzag chunk of length ``c``."""
    g = torch.Generator("cpu").manual_seed(seed + 7)
    n = min(n, L)
    pick = torch.randperm(L, generator=g)[:n].tolist()
    forced = {0, L - 1}
    for a in range(0, L, c):
        forced.add(a)
        forced.add(min(a + c - 1, L - 1))
    return sorted(set(pick) | forced)


def make_merge_inputs(rows: int, hd: int, dtype: str, seed: int, neg_inf_frac: float = 0.0):
    """Two (o, lse) partial pairs for the standalone merge: o ~ N(0,1), lse ~ 4*N(0,1).
    A fraction of lse entries (chosen by the same generator) is set to -inf, the empty-partial case."""
    g = torch.Generator("cpu").manual_seed(seed)
    o1 = torch.randn(rows, hd, generator=g)
    o2 = torch.randn(rows, hd, generator=g)
    l1 = 4 * torch.randn(rows, generator=g)
    l2 = 4 * torch.randn(rows, generator=g)
    if neg_inf_frac > 0:
        m1 = torch.rand(rows, generator=g) < neg_inf_frac
        m2 = torch.rand(rows, generator=g) < neg_inf_frac
        l1[m1] = float("-inf")
        l2[m2] = float("-inf")
        o1[m1] = 0
        o2[m2] = 0
    if dtype == "bf16":
        o1, o2 = o1.to(torch.bfloat16), o2.to(torch.bfloat16)
    return o1, l1, o2, l2
