"""The five benchmark workloads, as seeded synthetic inputs.

Shapes, flags and value distributions follow the workloads the pages'
subject is measured on (head dim 64/128, prefill up to S = 8192, decode with
one query row): Q, K, V ~ N(0, 1) from the SplitMix64/Box-Muller generator of
this package (seed 0; streams q = 0, k = 1, v = 2), rounded to the storage
dtype; ALiBi slopes 2^(-8 (h+1) / Hq); the "rows given a window that masks all
keys" of the masked workload are round(1% of B * Sq) distinct (b, row) pairs
drawn from stream 3, given the empty per-row key range [1, 0].

No attention arithmetic lives here.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

from . import STREAM_K, STREAM_Q, STREAM_V, alibi_slopes, normal, row_kv_bounds_with_empty_rows


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: torch.dtype
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    causal: bool = False
    window_left: int | None = None
    window_right: int | None = None
    softcap: float | None = None
    alibi: bool = False
    empty_row_fraction: float = 0.0
    decode: bool = False
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def admissible_pairs(self, row_bounds: torch.Tensor | None = None) -> int:
        """Number of admissible (query, key) pairs summed over (b, h): the
        causal-adjusted work unit (4 D flops per pair: Q K^T and P V)."""
        total = 0
        for b in range(self.B):
            for i in range(self.Sq):
                a, e = 0, self.Sk - 1
                if self.causal:
                    e = min(e, i)
                if self.window_left is not None:
                    a = max(a, i - self.window_left)
                if self.window_right is not None:
                    e = min(e, i + self.window_right)
                if row_bounds is not None:
                    a = max(a, int(row_bounds[b, i, 0]))
                    e = min(e, int(row_bounds[b, i, 1]))
                total += max(0, e - a + 1)
        return total * self.Hq

    def flops(self, row_bounds=None) -> float:
        return 4.0 * self.D * self.admissible_pairs(row_bounds)

    def dense_flops(self) -> float:
        return 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.D

    def bytes_moved(self) -> int:
        """Q + K + V + O bytes (attention.fkc.md cost model, bytes_moved)."""
        es = 2 if self.dtype == torch.bfloat16 else 4
        return self.B * (2 * self.Hq * self.Sq * self.D + 2 * self.Hkv * self.Sk * self.D) * es


WORKLOADS = {
    "fp32_b1_h2_s64_d64": Workload("fp32_b1_h2_s64_d64", torch.float32, 1, 2, 1, 64, 64, 64,
                                   note="fp32 MHSDPA fwd, GQA group 2, non-causal"),
    "bf16_causal_b4_h32_s2048_d128": Workload("bf16_causal_b4_h32_s2048_d128", torch.bfloat16, 4, 32, 8,
                                              2048, 2048, 128, causal=True,
                                              note="bf16 causal prefill, GQA 32/8"),
    "bf16_causal_b1_h32_s8192_d128": Workload("bf16_causal_b1_h32_s8192_d128", torch.bfloat16, 1, 32, 8,
                                              8192, 8192, 128, causal=True,
                                              note="bf16 long causal prefill"),
    "bf16_masked_b2_h16_s4096_d64": Workload("bf16_masked_b2_h16_s4096_d64", torch.bfloat16, 2, 16, 16,
                                             4096, 4096, 64, causal=True, window_left=1024, window_right=0,
                                             softcap=50.0, alibi=True, empty_row_fraction=0.01,
                                             note="causal + window(1024,0) + softcap 50 + ALiBi + 1% empty rows"),
    "bf16_decode_b64_h32_sk8192_d128": Workload("bf16_decode_b64_h32_sk8192_d128", torch.bfloat16, 64, 32, 8,
                                                1, 8192, 128, decode=True,
                                                note="bf16 split-KV decode, Sq = 1"),
}

ORDER = list(WORKLOADS)


def make_inputs(w: Workload, device="cpu", seed: int = 0) -> dict:
    """Seeded inputs of a workload on `device` (generated there)."""
    q = normal((w.B, w.Hq, w.Sq, w.D), seed, STREAM_Q, w.dtype, device)
    k = normal((w.B, w.Hkv, w.Sk, w.D), seed, STREAM_K, w.dtype, device)
    v = normal((w.B, w.Hkv, w.Sk, w.D), seed, STREAM_V, w.dtype, device)
    slopes = alibi_slopes(w.Hq).to(device) if w.alibi else None
    rb = None
    if w.empty_row_fraction:
        rb = row_kv_bounds_with_empty_rows(w.B, w.Sq, w.Sk, w.empty_row_fraction, seed).to(device)
    return dict(q=q, k=k, v=v, alibi_slopes=slopes, row_kv_bounds=rb)


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (smaller parity cases)."""
    d = {f: getattr(w, f) for f in w.__dataclass_fields__}
    d.update(changes)
    return Workload(**d)


STREAM_PAGED = 4  # block placement and context lengths of paged inputs


def make_paged_inputs(B: int, Hq: int, Hkv: int, D: int, context_lens, block_size: int, dtype=torch.bfloat16,
                      device="cpu", seed: int = 0, spare_blocks: int = 3, max_blocks: int | None = None,
                      Sq: int = 1) -> dict:
    """Seeded paged-cache inputs: q [B, Hq, Sq, D]; k_cache / v_cache
    [num_blocks, block_size, Hkv, D] N(0,1); a block table [B, max_blocks]
    (int32) that places every sequence's blocks at seeded, shuffled physical
    positions of the pool (plus `spare_blocks` unused ones); context_lens [B]
    (int32).  Table entries past a sequence's last block hold num_blocks + 7,
    which no reader may dereference."""
    from . import uniform
    ctx = [int(c) for c in context_lens]
    nb = [(c + block_size - 1) // block_size for c in ctx]
    mb = max(max(nb), 1) if max_blocks is None else max_blocks
    num_blocks = sum(nb) + spare_blocks
    perm = torch.argsort(uniform(seed, STREAM_PAGED, 0, num_blocks))  # a seeded shuffle of the pool
    table = torch.full((B, mb), num_blocks + 7, dtype=torch.int32)
    i = 0
    for b in range(B):
        for j in range(nb[b]):
            table[b, j] = int(perm[i])
            i += 1
    q = normal((B, Hq, Sq, D), seed, STREAM_Q, dtype, device)
    k = normal((num_blocks, block_size, Hkv, D), seed, STREAM_K, dtype, device)
    v = normal((num_blocks, block_size, Hkv, D), seed, STREAM_V, dtype, device)
    return dict(q=q, k_cache=k, v_cache=v, block_table=table.to(device),
                context_lens=torch.tensor(ctx, dtype=torch.int32, device=device), num_blocks=num_blocks,
                block_size=block_size)
