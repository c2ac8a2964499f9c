"""Seeded synthetic inputs shaped like the Llama3-70B GQA workloads.

This module only draws random numbers; it holds none of the attention
arithmetic. Both the CUDA path (through the tests and ``bench.py``) and the
fp64 oracle read the tensors it returns.

Recipe: a CPU ``torch.Generator`` seeded per workload draws N(0, 1) in fp32,
in the order q, k, v, and each tensor is rounded to bf16 (round to nearest
even). Ragged decode lengths come from a second generator seeded with 1003,
uniform over [16384, 131072]. Shapes follow the page "ADR-0060: AHBM GQA
Fused Attention kernel (Llama3-70B)", §0 reference dimensions
(H_q = 64, H_kv = 8, G = 8, d = 128).
"""

from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H_q: int
    H_kv: int
    d: int
    S_max: int
    seed: int
    ragged: bool = False  # seqlens drawn per row instead of all S_max

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    H_q: int
    H_kv: int
    d: int
    T_q: int
    S_kv: int
    q_offset: int
    seed: int
    causal: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


TINY_DECODE = DecodeWorkload("tiny_decode_b1_hq8_hkv1_d64_s256", 1, 8, 1, 64, 256, seed=1)
LLAMA70B_DECODE_8K = DecodeWorkload("llama70b_decode_b1_s8192", 1, 64, 8, 128, 8192, seed=2)
RAGGED_DECODE_128K = DecodeWorkload("llama70b_ragged_decode_b4_s16k_128k", 4, 64, 8, 128,
                                    131072, seed=3, ragged=True)
CAUSAL_PREFILL_8K = PrefillWorkload("llama70b_causal_prefill_b1_t8192", 1, 64, 8, 128,
                                    8192, 8192, 0, seed=4)
CHUNKED_PREFILL_32K = PrefillWorkload("llama70b_chunked_prefill_b2_t2048_off30720", 2, 64, 8,
                                      128, 2048, 32768, 30720, seed=5)

# Not one of the five workloads: the 8K causal prefill with one query head per KV
# head (G = 1), for timing the odd-G work items.
CAUSAL_PREFILL_8K_MHA = PrefillWorkload("mha_causal_prefill_b1_t8192", 1, 64, 64, 128, 8192,
                                        8192, 0, seed=6)

# Not one of the five workloads: one sequence of 128K cached tokens (the
# single-row long-context decode the split plan gives one wave of 16 splits).
LLAMA70B_DECODE_128K_B1 = DecodeWorkload("llama70b_decode_b1_s131072", 1, 64, 8, 128, 131072,
                                         seed=7)

RAGGED_SEQLEN_SEED = 1003
RAGGED_SEQLEN_RANGE = (16384, 131072)  # inclusive


def _randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def ragged_seqlens(B: int, lo: int, hi: int, seed: int = RAGGED_SEQLEN_SEED) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def decode_inputs(w: DecodeWorkload, seqlens: torch.Tensor | None = None):
    """Host tensors q [B,H_q,d], k/v [B,H_kv,S_max,d] (bf16) and seqlens [B] int32."""
    g = torch.Generator().manual_seed(w.seed)
    q = _randn_bf16((w.B, w.H_q, w.d), g)
    k = _randn_bf16((w.B, w.H_kv, w.S_max, w.d), g)
    v = _randn_bf16((w.B, w.H_kv, w.S_max, w.d), g)
    if seqlens is None:
        if w.ragged:
            seqlens = ragged_seqlens(w.B, *RAGGED_SEQLEN_RANGE)
        else:
            seqlens = torch.full((w.B,), w.S_max, dtype=torch.int32)
    return q, k, v, seqlens.to(torch.int32)


def prefill_inputs(w: PrefillWorkload):
    """Host tensors q [B,H_q,T_q,d], k/v [B,H_kv,S_kv,d] (bf16)."""
    g = torch.Generator().manual_seed(w.seed)
    q = _randn_bf16((w.B, w.H_q, w.T_q, w.d), g)
    k = _randn_bf16((w.B, w.H_kv, w.S_kv, w.d), g)
    v = _randn_bf16((w.B, w.H_kv, w.S_kv, w.d), g)
    return q, k, v


def small_decode(B, H_q, H_kv, d, S_max, seed, seqlens=None):
    """A decode workload of any small shape (tests)."""
    return decode_inputs(DecodeWorkload("small", B, H_q, H_kv, d, S_max, seed),
                         None if seqlens is None else torch.as_tensor(seqlens, dtype=torch.int32))


def small_prefill(B, H_q, H_kv, d, T_q, S_kv, q_offset, seed, causal=True):
    return prefill_inputs(PrefillWorkload("small", B, H_q, H_kv, d, T_q, S_kv, q_offset, seed,
                                          causal))
