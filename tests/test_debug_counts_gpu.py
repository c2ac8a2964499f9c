"""Causal-skip check on the device (page "ADR-0060: AHBM GQA Fused Attention
kernel (Llama3-70B)", §11 verification plan: the tile GEMM count equals the
lower-triangle tile count; §5.4 tile classes).

The -DGQA_DEBUG build of the library counts, in the prefill MMA issuers, every
S = Q K^T tile they actually issue, by class. Those counts must equal the
oracle's classification of the (query block, KV tile) pairs, times the
(batch, head) count, bit for bit: every all-past and partial tile exactly
once, no all-future tile. Outputs of the debug build are checked too.
"""

import math

import numpy as np
import pytest
import torch

import oracle as orc
from gqa_attention_split_gb300 import api, build
from gqa_attention_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def DL():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return api.load(build.build(debug=True))


def _prefill(L, q, k, v, off, causal):
    B, H_q, T_q, d = q.shape
    H_kv, S_kv = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H_q, T_q), dtype=torch.float32, device=q.device)
    rc = L.gqa_attn_prefill_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), B, H_q, H_kv, d, T_q, S_kv, off,
                               1 if causal else 0, 1 / math.sqrt(d),
                               torch.cuda.current_stream().cuda_stream)
    assert rc == api.GQA_OK
    assert L.gqa_attn_check(torch.cuda.current_stream().cuda_stream) == api.GQA_OK
    return o, lse


def _expected(B, H_q, T_q, S_kv, off, causal):
    bm, bn = api.gqa_attn_prefill_block_m(), api.gqa_attn_prefill_block_n()
    cls = orc.prefill_tile_classes(T_q, S_kv, off, bm, bn)
    if not causal:
        return [B * H_q * cls.size, 0, 0]
    return [B * H_q * int((cls == orc.TILE_ALL_PAST).sum()),
            B * H_q * int((cls == orc.TILE_PARTIAL).sum()), 0]


@pytest.mark.parametrize("w", [wl.CAUSAL_PREFILL_8K, wl.CHUNKED_PREFILL_32K],
                         ids=lambda w: w.name)
def test_issued_tiles_equal_the_lower_triangle_full_size(DL, w):
    q, k, v = (t.cuda() for t in wl.prefill_inputs(w))
    assert api.gqa_attn_debug_tile_counts(clear=True, L=DL)[0] == api.GQA_OK
    _prefill(DL, q, k, v, w.q_offset, True)
    rc, got = api.gqa_attn_debug_tile_counts(clear=True, L=DL)
    assert rc == api.GQA_OK
    assert got == _expected(w.B, w.H_q, w.T_q, w.S_kv, w.q_offset, True)


@pytest.mark.parametrize("B,H_q,H_kv,T_q,S_kv,off,causal", [
    (1, 24, 8, 1100, 1300, 200, True),    # G = 3: block pairs of different extents
    (2, 16, 2, 300, 300, 0, True),        # ragged last block and tile
    (1, 8, 8, 257, 1000, 743, True),      # G = 1, chunk at the end of the prefix
    (1, 5, 5, 300, 300, 0, True),         # G = 1, three blocks: the last pair's second is empty
    (1, 16, 2, 200, 333, 0, False),       # full attention: every tile, no class split
])
@pytest.mark.parametrize("d", [64, 128])
def test_issued_tiles_and_outputs_small(DL, B, H_q, H_kv, T_q, S_kv, off, causal, d):
    q, k, v = wl.small_prefill(B, H_q, H_kv, d, T_q, S_kv, off, seed=40 + T_q)
    assert api.gqa_attn_debug_tile_counts(clear=True, L=DL)[0] == api.GQA_OK
    o, lse = _prefill(DL, q.cuda(), k.cuda(), v.cuda(), off, causal)
    rc, got = api.gqa_attn_debug_tile_counts(clear=True, L=DL)
    assert rc == api.GQA_OK
    assert got == _expected(B, H_q, T_q, S_kv, off, causal)
    O, L = orc.attention(q, k, v, scale=1 / math.sqrt(d), causal=causal, q_offset=off)
    err = np.abs(o.float().cpu().double().numpy() - O)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(lse.cpu().double().numpy() - L).max() <= 1e-3
