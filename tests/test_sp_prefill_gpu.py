"""Sequence-parallel prefill on one GPU: the keys of a prefill cut into R
contiguous slices (page "ADR-0060: AHBM GQA Fused Attention kernel
(Llama3-70B)", §5.5 prefill with SP, where the K/V slices travel between
ranks), each slice's partial computed on its own in fp32 with its lse
(gqa_attn_prefill_partial), and the partials folded with the §4 log-sum-exp
merge (gqa_attn_merge). Each slice lives in its own contiguous buffer, as it
would on its own device. The merged result must match the fp64 oracle's
attention over all keys: max |dO| <= 1e-2, mean |dO| <= 1e-3, |d lse| <= 1e-3.
Under a causal mask the slices past a query contribute nothing to it: those
rows must come back as O = 0 and lse = -inf exactly.
"""

import math

import numpy as np
import pytest
import torch

import oracle as orc
from _fullsize import attention_by_group
from gqa_attention_split_gb300 import api, build
from gqa_attention_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()


def _close(o, l, O, L, what):
    o = np.asarray(o, dtype=np.float64).reshape(O.shape)
    l = np.asarray(l, dtype=np.float64).reshape(L.shape)
    err = np.abs(o - O)
    assert np.isfinite(o).all(), what
    assert err.max() <= MAX_ABS, f"{what} max|dO|={err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what} mean|dO|={err.mean():.3e}"
    assert np.abs(l - L).max() <= LSE_ABS, f"{what} max|dlse|={np.abs(l - L).max():.3e}"


def _sharded_prefill(q, k, v, R, q_offset, causal):
    """Every slice's partial (its own contiguous K/V buffer) and the merge."""
    S = k.shape[2]
    rc, bounds = api.gqa_attn_split_bounds(S, R, S)
    assert rc == 0
    qd = q.cuda()
    parts = []
    for a, b in bounds:
        assert b > a
        ks, vs = k[:, :, a:b].contiguous().cuda(), v[:, :, a:b].contiguous().cuda()
        parts.append((a, b) + api.prefill_partial(qd, ks, vs, q_offset=q_offset, key_offset=a,
                                                  causal=causal))
    o, lse = api.merge(torch.stack([p[2] for p in parts]), torch.stack([p[3] for p in parts]))
    api.check()
    return o, lse, parts


def _check_empty_rows(parts, T_q, q_offset, causal):
    # a row t sees no key of slice [a, b) iff a > q_offset + t (causal)
    if not causal:
        return
    for a, b, o_r, l_r in parts:
        t_empty = max(0, min(T_q, a - q_offset))
        if t_empty:
            assert torch.isneginf(l_r[:, :, :t_empty]).all()
            assert (o_r[:, :, :t_empty] == 0).all()
            assert torch.isfinite(l_r[:, :, t_empty:]).all()


@pytest.mark.parametrize("B,H_q,H_kv,d,T_q,S,off,causal,R", [
    (1, 8, 2, 128, 300, 300, 0, True, 3),      # head pairs; later slices empty for early rows
    (1, 8, 2, 128, 130, 1000, 870, True, 4),   # a chunk at the end of a long prefix
    (2, 16, 2, 128, 200, 333, 0, False, 2),    # full attention, ragged slices
    (1, 6, 2, 128, 257, 700, 443, True, 5),    # odd G = 3: block pairs
    (1, 8, 2, 64, 384, 384, 0, True, 3),       # d = 64
    (1, 16, 2, 128, 1000, 1000, 0, True, 1),   # one slice: the whole prefill
    (1, 4, 4, 128, 129, 2000, 1871, True, 7),  # G = 1, slices of 286 keys
])
def test_sharded_prefill_matches_the_oracle(B, H_q, H_kv, d, T_q, S, off, causal, R):
    q, k, v = wl.small_prefill(B, H_q, H_kv, d, T_q, S, off, seed=1500 + T_q + R)
    o, lse, parts = _sharded_prefill(q, k, v, R, off, causal)
    O, L = orc.attention(q, k, v, scale=1 / math.sqrt(d), causal=causal, q_offset=off)
    _close(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, f"R={R}")
    _check_empty_rows(parts, T_q, off, causal)


@pytest.mark.parametrize("w,R", [(wl.CAUSAL_PREFILL_8K, 4), (wl.CHUNKED_PREFILL_32K, 4)],
                         ids=["causal8k_R4", "chunked32k_R4"])
def test_sharded_full_size_every_row(w, R):
    # 8K causal cut into four slices of 2048 keys (most rows see only some of
    # them); the chunked 32K prefill cut into four slices of 8192 keys (three
    # fully in the past of every query, the last one the causal diagonal)
    q, k, v = wl.prefill_inputs(w)
    o, lse, parts = _sharded_prefill(q, k, v, R, w.q_offset, True)
    O, L = attention_by_group(q, k, v, scale=w.scale, causal=True, q_offset=w.q_offset)
    _close(o.float().cpu().numpy(), lse.cpu().numpy(), O, L, w.name)
    _check_empty_rows(parts, w.T_q, w.q_offset, True)
    # and the same as the whole-cache prefill within the tolerance
    o1, _ = api.prefill(q.cuda(), k.cuda(), v.cuda(), q_offset=w.q_offset, causal=True)
    api.check()
    assert (o1.float() - o.float()).abs().max().item() <= MAX_ABS
