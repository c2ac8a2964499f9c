"""The prefill kernel under a host-made work order (gqa_attn_prefill_schedule).

Page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)", §5.4 prefill
scheduling. The order of the work items changes no result: each item is
computed the same way on whichever CTA runs it. A tiny L2 budget (test hook)
makes even small problems run a host-made order, one (batch, KV head) group
per super-group; the outputs must equal those of the closed-form order bit for
bit and match the fp64 oracle (max |dO| <= 1e-2, mean |dO| <= 1e-3,
|d lse| <= 1e-3).
"""

import math

import numpy as np
import pytest
import torch

from _fullsize import attention_by_group
from gqa_attention_split_gb300 import api, build
from gqa_attention_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()
    yield
    api.gqa_attn_debug_prefill_order(-1)


def _both_orders(fn):
    api.gqa_attn_debug_prefill_order(0)   # closed-form order
    a = fn()
    api.check()
    api.gqa_attn_debug_prefill_order(1)   # host-made order for every launch
    b = fn()
    api.check()
    api.gqa_attn_debug_prefill_order(-1)
    return a, b


@pytest.mark.parametrize("B,H_q,H_kv,d,T_q,S_kv,off,causal", [
    (1, 64, 8, 128, 2048, 2048, 0, True),     # 512 items over 152 CTAs
    (2, 64, 8, 128, 1024, 4096, 3072, True),  # chunk at an offset, two batch rows
    (1, 24, 8, 128, 1100, 1300, 200, True),   # G = 3: block pairs, ragged last block
    (1, 64, 64, 128, 1024, 1024, 0, True),    # G = 1: 256 block-pair items
    (2, 16, 4, 128, 200, 333, 0, False),      # full attention, ragged keys
    (1, 64, 8, 64, 1024, 1024, 0, True),      # d = 64
    (3, 8, 1, 128, 129, 129, 0, True),        # fewer items than SMs
])
def test_host_order_matches_closed_form_bitwise_and_the_oracle(B, H_q, H_kv, d, T_q, S_kv,
                                                               off, causal):
    q, k, v = wl.small_prefill(B, H_q, H_kv, d, T_q, S_kv, off, seed=300 + T_q + H_q + d)
    rc, lists = api.gqa_attn_prefill_schedule(B, H_q, H_kv, d, T_q, S_kv, off, int(causal), 152)
    assert rc == 0  # these fit in L2: the library keeps the closed form by default
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    (o0, l0), (o1, l1) = _both_orders(
        lambda: api.prefill(qd, kd, vd, q_offset=off, causal=causal))
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    O, L = attention_by_group(q, k, v, scale=1 / math.sqrt(d), causal=causal, q_offset=off)
    o = o1.float().cpu().double().numpy()
    err = np.abs(o - O)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(l1.cpu().double().numpy() - L).max() <= 1e-3


def _random_prefill_shapes(n, seed):
    """Seeded shapes for the prefill under both orders, small enough for the
    oracle: (B, H_q, H_kv, d, T_q, S_kv, q_offset, causal)."""
    rng = np.random.default_rng(seed)
    shapes = []
    while len(shapes) < n:
        B = int(rng.integers(1, 4))
        H_kv = int(rng.choice([1, 2, 4]))
        G = int(rng.integers(1, 9))
        d = int(rng.choice([64, 128]))
        causal = bool(rng.integers(0, 2))
        T = int(rng.integers(1, 1200))
        off = int(rng.integers(0, 1500)) if causal else 0
        S = T + off + (0 if causal else int(rng.integers(0, 800)))
        if B * H_kv * G * T * S * d > 2_000_000_000:
            continue
        shapes.append((B, H_kv * G, H_kv, d, T, S, off, causal))
    return shapes


@pytest.mark.parametrize("B,H_q,H_kv,d,T_q,S_kv,off,causal", _random_prefill_shapes(12, 77))
def test_random_shapes_both_orders(B, H_q, H_kv, d, T_q, S_kv, off, causal):
    q, k, v = wl.small_prefill(B, H_q, H_kv, d, T_q, S_kv, off, seed=900 + T_q + S_kv)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    (o0, l0), (o1, l1) = _both_orders(
        lambda: api.prefill(qd, kd, vd, q_offset=off, causal=causal))
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    O, L = attention_by_group(q, k, v, scale=1 / math.sqrt(d), causal=causal, q_offset=off)
    o = o1.float().cpu().double().numpy()
    err = np.abs(o - O)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(l1.cpu().double().numpy() - L).max() <= 1e-3


@pytest.mark.parametrize("G", [8, 3])
def test_slice_prefill_under_a_host_order(G):
    # a key slice that starts past some query blocks: items with no visible key
    H_kv, d, T_q, S = 4, 128, 700, 1500
    q, k, v = wl.small_prefill(1, G * H_kv, H_kv, d, T_q, S, 800, seed=330 + G)
    ks, vs = k[:, :, 1100:].contiguous().cuda(), v[:, :, 1100:].contiguous().cuda()
    qd = q.cuda()
    (o0, l0), (o1, l1) = _both_orders(
        lambda: api.prefill_partial(qd, ks, vs, q_offset=800, key_offset=1100, causal=True))
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
