"""GPU parity of the ring-buffer cache (attention sinks + local window).

Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §2 item 4 and §4
item 2. The append kernel must place tokens exactly where the oracle's
token-by-token replay puts them (bit-exact copy), and decode over the cache
must match the oracle's token-level definition (softmax over the sink and
window tokens of each row's stream) within the decode tolerance:
max |dO| <= 1e-2, mean |dO| <= 1e-3, |d lse| <= 1e-3.
"""

import math

import numpy as np
import pytest
import torch

import oracle as orc
from gqa_attention_split_gb300 import api, build

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()


def _stream(B, H_kv, T, d, seed):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(B, H_kv, T, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H_kv, T, d, generator=g).to(torch.bfloat16)
    return k, v


def _cache_from_oracle(stream, seqlens, capacity, n_sink):
    """bf16 cache [B, H_kv, capacity, d] holding each row's replayed tokens;
    slots never written hold NaN (a decode must never read them)."""
    B, H_kv, _, d = stream.shape
    out = np.empty((B, H_kv, capacity, d))
    for b in range(B):
        for h in range(H_kv):
            out[b, h] = orc.ring_write(stream[b, h].double().numpy(), int(seqlens[b]), capacity,
                                       n_sink)
    return torch.from_numpy(out).to(torch.bfloat16)


def _assert_close(o, lse, O_ref, L_ref, what):
    o = o.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    err = np.abs(o - O_ref)
    assert np.isfinite(o).all(), what
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, f"{what} max|dO|={err.max():.3e}"
    fin = np.isfinite(L_ref)
    assert (np.isneginf(l) == ~fin).all(), what
    if fin.any():
        assert np.abs(l[fin] - L_ref[fin]).max() <= LSE_ABS, what


@pytest.mark.parametrize("capacity,n_sink,d", [(48, 4, 128), (33, 0, 64), (64, 63, 128)])
def test_append_places_every_token_like_the_replay(capacity, n_sink, d):
    B, H_kv, T = 2, 2, 3 * capacity + 5
    k, v = _stream(B, H_kv, T, d, seed=capacity + d)
    kc = torch.zeros(B, H_kv, capacity, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    kd, vd = k.cuda(), v.cuda()
    for t in range(T):
        pos = torch.full((B,), t, dtype=torch.int32, device="cuda")
        api.ring_append(kc, vc, kd[:, :, t].contiguous(), vd[:, :, t].contiguous(), pos,
                        n_sink=n_sink)
        if t + 1 in (1, capacity - 1, capacity, capacity + 1, T):
            api.check()
            for src, got in ((k, kc), (v, vc)):
                want = np.stack([np.stack([orc.ring_write(src[b, h].double().numpy(), t + 1,
                                                          capacity, n_sink, fill=0.0)
                                           for h in range(H_kv)]) for b in range(B)])
                assert np.array_equal(got.float().cpu().double().numpy(), want), t


def test_append_with_a_negative_position_writes_nothing_and_reports():
    kc = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    new = torch.ones(1, 1, 64, dtype=torch.bfloat16, device="cuda")
    api.ring_append(kc, vc, new, new, torch.tensor([-1], dtype=torch.int32, device="cuda"),
                    n_sink=2)
    with pytest.raises(api.GqaError) as e:
        api.check()
    assert e.value.code == api.GQA_ERR_DEVICE_BAD_INPUT
    assert kc.abs().sum().item() == 0


@pytest.mark.parametrize("capacity,n_sink,d,G", [(1000, 4, 128, 8), (300, 0, 64, 4),
                                                 (257, 256, 128, 1), (4096, 16, 128, 8)])
def test_decode_matches_the_token_level_definition(capacity, n_sink, d, G):
    seqlens = [0, 1, 5, n_sink + 1, capacity - 1, capacity, capacity + 1, 3 * capacity + 7]
    B, H_kv = len(seqlens), 2
    H_q = G * H_kv
    T = max(seqlens)
    k, v = _stream(B, H_kv, T, d, seed=7 * capacity + d)
    g = torch.Generator().manual_seed(capacity)
    q = torch.randn(B, H_q, d, generator=g).to(torch.bfloat16)
    kc = _cache_from_oracle(k, seqlens, capacity, n_sink).cuda()
    vc = _cache_from_oracle(v, seqlens, capacity, n_sink).cuda()
    sl = torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(d)
    O, L = orc.attention_ring(q, k, v, scale=scale, seqlens=seqlens, capacity=capacity,
                              n_sink=n_sink)
    for ns in (0, 1, 3, 16):
        o, lse = api.decode_ring(q.cuda(), kc, vc, sl, n_sink=n_sink, num_splits=ns)
        api.check()  # lengths above capacity are legal here, not clamped-and-reported
        _assert_close(o, lse, O, L, f"cap={capacity} sink={n_sink} ns={ns}")


def test_decode_reports_a_negative_length():
    q = torch.randn(1, 8, 128).to(torch.bfloat16).cuda()
    kc = torch.randn(1, 1, 64, 128).to(torch.bfloat16).cuda()
    o, lse = api.decode_ring(q, kc, kc.clone(), torch.tensor([-3], dtype=torch.int32,
                                                               device="cuda"), n_sink=2)
    with pytest.raises(api.GqaError) as e:
        api.check()
    assert e.value.code == api.GQA_ERR_DEVICE_BAD_INPUT
    assert o.float().abs().max().item() == 0 and torch.isneginf(lse).all()
