"""Sequence-parallel decode on one GPU: a KV cache cut into R contiguous key
slices (page "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)", §5.3
decode with SP), each slice decoded on its own into an fp32 partial
(gqa_attn_decode_partial), and the partials folded with the §4 log-sum-exp
merge (gqa_attn_merge). Each slice lives in its own contiguous buffer, as it
would on its own device. The merged result must match the fp64 oracle's
attention over the whole row: max |dO| <= 1e-2, mean |dO| <= 1e-3,
|d lse| <= 1e-3; each partial must match the oracle on its slice.
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


def _close(o, l, O, L, what, tol=(MAX_ABS, MEAN_ABS, LSE_ABS)):
    o = np.asarray(o, dtype=np.float64).reshape(O.shape)
    l = np.asarray(l, dtype=np.float64).reshape(L.shape)
    err = np.abs(o - O)
    assert np.isfinite(o).all(), what
    assert err.max() <= tol[0], f"{what} max|dO|={err.max():.3e}"
    assert err.mean() <= tol[1], f"{what} mean|dO|={err.mean():.3e}"
    fin = np.isfinite(L)
    assert (np.isneginf(l) == ~fin).all(), what
    if fin.any():
        assert np.abs(l[fin] - L[fin]).max() <= tol[2], what


def _sharded_decode(q, k, v, seqlens, R, ns=0):
    """Decodes every slice into a partial and merges them; returns the merged
    (o, lse) and the per-slice (bounds, local seqlens, o_r, lse_r)."""
    B, H_kv, S_max, d = k.shape
    rc, bounds = api.gqa_attn_split_bounds(S_max, R, S_max)
    assert rc == 0
    qd = q.cuda()
    parts_o, parts_l, info = [], [], []
    for (a, b) in bounds:
        local = torch.tensor([max(0, min(int(n), b) - a) for n in seqlens.tolist()],
                             dtype=torch.int32)
        if b > a:
            ks = k[:, :, a:b].contiguous().cuda()
            vs = v[:, :, a:b].contiguous().cuda()
            o_r, l_r = api.decode_partial(qd, ks, vs, local.cuda(), num_splits=ns)
        else:  # an empty slice (R > S_max): a partial with no keys
            o_r = torch.zeros((B, q.shape[1], d), dtype=torch.float32, device="cuda")
            l_r = torch.full((B, q.shape[1]), float("-inf"), device="cuda")
        parts_o.append(o_r)
        parts_l.append(l_r)
        info.append(((a, b), local, o_r, l_r))
    o, lse = api.merge(torch.stack(parts_o), torch.stack(parts_l))
    api.check()
    return o, lse, info


@pytest.mark.parametrize("R", [1, 2, 3, 5])
def test_sharded_ragged_rows_match_the_oracle(R):
    S_max, d = 3000, 128
    lens = [3000, 2999, 1601, 700, 1, 0]  # rows ending inside early slices, and empty
    q, k, v, sl = wl.small_decode(len(lens), 16, 2, d, S_max, seed=1100 + R, seqlens=lens)
    o, lse, info = _sharded_decode(q, k, v, sl, R)
    O, L = orc.attention(q[:, :, None], k, v, scale=1 / math.sqrt(d), seqlens=lens)
    _close(o.float().cpu().numpy(), lse.cpu().numpy(), O[:, :, 0], L[:, :, 0], f"R={R}")
    for (a, b), local, o_r, l_r in info:  # each partial is attention over its slice
        Or, Lr = orc.attention(q[:, :, None], k[:, :, a:b], v[:, :, a:b],
                               scale=1 / math.sqrt(d), seqlens=local.tolist())
        # fp32 partial: only the kernel's own error, no output rounding
        _close(o_r.cpu().numpy(), l_r.cpu().numpy(), Or[:, :, 0], Lr[:, :, 0],
               f"R={R} slice [{a},{b})")


@pytest.mark.parametrize("R", [2, 4])
def test_sharded_llama70b_8k_all_rows(R):
    w = wl.LLAMA70B_DECODE_8K
    q, k, v, sl = wl.decode_inputs(w)
    o, lse, _ = _sharded_decode(q, k, v, sl, R)
    O, L = orc.attention(q[:, :, None], k, v, scale=w.scale, seqlens=sl.tolist())
    _close(o.float().cpu().numpy(), lse.cpu().numpy(), O[:, :, 0], L[:, :, 0], f"8K R={R}")
    # and the same as the one-device decode, within the decode tolerance
    o1, l1 = api.decode(q.cuda(), k.cuda(), v.cuda(), sl.cuda())
    api.check()
    assert (o1.float() - o.float()).abs().max().item() <= MAX_ABS


def test_sharded_ragged_128k_every_row():
    w = wl.RAGGED_DECODE_128K
    q, k, v, sl = wl.decode_inputs(w)
    o, lse, _ = _sharded_decode(q, k, v, sl, 4)
    O, L = attention_by_group(q[:, :, None], k, v, scale=w.scale, seqlens=sl.tolist(),
                              task_gb=3.0)
    _close(o.float().cpu().numpy(), lse.cpu().numpy(), O[:, :, 0], L[:, :, 0], "128K R=4")


def test_merge_alone_against_the_oracle_merge():
    # Random partials, some empty (lse = -inf, O = NaN: must be skipped), merged
    # in rank order; the oracle folds the same triples (m = lse_r, l = 1). The
    # partials and weights are fp32, so the only error left is the bf16
    # rounding of the result: |dO| <= 2^-8 |O| (8-bit significand), plus fp32
    # slack.
    g = torch.Generator().manual_seed(1200)
    R, rows, d = 7, 300, 64
    o_parts = torch.randn(R, rows, d, generator=g) * 0.7
    lse_parts = torch.randn(R, rows, generator=g) * 20
    empty = torch.rand(R, rows, generator=g) < 0.3
    empty[:, :5] = True                      # rows with no keys at all
    lse_parts[empty] = float("-inf")
    o_parts[empty] = float("nan")
    o, lse = api.merge(o_parts.cuda(), lse_parts.cuda())
    api.check()
    ms = lse_parts.double().numpy()
    Os = np.where(empty.numpy()[..., None], 0.0, o_parts.double().numpy())
    O, L = orc.combine_partials(ms, np.ones_like(ms), Os)
    og = o.float().cpu().double().numpy()
    lg = lse.cpu().double().numpy()
    assert np.isfinite(og).all()
    assert (np.abs(og - O) <= 2.0 ** -8 * np.abs(O) + 1e-6).all()
    fin = np.isfinite(L)
    assert (np.isneginf(lg) == ~fin).all()
    assert np.abs(lg[fin] - L[fin]).max() <= 1e-5 * np.abs(L[fin]).max() + 1e-5
    assert (o[:5] == 0).all() and torch.isneginf(lse[:5]).all()


def test_merge_more_parts_than_a_warp_has_lanes():
    # R > 32: the lse values are read 32 at a time; d = 128 uses float4 loads
    g = torch.Generator().manual_seed(1201)
    R, rows, d = 45, 70, 128
    o_parts = torch.randn(R, rows, d, generator=g) * 0.7
    lse_parts = torch.randn(R, rows, generator=g) * 5
    empty = torch.rand(R, rows, generator=g) < 0.2
    lse_parts[empty] = float("-inf")
    o_parts[empty] = float("nan")
    o, lse = api.merge(o_parts.cuda(), lse_parts.cuda())
    api.check()
    ms = lse_parts.double().numpy()
    Os = np.where(empty.numpy()[..., None], 0.0, o_parts.double().numpy())
    O, L = orc.combine_partials(ms, np.ones_like(ms), Os)
    og = o.float().cpu().double().numpy()
    assert (np.abs(og - O) <= 2.0 ** -8 * np.abs(O) + 1e-6).all()
    assert np.abs(lse.cpu().double().numpy() - L).max() <= 1e-4


def test_sharded_decode_group_of_16():
    # G = 16 runs two CTAs per (split, KV head); the partials keep fp32 O
    lens = [2500, 1200, 1]
    q, k, v, sl = wl.small_decode(3, 32, 2, 128, 2500, seed=1202, seqlens=lens)
    o, lse, _ = _sharded_decode(q, k, v, sl, 3)
    O, L = orc.attention(q[:, :, None], k, v, scale=1 / math.sqrt(128), seqlens=lens)
    _close(o.float().cpu().numpy(), lse.cpu().numpy(), O[:, :, 0], L[:, :, 0], "G=16 R=3")
