"""GPU parity of the causal prefill path (tcgen05) against the fp64 oracle.

Tolerance (bf16 outputs): max |dO| <= 1e-2, mean |dO| <= 1e-3, |d lse| <= 1e-3.
All calls go through the C ABI (ctypes binding).
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


def assert_close(o, l, O_ref, L_ref, what=""):
    o = np.asarray(o, dtype=np.float64).reshape(O_ref.shape)
    l = np.asarray(l, dtype=np.float64).reshape(L_ref.shape)
    err = np.abs(o - O_ref)
    assert np.isfinite(o).all(), what
    assert err.max() <= MAX_ABS, f"{what} max|dO|={err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what} mean|dO|={err.mean():.3e}"
    dl = np.abs(l - L_ref).max()
    assert dl <= LSE_ABS, f"{what} max|dlse|={dl:.3e}"


def run_prefill(q, k, v, q_offset, causal, scale=None):
    o, lse = api.prefill(q.cuda(), k.cuda(), v.cuda(), q_offset=q_offset, causal=causal,
                         scale=scale)
    api.check()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


@pytest.mark.parametrize("B,H_q,H_kv,T_q,S_kv,off,causal", [
    (1, 8, 2, 128, 128, 0, True),       # one tile, diagonal only
    (1, 8, 8, 256, 256, 0, True),       # G = 1
    (2, 16, 2, 300, 300, 0, True),      # ragged last block and tile, G = 8
    (1, 4, 1, 5, 5, 0, True),           # tiny
    (1, 8, 2, 130, 400, 270, True),     # chunk at an offset, ragged
    (1, 8, 2, 64, 1000, 936, True),     # chunk at the end of a long prefix
    (2, 8, 4, 200, 333, 0, False),      # full attention, ragged keys
    (1, 4, 2, 1, 1, 0, True),           # a single query and key
    (1, 6, 2, 257, 300, 43, True),      # odd G = 3 (block pairs), chunk at an offset
    (1, 16, 2, 128, 640, 0, False),     # full attention over more keys than queries
    (3, 8, 1, 129, 129, 0, True),       # three batch rows, one query row past a block
    (1, 8, 2, 1, 1000, 999, True),      # one query at the end of a long prefix (causal)
    (2, 8, 2, 1, 777, 0, False),        # one query, full attention over ragged keys
    # odd G: work items pair two consecutive query blocks of one head
    (1, 5, 5, 129, 700, 571, True),     # G = 1, the second block holds one row
    (2, 6, 2, 300, 300, 0, False),      # G = 3, full attention; last pair's second block empty
    (1, 9, 3, 640, 640, 0, True),       # G = 3, five blocks
    (1, 7, 7, 1, 50, 49, True),         # G = 1, a single query
])
def test_small_shapes(B, H_q, H_kv, T_q, S_kv, off, causal):
    q, k, v = wl.small_prefill(B, H_q, H_kv, 128, T_q, S_kv, off, seed=10 + T_q + S_kv)
    o, lse = run_prefill(q, k, v, off, causal)
    O, L = orc.attention(q, k, v, scale=1 / math.sqrt(128), causal=causal, q_offset=off)
    assert_close(o, lse, O, L, f"B={B} H={H_q}/{H_kv} T={T_q} S={S_kv} off={off} c={causal}")



@pytest.mark.parametrize("causal", [True, False])
def test_a_later_tile_with_much_larger_scores(causal):
    # Keys 256..383 scaled by 8 (exact in bf16): from the third KV tile on, the
    # running max of each row that sees them grows by far more than the rescale
    # threshold, so O and the sums are rescaled mid-row; the fourth tile then
    # runs against that larger max.
    B, H_q, H_kv, T, S = 1, 8, 2, 512, 512
    q, k, v = wl.small_prefill(B, H_q, H_kv, 128, T, S, 0, seed=77)
    k = k.clone()
    k[:, :, 256:384] *= 8
    o, lse = run_prefill(q, k, v, 0, causal)
    O, L = orc.attention(q, k, v, scale=1 / math.sqrt(128), causal=causal)
    assert_close(o, lse, O, L, f"large scores causal={causal}")

@pytest.mark.parametrize("w", [wl.CAUSAL_PREFILL_8K, wl.CHUNKED_PREFILL_32K],
                         ids=lambda w: w.name)
def test_full_size_workloads_every_row(w):
    # Every output row of the 8K causal prefill (2048 work items of the
    # persistent kernel over the SMs) and of the chunked 32K prefill at
    # q_offset 30720 (1024 items), against the fp64 oracle.
    q, k, v = wl.prefill_inputs(w)
    o, lse = run_prefill(q, k, v, w.q_offset, True)
    O, L = attention_by_group(q, k, v, scale=w.scale, causal=True, q_offset=w.q_offset)
    assert_close(o, lse, O, L, w.name)


@pytest.mark.parametrize("B,H_q,H_kv,T_q,S_kv,off,causal", [
    (1, 64, 8, 2048, 2048, 0, True),       # 512 items over at most 152 CTAs
    (2, 64, 8, 1024, 4096, 3072, True),    # chunk at an offset, two batch rows: 512 items
    (1, 64, 8, 1024, 1536, 0, False),      # full attention: 256 items
    (1, 48, 8, 1536, 1536, 0, True),       # G = 6: pairs cross no KV group, 288 items
    (1, 24, 8, 1100, 1300, 200, True),     # G = 3: block pairs, ragged last block
    (1, 64, 64, 1024, 1024, 0, True),      # G = 1: 256 block-pair items
    (2, 48, 16, 700, 1500, 800, True),     # G = 3, two batch rows, chunk at an offset
])
def test_many_work_items_per_cta_every_row(B, H_q, H_kv, T_q, S_kv, off, causal):
    # The persistent kernel runs several items per CTA here: barrier phases
    # counted across items, Q reloaded once the previous item's last S MMAs
    # completed, and PV(0) overwriting the previous item's O after its
    # epilogue read it. Every row is compared.
    q, k, v = wl.small_prefill(B, H_q, H_kv, 128, T_q, S_kv, off, seed=20 + T_q + S_kv + H_q)
    o, lse = run_prefill(q, k, v, off, causal)
    O, L = attention_by_group(q, k, v, scale=1 / math.sqrt(128), causal=causal, q_offset=off)
    assert_close(o, lse, O, L, f"B={B} H={H_q}/{H_kv} T={T_q} S={S_kv} off={off} c={causal}")


def p_rounding_bound(q, k, v, O, *, causal, q_offset):
    """Per-element bound on |O_gpu - O| from the kernels' arithmetic. P is
    rounded to bf16 before the P.V MMA (8-bit significand: relative error
    |d_j| <= u = 2^-8 per weight) and O is normalised by the sum of the rounded
    weights, so O_gpu is a convex combination of the visible V rows whose
    weights are the exact ones times (1 + d_j) / (1 + mean d). To first order
    |dO_c| <= 2u * max_j |v_jc - O_c| over the visible keys j, plus the
    output's own bf16 rounding, u |O_c|, plus 1e-4 for the fp32 sums."""
    v = orc.to_f64(v)
    G = q.shape[1] // k.shape[1]
    v_rep = np.repeat(v, G, axis=1)                      # [B, H_q, S, d]
    vmax = np.maximum.accumulate(v_rep, axis=2)          # prefix max / min over keys
    vmin = np.minimum.accumulate(v_rep, axis=2)
    T_q, S = q.shape[2], k.shape[2]
    last = [(min(S, q_offset + t + 1) if causal else S) - 1 for t in range(T_q)]
    hi, lo = vmax[:, :, last], vmin[:, :, last]          # [B, H_q, T_q, d]
    spread = np.maximum(np.abs(hi - O), np.abs(lo - O))
    return 2.0 ** -7 * spread + 2.0 ** -8 * np.abs(O) + 1e-4


@pytest.mark.parametrize("B,H_q,H_kv,T_q,S_kv,off,causal", [
    (1, 8, 2, 300, 300, 0, True),         # head pairs, ragged last block and tile
    (2, 16, 2, 200, 333, 0, False),       # full attention, ragged keys
    (1, 8, 2, 130, 400, 270, True),       # chunk at an offset
    (1, 6, 2, 257, 300, 43, True),        # odd G = 3: block pairs
    (1, 64, 8, 1024, 1024, 0, True),      # 256 items over at most 152 CTAs
    (1, 32, 32, 640, 640, 0, True),       # G = 1, five blocks
])
def test_head_dim_64(B, H_q, H_kv, T_q, S_kv, off, causal):
    # d = 64: one 64-column box per tile, four k-steps per S MMA, N = 64 for P.V
    q, k, v = wl.small_prefill(B, H_q, H_kv, 64, T_q, S_kv, off, seed=90 + T_q + H_q)
    o, lse = run_prefill(q, k, v, off, causal)
    O, L = attention_by_group(q, k, v, scale=1 / math.sqrt(64), causal=causal, q_offset=off)
    assert_close(o, lse, O, L, f"d=64 B={B} H={H_q}/{H_kv} T={T_q} S={S_kv} off={off}")


@pytest.mark.parametrize("scale", [0.05, 0.3])
@pytest.mark.parametrize("causal", [True, False])
def test_scales_other_than_one_over_sqrt_d(scale, causal):
    # Any finite scale > 0 is accepted. 0.05 flattens the scores and meets the
    # decode/prefill tolerance. 0.3 makes them ~3.4x sharper than 1/sqrt(128),
    # with many lazy rescales; the weight of a few keys then dominates each row
    # and their bf16 rounding no longer averages out, so the bar there is the
    # bound the arithmetic fixes (p_rounding_bound), element by element.
    B, H_q, H_kv, T, S, off = 1, 16, 2, 700, 900, 200
    off = off if causal else 0
    q, k, v = wl.small_prefill(B, H_q, H_kv, 128, T, S, off, seed=81)
    o, lse = run_prefill(q, k, v, off, causal, scale=scale)
    O, L = orc.attention(q, k, v, scale=scale, causal=causal, q_offset=off)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    err = np.abs(o - O)
    bound = p_rounding_bound(q, k, v, O, causal=causal, q_offset=off)
    assert (err <= bound).all(), f"scale={scale}: max excess {(err - bound).max():.3e}"
    assert np.abs(lse - L).max() <= LSE_ABS
    if scale <= 1 / math.sqrt(128):
        assert_close(o, lse, O, L, f"scale={scale} causal={causal}")


def test_non_positive_scale_is_rejected():
    q, k, v = wl.small_prefill(1, 8, 2, 128, 64, 64, 0, seed=82)
    for bad in (0.0, -0.088):
        with pytest.raises(api.GqaError) as e:
            api.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=bad)
        assert e.value.code == api.GQA_ERR_INVALID_ARG


def test_deterministic_bitwise():
    q, k, v = wl.small_prefill(1, 16, 2, 128, 1000, 1000, 0, seed=77)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    a = api.prefill(qd, kd, vd, causal=True)
    b = api.prefill(qd, kd, vd, causal=True)
    api.check()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_lse_null_and_output_bounds():
    B, H_q, H_kv, T, d = 1, 4, 2, 200, 128
    q, k, v = wl.small_prefill(B, H_q, H_kv, d, T, T, 0, seed=78)
    pad = 256
    buf = torch.full((B * H_q * T * d + 2 * pad,), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    o = buf[pad:pad + B * H_q * T * d].view(B, H_q, T, d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    rc = api.gqa_attn_prefill_ex(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), None,
                                 B, H_q, H_kv, d, T, T, 0, 1, 1 / math.sqrt(d),
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    api.check()
    assert torch.isnan(buf[:pad].float()).all() and torch.isnan(buf[-pad:].float()).all()
    O, _ = orc.attention(q, k, v, scale=1 / math.sqrt(d), causal=True)
    assert np.abs(o.float().cpu().double().numpy() - O).max() <= MAX_ABS


def test_fixed_geometry_entry_point_matches_ex():
    q, k, v = wl.small_prefill(1, 64, 8, 128, 256, 512, 256, seed=79)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1 = torch.empty_like(qd)
    st = torch.cuda.current_stream().cuda_stream
    rc = api.gqa_attn_prefill(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o1.data_ptr(), None,
                              1, 256, 512, 256, 1, 1 / math.sqrt(128), st)
    assert rc == 0
    o2, _ = api.prefill(qd, kd, vd, q_offset=256, causal=True)
    api.check()
    assert torch.equal(o1, o2)


def test_bad_offset_rejected():
    q, k, v = wl.small_prefill(1, 8, 2, 128, 100, 150, 0, seed=80)
    with pytest.raises(api.GqaError) as e:
        api.prefill(q.cuda(), k.cuda(), v.cuda(), q_offset=60, causal=True)
    assert e.value.code == api.GQA_ERR_INVALID_ARG
