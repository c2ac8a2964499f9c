"""Pins for the INT4 KV part of the oracle.

Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §4 item 3
(optional INT4 / INT8 KV quantisation; the scheme is the reading stated in
the oracle: symmetric per-token absmax, fp32 scale max|x|/7, codes
rint(x / scale) in [-7, 7] with ties to even). The pins check the rounding
rule on hand-made ties, the error bound of the scheme, the all-zero case, and
that attention over a cache whose values are exact multiples of their scales
equals plain attention on the original values.
"""

import numpy as np
import torch

import oracle


def test_codes_follow_round_half_to_even_on_ties():
    # max |x| = 7 makes the scale exactly 1, so each x / scale is x itself
    x = np.array([[7.0, 2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5, 6.5, -7.0, 4.5, -5.5]])
    codes, scales = oracle.quantize_q4(x)
    assert scales.dtype == np.float32 and scales[0] == 1.0
    assert codes.tolist() == [[7, 2, 4, -2, -4, 0, 0, 2, 6, -7, 4, -6]]


def test_scale_is_the_fp32_quotient_and_the_absmax_maps_to_7():
    x = torch.randn(64, 128, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    codes, scales = oracle.quantize_q4(x)
    xf = x.float().numpy()
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(scales, (amax / np.float32(7)).astype(np.float32))
    assert (np.abs(codes.astype(np.int32)).max(axis=1) == 7).all()
    assert codes.dtype == np.int8 and np.abs(codes.astype(np.int32)).max() <= 7


def test_round_trip_error_is_at_most_half_a_step():
    x = torch.randn(256, 128, generator=torch.Generator().manual_seed(10)).to(torch.bfloat16)
    codes, scales = oracle.quantize_q4(x)
    back = codes.astype(np.float64) * scales.astype(np.float64)[:, None]
    err = np.abs(back - x.double().numpy())
    # half a step, plus the fp32 roundings of max|x| / 7 and of x / scale
    assert (err <= scales.astype(np.float64)[:, None] * (0.5 + 2e-6)).all()


def test_zero_tokens_get_zero_scale_and_codes():
    x = np.zeros((3, 64))
    x[1, 5] = -2.0
    codes, scales = oracle.quantize_q4(x)
    assert scales[0] == 0 and scales[2] == 0 and (codes[[0, 2]] == 0).all()
    assert codes[1, 5] == -7 and np.count_nonzero(codes[1]) == 1


def test_exactly_representable_cache_gives_plain_attention():
    rng = np.random.default_rng(22)
    B, H_q, H_kv, S, d = 2, 8, 2, 40, 32
    sk = 2.0 ** -rng.integers(1, 6, size=(B, H_kv, S))
    sv = 2.0 ** -rng.integers(1, 6, size=(B, H_kv, S))
    ik = rng.integers(-7, 8, size=(B, H_kv, S, d))
    iv = rng.integers(-7, 8, size=(B, H_kv, S, d))
    ik[..., 0], iv[..., 0] = 7, -7  # pin each token's absmax
    sk, sv = sk.astype(np.float32), sv.astype(np.float32)
    K = ik * sk.astype(np.float64)[..., None]
    V = iv * sv.astype(np.float64)[..., None]
    kc, ks = oracle.quantize_q4(K.astype(np.float32))
    vc, vs = oracle.quantize_q4(V.astype(np.float32))
    q = rng.standard_normal((B, H_q, d))
    seqlens = [40, 13]
    assert np.array_equal(kc, ik) and np.array_equal(ks, sk)
    assert np.array_equal(vc, iv) and np.array_equal(vs, sv)
    O, L = oracle.attention_q4(q, kc, ks, vc, vs, scale=0.2, seqlens=seqlens)
    O2, L2 = oracle.attention(q[:, :, None], K, V, scale=0.2, seqlens=seqlens)
    assert np.allclose(O, O2[:, :, 0], rtol=0, atol=1e-12)
    assert np.allclose(L, L2[:, :, 0], rtol=0, atol=1e-12)


def test_attention_reads_the_codes_as_integers_times_scales():
    # a one-token cache: the output is that token's dequantised V row, and lse
    # is its single score, (q . k_codes * k_scale) * scale
    q = np.array([[[1.0, -2.0, 0.5, 0.0]]])
    kc = np.array([[[[3, -1, 7, 0]]]], dtype=np.int8)
    vc = np.array([[[[-7, 2, 0, 5]]]], dtype=np.int8)
    ks = np.array([[[0.25]]], dtype=np.float32)
    vs = np.array([[[0.5]]], dtype=np.float32)
    O, L = oracle.attention_q4(q, kc, ks, vc, vs, scale=0.5)
    assert np.array_equal(O[0, 0], [-3.5, 1.0, 0.0, 2.5])
    assert L[0, 0] == (1 * 3 + 2 * 1 + 0.5 * 7) * 0.25 * 0.5
