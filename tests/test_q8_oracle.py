"""Pins for the INT8 KV part of the oracle.

Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §4 item 3
(optional INT4 / INT8 KV quantisation; the scheme is the reading stated in
the oracle: symmetric per-token absmax, fp32 scale max|x|/127, codes
rint(x / scale) with ties to even). The pins check the rounding rule on
hand-made ties, the error bound of the scheme, the all-zero case, and that
attention over a cache whose values are exact multiples of their scales
equals plain attention on the original values.
"""

import numpy as np
import torch

import oracle


def test_codes_follow_round_half_to_even_on_ties():
    # max |x| = 127 makes the scale exactly 1, so each x / scale is x itself
    x = np.array([[127.0, 2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5, 126.5, -127.0]])
    codes, scales = oracle.quantize_q8(x)
    assert scales.dtype == np.float32 and scales[0] == 1.0
    assert codes.tolist() == [[127, 2, 4, -2, -4, 0, 0, 2, 126, -127]]


def test_scale_is_the_fp32_quotient_and_the_absmax_maps_to_127():
    x = torch.randn(64, 128, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    codes, scales = oracle.quantize_q8(x)
    xf = x.float().numpy()
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(scales, (amax / np.float32(127)).astype(np.float32))
    row_max_code = np.abs(codes.astype(np.int32)).max(axis=1)
    assert (row_max_code == 127).all()
    assert codes.dtype == np.int8 and np.abs(codes.astype(np.int32)).max() <= 127


def test_round_trip_error_is_at_most_half_a_step():
    x = torch.randn(256, 128, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    codes, scales = oracle.quantize_q8(x)
    back = oracle.dequantize_q8(codes, scales)
    err = np.abs(back - x.double().numpy())
    # half a quantisation step, plus the fp32 roundings of max|x| / 127 and of
    # x / scale (each at most 127 * 2^-24 of a step)
    assert (err <= scales.astype(np.float64)[:, None] * (0.5 + 2e-5)).all()


def test_zero_tokens_get_zero_scale_and_codes():
    x = np.zeros((3, 64))
    x[1, 5] = -2.0
    codes, scales = oracle.quantize_q8(x)
    assert scales[0] == 0 and scales[2] == 0 and (codes[[0, 2]] == 0).all()
    assert codes[1, 5] == -127 and np.count_nonzero(codes[1]) == 1


def test_exactly_representable_cache_gives_plain_attention():
    # values that are integer multiples of a power-of-two per-token scale are
    # exact in fp32 and quantise without loss, so attention over the codes must
    # equal attention over the values
    rng = np.random.default_rng(21)
    B, H_q, H_kv, S, d = 2, 8, 2, 40, 32
    sk = 2.0 ** -rng.integers(4, 9, size=(B, H_kv, S))
    sv = 2.0 ** -rng.integers(4, 9, size=(B, H_kv, S))
    ik = rng.integers(-127, 128, size=(B, H_kv, S, d))
    iv = rng.integers(-127, 128, size=(B, H_kv, S, d))
    ik[..., 0], iv[..., 0] = 127, -127  # pin each token's absmax
    sk, sv = sk.astype(np.float32), sv.astype(np.float32)
    K = ik * sk.astype(np.float64)[..., None]
    V = iv * sv.astype(np.float64)[..., None]
    kc, ks = oracle.quantize_q8(K.astype(np.float32))
    vc, vs = oracle.quantize_q8(V.astype(np.float32))
    q = rng.standard_normal((B, H_q, d))
    seqlens = [40, 13]
    assert np.array_equal(kc, ik) and np.array_equal(ks, sk)
    assert np.array_equal(vc, iv) and np.array_equal(vs, sv)
    O, L = oracle.attention_q8(q, kc, ks, vc, vs, scale=0.2, seqlens=seqlens)
    O2, L2 = oracle.attention(q[:, :, None], K, V, scale=0.2, seqlens=seqlens)
    assert np.allclose(O, O2[:, :, 0], rtol=0, atol=1e-12)
    assert np.allclose(L, L2[:, :, 0], rtol=0, atol=1e-12)
