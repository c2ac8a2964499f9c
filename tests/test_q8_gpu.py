"""GPU parity of the INT8 KV cache path.

Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §4 item 3 (INT8
KV quantisation; the scheme is the reading stated in the header and the
oracle). The quantiser must reproduce the oracle's codes and scales bit for
bit (integer work), and decode over a cache of the oracle's codes must match
the oracle's attention over the dequantised cache within the decode
tolerance: max |dO| <= 1e-2, mean |dO| <= 1e-3, |d lse| <= 1e-3.
"""

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle as orc
from _fullsize import workers
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


def _assert_close(o, lse, O_ref, L_ref, what):
    o = o.float().cpu().double().numpy().reshape(O_ref.shape)
    l = lse.cpu().double().numpy().reshape(L_ref.shape)
    err = np.abs(o - O_ref)
    assert np.isfinite(o).all(), what
    assert err.max() <= MAX_ABS, f"{what} max|dO|={err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what} mean|dO|={err.mean():.3e}"
    fin = np.isfinite(L_ref)
    assert (np.isneginf(l) == ~fin).all(), what
    if fin.any():
        assert np.abs(l[fin] - L_ref[fin]).max() <= LSE_ABS, what


def _stored(codes):
    """The library's storage of int8 codes: the bytes code + 128."""
    return (np.asarray(codes).astype(np.int16) + 128).astype(np.uint8)


def _oracle_cache(k, v):
    """The oracle's codes and scales, in the kernel's layouts, on the GPU."""
    kc, ks = orc.quantize_q8(k)
    vc, vs = orc.quantize_q8(v)
    dev = "cuda"
    return (kc, ks, vc, vs,
            torch.from_numpy(_stored(kc)).to(dev),
            torch.from_numpy(np.ascontiguousarray(np.swapaxes(_stored(vc), 2, 3))).to(dev),
            torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev))


def test_quantiser_matches_the_oracle_bit_for_bit():
    B, H_kv, S, d = 2, 3, 96, 128
    g = torch.Generator().manual_seed(41)
    k = torch.randn(B, H_kv, S, d, generator=g).to(torch.bfloat16)
    v = (3 * torch.randn(B, H_kv, S, d, generator=g)).to(torch.bfloat16)
    # a token whose scale is exactly 1 and whose other values are ties
    tie = torch.tensor([127.0] + [(-1) ** i * (i % 5 + 0.5) for i in range(d - 1)])
    k[0, 0, 5] = tie.to(torch.bfloat16)
    v[1, 2, 7] = (-tie).to(torch.bfloat16)
    k[1, 1, 9] = 0   # all-zero tokens
    v[0, 1, 95] = 0
    kc, vc, ks, vs = api.quantize_kv_q8(k.cuda(), v.cuda())
    api.check()
    okc, oks = orc.quantize_q8(k)
    ovc, ovs = orc.quantize_q8(v)
    assert np.array_equal(kc.cpu().numpy(), _stored(okc))
    assert np.array_equal(vc.cpu().numpy(), np.swapaxes(_stored(ovc), 2, 3))
    assert np.array_equal(ks.cpu().numpy(), oks)
    assert np.array_equal(vs.cpu().numpy(), ovs)
    assert oks[0, 0, 5] == 1.0 and okc[0, 0, 5, 1] == 0  # rint(0.5) = 0


@pytest.mark.parametrize("S_max,G", [(1024, 8), (3008, 4), (160, 1), (1024, 16)])
def test_decode_matches_the_oracle_on_ragged_rows(S_max, G):
    lens = sorted({0, 1, 15, 16, 17, 63, 64, 65, min(100, S_max), S_max // 2 + 3, S_max})
    B, H_kv, d = len(lens), 2, 128
    q, k, v, _ = wl.small_decode(B, G * H_kv, H_kv, d, S_max, seed=900 + S_max + G)
    kc, ks, vc, vs, dkc, dvc, dks, dvs = _oracle_cache(k, v)
    # padding beyond each row's length: garbage codes and NaN scales must not leak
    for b, n in enumerate(lens):
        dkc[b, :, n:] = 205
        dvc[b, :, :, n:] = 37
        dks[b, :, n:] = float("nan")
        dvs[b, :, n:] = float("nan")
    sl = torch.tensor(lens, dtype=torch.int32)
    O, L = orc.attention_q8(q, kc, ks, vc, vs, scale=1 / math.sqrt(d), seqlens=lens)
    for ns in (0, 1, 2, 3, 16, 32):
        o, lse = api.decode_q8(q.cuda(), dkc, dvc, dks, dvs, sl.cuda(), num_splits=ns)
        api.check()
        _assert_close(o, lse, O, L, f"S={S_max} G={G} ns={ns}")


def test_full_size_8k_decode_through_the_gpu_quantiser():
    w = wl.LLAMA70B_DECODE_8K
    q, k, v, sl = wl.decode_inputs(w)
    kc, vc, ks, vs = api.quantize_kv_q8(k.cuda(), v.cuda())
    o, lse = api.decode_q8(q.cuda(), kc, vc, ks, vs, sl.cuda())
    api.check()
    okc, oks = orc.quantize_q8(k)
    ovc, ovs = orc.quantize_q8(v)
    assert np.array_equal(kc.cpu().numpy(), _stored(okc))
    assert np.array_equal(ks.cpu().numpy(), oks)
    O, L = orc.attention_q8(q, okc, oks, ovc, ovs, scale=w.scale, seqlens=sl.tolist())
    _assert_close(o, lse, O, L, "8K")
    # the quantised cache stays close to the bf16 one (information only: the
    # parity bar above is against the dequantised cache)
    O16, _ = orc.attention(q[:, :, None], k, v, scale=w.scale, seqlens=sl.tolist())
    assert np.abs(O - O16[:, :, 0]).max() < 0.05


def test_small_batch_one_wave_every_row():
    # B = 4 at 8K: the plan takes one wave of 4-split clusters (3 warps x 2
    # stages per CTA); every row against attention over the oracle's cache
    B, H_kv, G, S, d = 4, 8, 8, 8192, 128
    lens = [8192, 6000, 64, 8191]
    q, k, v, _ = wl.small_decode(B, G * H_kv, H_kv, d, S, seed=960, seqlens=lens)
    kc, ks, vc, vs, dkc, dvc, dks, dvs = _oracle_cache(k, v)
    o, lse = api.decode_q8(q.cuda(), dkc, dvc, dks, dvs,
                           torch.tensor(lens, dtype=torch.int32).cuda())
    api.check()
    O, L = orc.attention_q8(q, kc, ks, vc, vs, scale=1 / math.sqrt(d), seqlens=lens)
    _assert_close(o, lse, O, L, "B=4 8K one wave")


def test_ragged_128k_every_head():
    # All 4 x 64 query-head rows of the ragged 128K batch over the GPU
    # quantiser's cache, against attention over the oracle's dequantised
    # cache (the codes are compared bit for bit on one group first).
    w = wl.RAGGED_DECODE_128K
    q, k, v, sl = wl.decode_inputs(w)
    kc, vc, ks, vs = api.quantize_kv_q8(k.cuda(), v.cuda())
    o, lse = api.decode_q8(q.cuda(), kc, vc, ks, vs, sl.cuda())
    api.check()
    o, lse = o.cpu(), lse.cpu()
    G = w.H_q // w.H_kv
    n0 = int(sl[0])
    kc0, ks0 = orc.quantize_q8(k[0:1, 0:1, :n0])
    assert np.array_equal(kc[0:1, 0:1, :n0].cpu().numpy(), _stored(kc0))
    assert np.array_equal(ks[0:1, 0:1, :n0].cpu().numpy(), ks0)
    del kc, vc, ks, vs

    def group(bk):
        b, kv = bk
        n = int(sl[b])
        kcb, ksb = orc.quantize_q8(k[b:b + 1, kv:kv + 1, :n])
        vcb, vsb = orc.quantize_q8(v[b:b + 1, kv:kv + 1, :n])
        return bk, orc.attention_q8(q[b:b + 1, kv * G:(kv + 1) * G], kcb, ksb, vcb, vsb,
                                    scale=w.scale)

    with ThreadPoolExecutor(workers(3.0)) as ex:
        for (b, kv), (O, L) in ex.map(group, [(b, kv) for b in range(w.B)
                                              for kv in range(w.H_kv)]):
            _assert_close(o[b:b + 1, kv * G:(kv + 1) * G], lse[b:b + 1, kv * G:(kv + 1) * G],
                          O, L, f"b={b} kv={kv}")


@pytest.mark.parametrize("e", [16, -20])
def test_query_magnitudes_outside_the_f16_range(e):
    # The kernel runs its MMAs in f16. q * 2^16 has entries beyond f16's
    # largest value (65504) and q * 2^-20 entries in f16's subnormals; with the
    # scale divided by the same power of two the scores are those of q itself,
    # so the result must match the oracle on (q * 2^e, scale * 2^-e).
    S_max, G, H_kv, d = 1024, 8, 2, 128
    lens = [1024, 700, 1]
    q, k, v, _ = wl.small_decode(len(lens), G * H_kv, H_kv, d, S_max, seed=930)
    qs = (q.float() * 2.0 ** e).to(torch.bfloat16)
    assert torch.equal(qs.float(), q.float() * 2.0 ** e)  # exact power-of-two scaling
    if e > 0:
        assert qs.float().abs().max() > 65504
    scale = 2.0 ** -e / math.sqrt(d)
    kc, ks, vc, vs, dkc, dvc, dks, dvs = _oracle_cache(k, v)
    O, L = orc.attention_q8(qs, kc, ks, vc, vs, scale=scale, seqlens=lens)
    for ns in (1, 4):
        o, lse = api.decode_q8(qs.cuda(), dkc, dvc, dks, dvs,
                               torch.tensor(lens, dtype=torch.int32).cuda(), num_splits=ns,
                               scale=scale)
        api.check()
        _assert_close(o, lse, O, L, f"q x 2^{e} ns={ns}")


def test_decode_rejects_unsupported_shapes():
    q = torch.zeros(1, 8, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, 1, 64, 64, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(1, 1, 64, device="cuda")
    with pytest.raises(api.GqaError) as e:
        api.decode_q8(q, kc, kc.clone(), sc, sc.clone())
    assert e.value.code == api.GQA_ERR_UNSUPPORTED
