"""GPU parity of the INT4 KV cache path.

Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §4 item 3 (INT4 /
INT8 KV quantisation; the scheme is the reading stated in the header and the
oracle: codes in [-7, 7], scale max|x|/7). The quantiser must reproduce the
oracle's codes and scales bit for bit (integer work), and decode over a cache
of the oracle's codes must match the oracle's attention over the dequantised
cache within the decode tolerance: max |dO| <= 1e-2, mean |dO| <= 1e-3,
|d lse| <= 1e-3.
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


def _packed(codes, axis):
    """The library's storage of int4 codes along `axis` (length even): nibbles
    code + 8, two per byte, the lower index in the low nibble."""
    nib = (np.asarray(codes).astype(np.int16) + 8).astype(np.uint8)
    nib = np.moveaxis(nib, axis, -1)
    out = nib[..., 0::2] | (nib[..., 1::2] << 4)
    return np.ascontiguousarray(np.moveaxis(out, -1, axis))


def _k_store(kc):   # [B, H_kv, S, d] codes -> [B, H_kv, S, d/2] bytes
    return _packed(kc, 3)


def _v_store(vc):   # [B, H_kv, S, d] codes -> [B, H_kv, d, S/2] bytes (dim-major)
    return _packed(np.swapaxes(vc, 2, 3), 3)


def _oracle_cache(k, v):
    kc, ks = orc.quantize_q4(k)
    vc, vs = orc.quantize_q4(v)
    dev = "cuda"
    return (kc, ks, vc, vs, torch.from_numpy(_k_store(kc)).to(dev),
            torch.from_numpy(_v_store(vc)).to(dev), torch.from_numpy(ks).to(dev),
            torch.from_numpy(vs).to(dev))


def test_storage_helper_by_hand():
    c = np.array([[-7, 7, 0, -1]])
    assert _packed(c, 1).tolist() == [[0x1 | (0xF << 4), 0x8 | (0x7 << 4)]]


def test_quantiser_matches_the_oracle_bit_for_bit():
    B, H_kv, S, d = 2, 3, 96, 128
    g = torch.Generator().manual_seed(42)
    k = torch.randn(B, H_kv, S, d, generator=g).to(torch.bfloat16)
    v = (3 * torch.randn(B, H_kv, S, d, generator=g)).to(torch.bfloat16)
    # a token whose scale is exactly 1 and whose other values are ties
    tie = torch.tensor([7.0] + [(-1) ** i * (i % 7 + 0.5) for i in range(d - 1)])
    k[0, 0, 5] = tie.to(torch.bfloat16)
    v[1, 2, 7] = (-tie).to(torch.bfloat16)
    k[1, 1, 9] = 0   # all-zero tokens
    v[0, 1, 95] = 0
    kc, vc, ks, vs = api.quantize_kv_q4(k.cuda(), v.cuda())
    api.check()
    okc, oks = orc.quantize_q4(k)
    ovc, ovs = orc.quantize_q4(v)
    assert np.array_equal(kc.cpu().numpy(), _k_store(okc))
    assert np.array_equal(vc.cpu().numpy(), _v_store(ovc))
    assert np.array_equal(ks.cpu().numpy(), oks)
    assert np.array_equal(vs.cpu().numpy(), ovs)
    assert oks[0, 0, 5] == 1.0 and okc[0, 0, 5, 1] == 0  # rint(0.5) = 0


@pytest.mark.parametrize("S_max,G", [(1024, 8), (3008, 4), (160, 1), (1024, 16)])
def test_decode_matches_the_oracle_on_ragged_rows(S_max, G):
    lens = sorted({0, 1, 15, 16, 17, 63, 64, 65, min(100, S_max), S_max // 2 + 3, S_max})
    B, H_kv, d = len(lens), 2, 128
    q, k, v, _ = wl.small_decode(B, G * H_kv, H_kv, d, S_max, seed=1400 + S_max + G)
    kc, ks, vc, vs, dkc, dvc, dks, dvs = _oracle_cache(k, v)
    # padding beyond each row's length: garbage codes and NaN scales must not leak
    for b, n in enumerate(lens):
        dkc[b, :, n:] = 0xA5
        n2 = (n + 1) // 2  # a byte shared by the last valid token keeps it
        dvc[b, :, :, n2:] = 0x3C
        dks[b, :, n:] = float("nan")
        dvs[b, :, n:] = float("nan")
    sl = torch.tensor(lens, dtype=torch.int32)
    O, L = orc.attention_q4(q, kc, ks, vc, vs, scale=1 / math.sqrt(d), seqlens=lens)
    for ns in (0, 1, 2, 3, 16, 32):
        o, lse = api.decode_q4(q.cuda(), dkc, dvc, dks, dvs, sl.cuda(), num_splits=ns)
        api.check()
        _assert_close(o, lse, O, L, f"S={S_max} G={G} ns={ns}")


def test_full_size_8k_decode_through_the_gpu_quantiser():
    w = wl.LLAMA70B_DECODE_8K
    q, k, v, sl = wl.decode_inputs(w)
    kc, vc, ks, vs = api.quantize_kv_q4(k.cuda(), v.cuda())
    o, lse = api.decode_q4(q.cuda(), kc, vc, ks, vs, sl.cuda())
    api.check()
    okc, oks = orc.quantize_q4(k)
    ovc, ovs = orc.quantize_q4(v)
    assert np.array_equal(kc.cpu().numpy(), _k_store(okc))
    assert np.array_equal(vc.cpu().numpy(), _v_store(ovc))
    assert np.array_equal(ks.cpu().numpy(), oks)
    O, L = orc.attention_q4(q, okc, oks, ovc, ovs, scale=w.scale, seqlens=sl.tolist())
    _assert_close(o, lse, O, L, "8K")


def test_ragged_128k_every_head():
    w = wl.RAGGED_DECODE_128K
    q, k, v, sl = wl.decode_inputs(w)
    kc, vc, ks, vs = api.quantize_kv_q4(k.cuda(), v.cuda())
    o, lse = api.decode_q4(q.cuda(), kc, vc, ks, vs, sl.cuda())
    api.check()
    o, lse = o.cpu(), lse.cpu()
    G = w.H_q // w.H_kv
    n0 = int(sl[0])
    kc0, ks0 = orc.quantize_q4(k[0:1, 0:1, :n0])
    assert np.array_equal(kc[0:1, 0:1, :n0].cpu().numpy(), _k_store(kc0))
    assert np.array_equal(ks[0:1, 0:1, :n0].cpu().numpy(), ks0)
    del kc, vc, ks, vs

    def group(bk):
        b, kv = bk
        n = int(sl[b])
        kcb, ksb = orc.quantize_q4(k[b:b + 1, kv:kv + 1, :n])
        vcb, vsb = orc.quantize_q4(v[b:b + 1, kv:kv + 1, :n])
        return bk, orc.attention_q4(q[b:b + 1, kv * G:(kv + 1) * G], kcb, ksb, vcb, vsb,
                                    scale=w.scale)

    with ThreadPoolExecutor(workers(3.0)) as ex:
        for (b, kv), (O, L) in ex.map(group, [(b, kv) for b in range(w.B)
                                              for kv in range(w.H_kv)]):
            _assert_close(o[b:b + 1, kv * G:(kv + 1) * G], lse[b:b + 1, kv * G:(kv + 1) * G],
                          O, L, f"b={b} kv={kv}")


@pytest.mark.parametrize("e", [16, -20])
def test_query_magnitudes_outside_the_f16_range(e):
    S_max, G, H_kv, d = 1024, 8, 2, 128
    lens = [1024, 700, 1]
    q, k, v, _ = wl.small_decode(len(lens), G * H_kv, H_kv, d, S_max, seed=1430)
    qs = (q.float() * 2.0 ** e).to(torch.bfloat16)
    assert torch.equal(qs.float(), q.float() * 2.0 ** e)  # exact power-of-two scaling
    scale = 2.0 ** -e / math.sqrt(d)
    kc, ks, vc, vs, dkc, dvc, dks, dvs = _oracle_cache(k, v)
    O, L = orc.attention_q4(qs, kc, ks, vc, vs, scale=scale, seqlens=lens)
    for ns in (1, 4):
        o, lse = api.decode_q4(qs.cuda(), dkc, dvc, dks, dvs,
                               torch.tensor(lens, dtype=torch.int32).cuda(), num_splits=ns,
                               scale=scale)
        api.check()
        _assert_close(o, lse, O, L, f"q x 2^{e} ns={ns}")


def test_decode_rejects_unsupported_shapes():
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, 1, 48, 64, dtype=torch.uint8, device="cuda")   # S = 48: not % 32
    vc = torch.zeros(1, 1, 128, 24, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(1, 1, 48, device="cuda")
    with pytest.raises(api.GqaError) as e:
        api.decode_q4(q, kc, vc, sc, sc.clone())
    assert e.value.code == api.GQA_ERR_UNSUPPORTED
