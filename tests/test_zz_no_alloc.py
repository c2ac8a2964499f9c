"""gqa_attn_decode_noalloc: decode for callers that must not allocate device memory.

Some callers cannot call cudaMalloc (a server that fixes its HBM budget at
start-up, a host with its own allocator, a path that cannot take cudaMalloc's
implicit synchronisation). This entry point keeps its scratch in a fixed array
inside the library instead. The test calls it through the C ABI twice in a
row, on different problems that both need scratch, and checks each result
against gqa_attn_decode on the same inputs within the decode tolerance. Its
device-side errors (a bounded wait that ran out, a clamped seqlen) reach the
caller through gqa_attn_check(), which allocates nothing either. This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""

import math

import numpy as np
import pytest
import torch

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


def _both_entry_points(B, H_q, H_kv, d, S_max, lens, ns, seed):
    q, k, v, sl = wl.small_decode(B, H_q, H_kv, d, S_max, seed=seed, seqlens=lens)
    q, k, v, sl = q.cuda(), k.cuda(), v.cuda(), sl.cuda()
    stream = torch.cuda.current_stream().cuda_stream
    scale = 1.0 / math.sqrt(d)
    outs = []
    for fn in (api.gqa_attn_decode, api.gqa_attn_decode_noalloc):
        o = torch.full((B, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H_q), float("nan"), dtype=torch.float32, device="cuda")
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                sl.data_ptr(), B, H_q, H_kv, d, S_max, scale, ns, stream)
        assert rc == api.GQA_OK, api.strerror(rc)
        outs.append((o, lse))
    torch.cuda.synchronize()
    return outs


def _assert_within_tolerance(ref, got):
    (o_ref, l_ref), (o, l) = ref, got
    d_o = (o.float() - o_ref.float()).abs()
    assert torch.isfinite(o.float()).all()
    assert d_o.max().item() <= MAX_ABS and d_o.mean().item() <= MEAN_ABS
    fin = torch.isfinite(l_ref)
    assert torch.equal(torch.isneginf(l), ~fin)  # empty rows: lse = -inf on both
    assert (l[fin] - l_ref[fin]).abs().max().item() <= LSE_ABS


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    # Both problems span several 16-split clusters per row, so the partials go
    # through the fixed scratch; the second call runs over what the first left.
    cases = [dict(B=2, H_q=16, H_kv=2, d=128, S_max=40000, lens=[40000, 12345], ns=64, seed=901),
             dict(B=3, H_q=32, H_kv=4, d=64, S_max=20000, lens=[20000, 1, 9999], ns=32, seed=902)]
    for c in cases:
        need = api.gqa_attn_decode_workspace_size(c["B"], c["H_q"], c["d"], c["ns"])
        assert 0 < need <= api.NOALLOC_SCRATCH_BYTES
        ref, got = _both_entry_points(**c)
        _assert_within_tolerance(ref, got)


def test_noalloc_rejects_problems_beyond_its_scratch():
    B, H_q, d, ns = 64, 64, 128, 512
    assert api.gqa_attn_decode_workspace_size(B, H_q, d, ns) > api.NOALLOC_SCRATCH_BYTES
    fake = 1 << 16  # never dereferenced: the size check comes before any launch
    rc = api.gqa_attn_decode_noalloc(fake, fake, fake, fake, None, None, B, H_q, 8, d, 65536,
                                     0.088, ns, None)
    assert rc == api.GQA_ERR_WORKSPACE


def _noalloc(q, k, v, sl, o, lse, B, H_q, H_kv, d, S_max, ns):
    rc = api.gqa_attn_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), sl.data_ptr(), B, H_q, H_kv, d, S_max,
                                     1.0 / math.sqrt(d), ns,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == api.GQA_OK, api.strerror(rc)


def test_noalloc_device_errors_reach_check():
    B, H_q, H_kv, d, S_max, ns = 2, 8, 1, 128, 4096, 32  # two 16-split clusters per row
    q, k, v, sl = wl.small_decode(B, H_q, H_kv, d, S_max, seed=903, seqlens=[4096, 2500])
    q, k, v, sl = q.cuda(), k.cuda(), v.cuda(), sl.cuda()
    o = torch.empty((B, H_q, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H_q), dtype=torch.float32, device="cuda")
    api.check()  # start from a clear status word
    # 1) the first block withholds one copy: its bounded wait runs out (~1 s)
    assert api.gqa_attn_debug_inject_timeout(1) == api.GQA_OK
    _noalloc(q, k, v, sl, o, lse, B, H_q, H_kv, d, S_max, ns)
    with pytest.raises(api.GqaError) as e:
        api.check()
    assert e.value.code == api.GQA_ERR_DEVICE_TIMEOUT
    # the next call is correct and reports nothing
    _noalloc(q, k, v, sl, o, lse, B, H_q, H_kv, d, S_max, ns)
    api.check()
    ref = api.decode(q, k, v, sl, num_splits=ns)
    api.check()
    _assert_within_tolerance(ref, (o, lse))
    # 2) a seqlen outside [0, S_max] is clamped and reported
    bad = torch.tensor([S_max + 100, -3], dtype=torch.int32, device="cuda")
    _noalloc(q, k, v, bad, o, lse, B, H_q, H_kv, d, S_max, ns)
    with pytest.raises(api.GqaError) as e:
        api.check()
    assert e.value.code == api.GQA_ERR_DEVICE_BAD_INPUT
    api.check()  # cleared by the read
    ref = api.decode(q, k, v, torch.tensor([S_max, 0], dtype=torch.int32, device="cuda"),
                     num_splits=ns)
    api.check()
    _assert_within_tolerance(ref, (o, lse))
