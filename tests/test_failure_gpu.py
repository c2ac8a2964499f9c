"""Failure reporting on the GPU without a fault: a decode launch whose first
block withholds one K/V copy (a prefill launch: one Q copy) must time out its
bounded waits (~1 s each), record the timeout in the device status word,
finish, and leave the context usable."""

import math

import numpy as np
import pytest
import torch

import oracle as orc
from gqa_attention_split_gb300 import api, build
from gqa_attention_split_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    api.lib()


@pytest.mark.parametrize("ns", [1, 16])
def test_bounded_wait_timeout_is_reported_and_next_call_is_correct(ns):
    q, k, v, sl = wl.small_decode(1, 8, 1, 128, 4096, seed=950 + ns)
    qd, kd, vd, sd = q.cuda(), k.cuda(), v.cuda(), sl.cuda()
    api.check()  # status word starts clear
    assert api.gqa_attn_debug_inject_timeout(1) == api.GQA_OK
    api.decode(qd, kd, vd, sd, num_splits=ns)
    with pytest.raises(api.GqaError) as e:
        api.check()
    assert e.value.code == api.GQA_ERR_DEVICE_TIMEOUT
    # the hook was one-shot, the context still works, the status word was cleared
    o, lse = api.decode(qd, kd, vd, sd, num_splits=ns)
    api.check()
    O, L = orc.attention(q[:, :, None], k, v, scale=1 / math.sqrt(128), seqlens=sl.tolist())
    err = np.abs(o.float().cpu().double().numpy() - O[:, :, 0])
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(lse.cpu().double().numpy() - L[:, :, 0]).max() <= 1e-3


def test_inject_rejects_negative_count():
    assert api.gqa_attn_debug_inject_timeout(-1) == api.GQA_ERR_INVALID_ARG
    assert api.gqa_attn_debug_inject_timeout(0) == api.GQA_OK


@pytest.mark.parametrize("H_q,H_kv", [(16, 2), (3, 3)])  # head pairs; block pairs (G = 1)
def test_prefill_timeout_is_reported_and_next_call_is_correct(H_q, H_kv):
    T, off = 300, 200
    q, k, v = wl.small_prefill(1, H_q, H_kv, 128, T, T + off, off, seed=960 + H_q)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    api.check()
    assert api.gqa_attn_debug_inject_timeout(1) == api.GQA_OK
    api.prefill(qd, kd, vd, q_offset=off, causal=True)
    with pytest.raises(api.GqaError) as e:
        api.check()
    assert e.value.code == api.GQA_ERR_DEVICE_TIMEOUT
    o, lse = api.prefill(qd, kd, vd, q_offset=off, causal=True)
    api.check()
    O, L = orc.attention(q, k, v, scale=1 / math.sqrt(128), causal=True, q_offset=off)
    err = np.abs(o.float().cpu().double().numpy() - O)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(lse.cpu().double().numpy() - L).max() <= 1e-3
