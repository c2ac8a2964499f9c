"""GPU parity of the split-KV decode path against the fp64 oracle.

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


def assert_close(o_gpu, lse_gpu, O_ref, lse_ref, what=""):
    o = o_gpu.float().cpu().double().numpy().reshape(O_ref.shape)
    l = lse_gpu.float().cpu().double().numpy().reshape(lse_ref.shape)
    err = np.abs(o - O_ref)
    assert np.isfinite(o).all(), what
    assert err.max() <= MAX_ABS, f"{what} max|dO|={err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what} mean|dO|={err.mean():.3e}"
    fin = np.isfinite(lse_ref)
    assert (np.isneginf(l) == ~fin).all(), what
    if fin.any():
        dl = np.abs(l[fin] - lse_ref[fin]).max()
        assert dl <= LSE_ABS, f"{what} max|dlse|={dl:.3e}"


def run_decode(q, k, v, seqlens, ns, **kw):
    dev = "cuda"
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    sl = None if seqlens is None else seqlens.to(dev)
    o, lse = api.decode(qd, kd, vd, sl, num_splits=ns, **kw)
    api.check()
    return o, lse


def oracle_decode(q, k, v, seqlens, scale):
    return orc.attention(q[:, :, None, :], k, v, scale=scale,
                         seqlens=None if seqlens is None else seqlens.tolist())


@pytest.mark.parametrize("ns", [0, 1, 4])
def test_tiny_decode_workload(ns):
    w = wl.TINY_DECODE
    q, k, v, sl = wl.decode_inputs(w)
    o, lse = run_decode(q, k, v, sl, ns)
    O, L = oracle_decode(q, k, v, sl, w.scale)
    assert_close(o, lse, O[:, :, 0], L[:, :, 0], f"tiny ns={ns}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 12, 16])
def test_small_shapes_group_sizes(d, G):
    # G > 8: two CTAs per (split, KV head), 8 and G - 8 heads
    H_kv = 2
    q, k, v, _ = wl.small_decode(2, H_kv * G, H_kv, d, 300, seed=100 + G + d)
    sl = torch.tensor([300, 97], dtype=torch.int32)
    for ns in (1, 3, 7):
        o, lse = run_decode(q, k, v, sl, ns)
        O, L = oracle_decode(q, k, v, sl, 1 / math.sqrt(d))
        assert_close(o, lse, O[:, :, 0], L[:, :, 0], f"d={d} G={G} ns={ns}")


@pytest.mark.parametrize("d,G", [(128, 8), (64, 4), (128, 1), (128, 16), (64, 10)])
def test_cluster_merge_every_cluster_size(d, G):
    # ns = 2, 4, 8, 16 merge one cluster per row on chip; 32, 48, 64 add the
    # cross-cluster combine; 6 and 24 use clusters of 2 and 8.
    q, k, v, _ = wl.small_decode(3, 2 * G, 2, d, 3000, seed=700 + d + G)
    sl = torch.tensor([3000, 1601, 17], dtype=torch.int32)
    O, L = oracle_decode(q, k, v, sl, 1 / math.sqrt(d))
    for ns in (2, 4, 6, 8, 16, 24, 32, 48, 64):
        o, lse = run_decode(q, k, v, sl, ns)
        assert_close(o, lse, O[:, :, 0], L[:, :, 0], f"d={d} G={G} ns={ns}")


@pytest.mark.parametrize("S_max", [1, 15, 16, 17, 31, 32, 33, 100, 255, 1000])
def test_ragged_and_tiny_lengths(S_max):
    lens = sorted({0, 1, S_max // 2, max(S_max - 1, 0), S_max})
    B = len(lens)
    q, k, v, _ = wl.small_decode(B, 8, 1, 128, S_max, seed=200 + S_max)
    sl = torch.tensor(lens, dtype=torch.int32)
    for ns in sorted({1, 2, 4, S_max}):
        o, lse = run_decode(q, k, v, sl, ns)
        O, L = oracle_decode(q, k, v, sl, 1 / math.sqrt(128))
        assert_close(o, lse, O[:, :, 0], L[:, :, 0], f"S_max={S_max} ns={ns}")


def test_garbage_beyond_seqlen_is_ignored():
    # Padded cache slots past seqlen may hold anything, NaN included.
    q, k, v, _ = wl.small_decode(3, 16, 2, 128, 700, seed=300)
    sl = torch.tensor([700, 333, 1], dtype=torch.int32)
    k2, v2 = k.clone(), v.clone()
    for b, n in enumerate(sl.tolist()):
        k2[b, :, n:] = float("nan")
        v2[b, :, n:] = float("inf")
    for ns in (1, 2, 5, 29):
        o, lse = run_decode(q, k2, v2, sl, ns)
        O, L = oracle_decode(q, k, v, sl, 1 / math.sqrt(128))
        assert_close(o, lse, O[:, :, 0], L[:, :, 0], f"nan padding ns={ns}")


def test_llama70b_decode_8k_all_rows():
    w = wl.LLAMA70B_DECODE_8K
    q, k, v, sl = wl.decode_inputs(w)
    o, lse = run_decode(q, k, v, sl, 0)
    rows = [(0, h, 0) for h in range(w.H_q)]
    O, L = orc.attention_rows(q[:, :, None], k, v, rows, scale=w.scale, seqlens=sl.tolist())
    assert_close(o, lse, O.reshape(1, w.H_q, w.d), L.reshape(1, w.H_q), "llama70b 8k")
    for ns in (1, 8, 64):
        o2, lse2 = run_decode(q, k, v, sl, ns)
        assert_close(o2, lse2, O.reshape(1, w.H_q, w.d), L.reshape(1, w.H_q), f"8k ns={ns}")


@pytest.mark.parametrize("B,H_q,S,lens", [
    (1, 128, 8192, None),                 # 128 query heads on 8 KV heads (G = 16): 8 splits
    (2, 64, 8192, [8192, 5000]),          # two rows: one wave of 8-split clusters
    (4, 64, 4096, [4096, 1, 0, 3333]),    # four rows: 4 splits of 1024 keys
])
def test_automatic_plans_every_row(B, H_q, S, lens):
    # num_splits = 0 on shapes where the plan takes one wave of whole-row
    # clusters (a G = 16 group counts as two CTAs per split and KV head);
    # every row against the fp64 oracle.
    H_kv, d = 8, 128
    q, k, v, sl = wl.small_decode(B, H_q, H_kv, d, S, seed=560 + B + H_q, seqlens=lens)
    o, lse = run_decode(q, k, v, sl, 0)
    O, L = attention_by_group(q[:, :, None], k, v, scale=1 / math.sqrt(d),
                              seqlens=None if sl is None else sl.tolist())
    assert_close(o, lse, O[:, :, 0], L[:, :, 0], f"B={B} H_q={H_q} S={S}")


@pytest.mark.parametrize("B,S,lens", [
    (4, 8192, [8192, 8000, 4097, 31]),      # one wave of 4-split clusters, 6-stage rings
    (5, 20000, [20000, 1, 19999, 777, 0]),  # more CTAs than SMs: 4 warps x 2 stages
])
def test_head_dim_64_every_row(B, S, lens):
    # d = 64 streams 8 KB stages, twice as many per ring as d = 128
    H_q, H_kv, d = 32, 8, 64
    q, k, v, sl = wl.small_decode(B, H_q, H_kv, d, S, seed=580 + B, seqlens=lens)
    o, lse = run_decode(q, k, v, sl, 0)
    O, L = attention_by_group(q[:, :, None], k, v, scale=1 / math.sqrt(d), seqlens=sl.tolist())
    assert_close(o, lse, O[:, :, 0], L[:, :, 0], f"d=64 B={B} S={S}")


def _random_decode_shapes(n, seed):
    """Seeded shapes across the split plan's clauses (one wave at any SM use,
    multi-wave with a combine, G > 8 as two CTAs per split), small enough for
    the oracle: (B, H_q, H_kv, d, S_max, seqlens)."""
    rng = np.random.default_rng(seed)
    shapes = []
    while len(shapes) < n:
        B = int(rng.integers(1, 7))
        H_kv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.integers(1, 17))
        d = int(rng.choice([64, 128]))
        S = int(rng.choice([1, 200, 1000, 3000, 8192, 20000]))
        if B * H_kv * G * S * d > 60_000_000:
            continue
        lens = [int(x) for x in rng.integers(0, S + 1, size=B)]
        lens[0] = S  # one full row
        shapes.append((B, H_kv * G, H_kv, d, S, lens))
    return shapes


@pytest.mark.parametrize("B,H_q,H_kv,d,S,lens", _random_decode_shapes(16, 2024))
def test_random_shapes_automatic_plan(B, H_q, H_kv, d, S, lens):
    q, k, v, sl = wl.small_decode(B, H_q, H_kv, d, S, seed=7000 + B * S + H_q, seqlens=lens)
    o, lse = run_decode(q, k, v, sl, 0)
    O, L = attention_by_group(q[:, :, None], k, v, scale=1 / math.sqrt(d), seqlens=lens)
    assert_close(o, lse, O[:, :, 0], L[:, :, 0], f"B={B} H={H_q}/{H_kv} d={d} S={S} {lens}")


def test_single_row_128k_every_head():
    # One 128K row: the plan takes one wave of 16 splits of 8192 keys; all
    # 64 query heads against the fp64 oracle.
    w = wl.LLAMA70B_DECODE_128K_B1
    q, k, v, sl = wl.decode_inputs(w)
    o, lse = run_decode(q, k, v, sl, 0)
    O, L = attention_by_group(q[:, :, None], k, v, scale=w.scale, seqlens=sl.tolist())
    assert_close(o, lse, O[:, :, 0], L[:, :, 0], "128K single row")


def test_ragged_long_context_every_row():
    # All 4 x 64 query-head rows of the ragged 128K batch (every (row, KV head)
    # group, padded cache masked by seqlens), against the fp64 oracle.
    w = wl.RAGGED_DECODE_128K
    q, k, v, sl = wl.decode_inputs(w)
    assert sl.min() >= 16384 and sl.max() <= 131072
    o, lse = run_decode(q, k, v, sl, 0)
    O, L = attention_by_group(q[:, :, None], k, v, scale=w.scale, seqlens=sl.tolist(),
                              task_gb=3.0)
    assert_close(o, lse, O[:, :, 0], L[:, :, 0], "ragged 128K")


def test_deterministic_bitwise():
    q, k, v, sl = wl.decode_inputs(wl.LLAMA70B_DECODE_8K)
    a = run_decode(q, k, v, sl, 0)
    b = run_decode(q, k, v, sl, 0)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_lse_may_be_null_and_outputs_stay_in_bounds():
    q, k, v, _ = wl.small_decode(2, 8, 1, 64, 129, seed=400)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    pad = 64
    buf = torch.full((2 * 8 * 64 + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = buf[pad:pad + 2 * 8 * 64].view(2, 8, 64)
    rc = api.gqa_attn_decode(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), None,
                             None, 2, 8, 1, 64, 129, 0.125, 3,
                             torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    api.check()
    assert torch.isnan(buf[:pad].float()).all() and torch.isnan(buf[-pad:].float()).all()
    O, _ = oracle_decode(q, k, v, None, 0.125)
    err = np.abs(o.float().cpu().double().numpy() - O[:, :, 0])
    assert err.max() <= MAX_ABS


def test_caller_workspace_entry_point():
    q, k, v, sl = wl.small_decode(2, 16, 2, 128, 2000, seed=500, seqlens=[2000, 1234])
    ns = 6
    need = api.gqa_attn_decode_workspace_size(2, 16, 128, ns)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o, lse = run_decode(q, k, v, sl, ns, workspace=ws)
    O, L = oracle_decode(q, k, v, sl, 1 / math.sqrt(128))
    assert_close(o, lse, O[:, :, 0], L[:, :, 0], "caller workspace")
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.GqaError) as e:
        run_decode(q, k, v, sl, ns, workspace=small)
    assert e.value.code == api.GQA_ERR_WORKSPACE


def test_out_of_range_seqlen_is_clamped_and_reported():
    q, k, v, _ = wl.small_decode(2, 8, 1, 64, 100, seed=600)
    sl = torch.tensor([150, -3], dtype=torch.int32, device="cuda")
    o, lse = api.decode(q.cuda(), k.cuda(), v.cuda(), sl, num_splits=2)
    with pytest.raises(api.GqaError) as e:
        api.check()
    assert e.value.code == api.GQA_ERR_DEVICE_BAD_INPUT
    api.check()  # the status word was cleared
    O, L = oracle_decode(q, k, v, torch.tensor([100, 0]), 1 / math.sqrt(64))
    assert_close(o, lse, O[:, :, 0], L[:, :, 0], "clamped")


def test_graph_captured_before_workspace_growth_stays_valid():
    # A CUDA graph captured on a stream keeps the workspace address it saw. A
    # later call on that stream that needs a larger workspace gets a new
    # buffer; the old one must stay allocated so the graph still replays
    # correctly (the library keeps replaced buffers instead of freeing them).
    st = torch.cuda.Stream()
    q, k, v, sl = wl.small_decode(1, 16, 2, 128, 4000, seed=510, seqlens=[3999])
    qd, kd, vd, sd = q.cuda(), k.cuda(), v.cuda(), sl.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty((1, 16), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(st):
        api.decode(qd, kd, vd, sd, num_splits=32, out=o, lse=lse)  # two clusters per row
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        api.decode(qd, kd, vd, sd, num_splits=32, out=o, lse=lse)
    # a much larger problem on the same stream: the workspace grows
    q2, k2, v2, sl2 = wl.small_decode(4, 64, 8, 128, 8192, seed=511)
    with torch.cuda.stream(st):
        api.decode(q2.cuda(), k2.cuda(), v2.cuda(), sl2.cuda(), num_splits=64)
    st.synchronize()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        o.zero_()
        lse.zero_()
        g.replay()
    st.synchronize()
    api.check(st)
    O, L = oracle_decode(q, k, v, sl, 1 / math.sqrt(128))
    assert_close(o, lse, O[:, :, 0], L[:, :, 0], "graph replay after workspace growth")
