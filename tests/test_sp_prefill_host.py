"""Sequence-parallel prefill across ranks, host side (no GPU): world size 2
over gloo. Page "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)", §5.5
(prefill with SP: the ranks hold slices of the keys) and §4 (the partials
meet in a log-sum-exp reduce-to-root, normalised once at the root).

Each rank takes its key slice from the library's split plan
(gqa_attn_split_bounds with one split per rank) and computes the partial of
every query row over that slice, causal in global positions (the fp64 oracle
stands in for the rank's GPU prefill here; a row that sees no key of the slice
is (O = 0, lse = -inf)). The partials travel to rank 0 with one all_gather of
(d + 1) fp32 values per row; rank 0 merges them with the log-sum-exp rule,
written out in this test, and the result must equal the oracle's causal
prefill over all keys.
"""

import math
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as orc
from gqa_attention_split_gb300 import api, build
from gqa_attention_split_gb300 import workloads as wl

B, H_q, H_kv, D, T_Q, S, OFF = 1, 4, 2, 32, 96, 300, 100


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _slice_partial(q, k, v, a, b):
    """Rows' partial over keys [a, b): query t (global OFF + t) sees key a + j
    iff a + j <= OFF + t; built from the oracle's plain definition."""
    O = np.zeros((B, H_q, T_Q, D))
    L = np.full((B, H_q, T_Q), -np.inf)
    G = H_q // H_kv
    for h in range(H_q):
        for t in range(T_Q):
            n = min(b, OFF + t + 1) - a  # visible keys of the slice
            if n <= 0:
                continue
            o, l = orc.attention_rows(q, k[:, :, a:a + n], v[:, :, a:a + n], [(0, h, t)],
                                      scale=1 / math.sqrt(D))
            O[0, h, t], L[0, h, t] = o[0], l[0]
    return O, L


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        build.build()
        q, k, v = wl.small_prefill(B, H_q, H_kv, D, T_Q, S, OFF, seed=1600)
        rc, bounds = api.gqa_attn_split_bounds(S, world, S)
        assert rc == 0
        a, b = bounds[rank]
        O_r, L_r = _slice_partial(q, k, v, a, b)
        rec = torch.cat([torch.from_numpy(O_r).float(),
                         torch.from_numpy(L_r).float()[..., None]], dim=-1)
        gathered = [torch.empty_like(rec) for _ in range(world)]
        dist.all_gather(gathered, rec)
        if rank == 0:
            parts = torch.stack(gathered).double().numpy()   # [R, B, H_q, T_q, D + 1]
            Os, lses = parts[..., :D], parts[..., D]
            mx = lses.max(axis=0)
            w = np.exp(lses - mx)                           # every row sees key 0 somewhere
            tot = w.sum(axis=0)
            out["o"] = ((w[..., None] * Os).sum(axis=0) / tot[..., None]).tolist()
            out["lse"] = (mx + np.log(tot)).tolist()
            out["empty_rows_rank1"] = int(np.isneginf(lses[1]).sum())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_merge_to_the_whole_causal_prefill():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        O, L = np.array(out["o"]), np.array(out["lse"])
        # rank 1 holds keys [150, 300): queries 100 .. 149 see none of them, and
        # their (0, -inf) partials must drop out of the merge
        assert out["empty_rows_rank1"] == H_q * 50
    q, k, v = wl.small_prefill(B, H_q, H_kv, D, T_Q, S, OFF, seed=1600)
    O_ref, L_ref = orc.attention(q, k, v, scale=1 / math.sqrt(D), causal=True, q_offset=OFF)
    assert np.abs(O - O_ref).max() < 1e-5
    assert np.abs(L - L_ref).max() < 1e-4
