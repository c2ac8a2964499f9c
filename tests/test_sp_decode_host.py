"""Sequence-parallel decode across ranks, host side (no GPU): world size 2 over
gloo. Page "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)", §5.3
(decode with SP: every rank sweeps its own slice of the keys) and §4 (the
partials meet in a log-sum-exp reduce-to-root, normalised once at the root).

Each rank takes its slice from the library's split plan (gqa_attn_split_bounds
with one split per rank), computes its partial (O_r, lse_r) over that slice
(the fp64 oracle stands in for the rank's GPU decode here), and the partials
travel to rank 0 with one all_gather of (d + 1) fp32 values per row. Rank 0
merges them with the log-sum-exp rule, written out in this test, and the
result must equal the oracle's attention over the whole row.
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

LENS = [5000, 4999, 2501, 2500, 17, 0]
B, H_q, H_kv, D, S_MAX = len(LENS), 16, 2, 64, 5000


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        build.build()
        q, k, v, _ = wl.small_decode(B, H_q, H_kv, D, S_MAX, seed=1300, seqlens=LENS)
        rc, bounds = api.gqa_attn_split_bounds(S_MAX, world, S_MAX)
        assert rc == 0
        a, b = bounds[rank]
        local = [max(0, min(n, b) - a) for n in LENS]
        O_r, L_r = orc.attention(q[:, :, None], k[:, :, a:b], v[:, :, a:b],
                                 scale=1 / math.sqrt(D), seqlens=local)
        # the exchanged record: O_r and lse_r per (row, query head), fp32
        rec = torch.cat([torch.from_numpy(O_r[:, :, 0]).float(),
                         torch.from_numpy(L_r[:, :, 0]).float()[..., None]], dim=-1)
        gathered = [torch.empty_like(rec) for _ in range(world)]
        dist.all_gather(gathered, rec)
        if rank == 0:
            parts = torch.stack(gathered).double().numpy()      # [R, B, H_q, D + 1]
            Os, lses = parts[..., :D], parts[..., D]
            mx = lses.max(axis=0)
            safe = np.where(np.isfinite(mx), mx, 0.0)
            w = np.where(np.isfinite(lses), np.exp(lses - safe), 0.0)
            tot = w.sum(axis=0)
            O = np.where(tot[..., None] > 0,
                         (w[..., None] * Os).sum(axis=0) / np.where(tot > 0, tot, 1)[..., None],
                         0.0)
            lse = np.where(tot > 0, safe + np.log(np.where(tot > 0, tot, 1)), -np.inf)
            out["o"], out["lse"] = O.tolist(), lse.tolist()
            out["bytes_per_rank"] = rec.numel() * rec.element_size()
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_merge_to_the_whole_row():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        O, L = np.array(out["o"]), np.array(out["lse"])
        assert out["bytes_per_rank"] == B * H_q * (D + 1) * 4
    q, k, v, _ = wl.small_decode(B, H_q, H_kv, D, S_MAX, seed=1300, seqlens=LENS)
    O_ref, L_ref = orc.attention(q[:, :, None], k, v, scale=1 / math.sqrt(D), seqlens=LENS)
    # fp32 records: agreement to fp32 precision
    assert np.abs(O - O_ref[:, :, 0]).max() < 1e-5
    fin = np.isfinite(L_ref[:, :, 0])
    assert (np.isneginf(L) == ~fin).all()
    assert np.abs(L[fin] - L_ref[:, :, 0][fin]).max() < 1e-4
