"""Full-size oracle runs for the GPU parity tests (test infrastructure only).

The fp64 oracle (``oracle.attention``, unchanged) is applied to every (batch
row, KV head) group of a problem, each group with its own G query heads, in a
thread pool: numpy releases the GIL inside its array operations, and the
oracle's time goes to element-wise exp and normalisation. The number of
threads is bounded by the host's cores and free memory (one 8K causal group
holds about 3.6 GB while it runs).
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle as orc


def workers(task_gb: float) -> int:
    cpu = os.cpu_count() or 1
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE") / 2 ** 30
    except (ValueError, OSError, AttributeError):
        avail = 16.0
    return max(1, min(8, max(1, cpu // 2), int(avail // task_gb)))


def attention_by_group(q, k, v, *, scale, causal=False, q_offset=0, seqlens=None,
                       task_gb=4.0):
    """O [B, H_q, T_q, d] and lse [B, H_q, T_q] of ``oracle.attention`` on the
    whole problem, computed group by group. q [B, H_q, T_q, d], k/v
    [B, H_kv, S, d] (torch or numpy), seqlens None or [B]."""
    B, H_q = q.shape[0], q.shape[1]
    H_kv = k.shape[1]
    G = H_q // H_kv
    O = np.empty(tuple(q.shape), dtype=np.float64)
    L = np.empty(tuple(q.shape[:-1]), dtype=np.float64)

    def one(bk):
        b, kv = bk
        sl = None if seqlens is None else [int(seqlens[b])]
        o, l = orc.attention(q[b:b + 1, kv * G:(kv + 1) * G], k[b:b + 1, kv:kv + 1],
                             v[b:b + 1, kv:kv + 1], scale=scale, causal=causal,
                             q_offset=q_offset, seqlens=sl)
        O[b, kv * G:(kv + 1) * G] = o[0]
        L[b, kv * G:(kv + 1) * G] = l[0]

    with ThreadPoolExecutor(workers(task_gb)) as ex:
        list(ex.map(one, [(b, kv) for b in range(B) for kv in range(H_kv)]))
    return O, L
