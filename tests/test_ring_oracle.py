"""Pins for the ring-buffer (attention sink + local window) part of the oracle.

Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §2 item 4 and §4
item 2: a KV cache of fixed capacity that, once full, overwrites its oldest
entry, keeping the attention-sink tokens. Each pin below checks the oracle
against something other than its own formulas: an explicit eviction queue,
the plain decode definition, or a closed form.
"""

import collections
import math

import numpy as np
import pytest

import oracle


def _held_by_eviction_queue(seqlen, capacity, n_sink):
    """Token ids a cache holds after `seqlen` appends, by direct simulation:
    the first n_sink ids are pinned; the others go through a FIFO that drops
    its oldest entry when the cache is full."""
    pinned, fifo = [], collections.deque()
    for t in range(seqlen):
        if len(pinned) < n_sink:
            pinned.append(t)
            continue
        if len(pinned) + len(fifo) == capacity:
            fifo.popleft()
        fifo.append(t)
    return pinned + list(fifo)


@pytest.mark.parametrize("capacity,n_sink", [(1, 0), (5, 0), (6, 2), (8, 7), (16, 4)])
def test_visible_tokens_match_an_eviction_queue(capacity, n_sink):
    for seqlen in range(0, 4 * capacity + 3):
        want = _held_by_eviction_queue(seqlen, capacity, n_sink)
        assert oracle.ring_visible_tokens(seqlen, capacity, n_sink) == want, seqlen


@pytest.mark.parametrize("capacity,n_sink", [(1, 0), (6, 2), (8, 7), (16, 4)])
def test_ring_write_holds_exactly_the_visible_tokens(capacity, n_sink):
    ids = np.arange(5 * capacity, dtype=np.float64)[:, None]  # token t carries value t
    for seqlen in range(0, 5 * capacity):
        cache = oracle.ring_write(ids, seqlen, capacity, n_sink)
        held = sorted(int(x) for x in cache[:, 0] if not np.isnan(x))
        assert held == sorted(_held_by_eviction_queue(seqlen, capacity, n_sink))
        # slots fill in order until the first wrap
        if seqlen <= capacity:
            assert np.array_equal(cache[:seqlen, 0], np.arange(seqlen))


def test_short_rows_reduce_to_plain_decode():
    rng = np.random.default_rng(11)
    B, H_q, H_kv, T, d = 3, 8, 2, 40, 16
    q = rng.standard_normal((B, H_q, d))
    k = rng.standard_normal((B, H_kv, T, d))
    v = rng.standard_normal((B, H_kv, T, d))
    seqlens = [0, 17, 40]
    O, L = oracle.attention_ring(q, k, v, scale=0.25, seqlens=seqlens, capacity=40, n_sink=3)
    O2, L2 = oracle.attention(q[:, :, None], k, v, scale=0.25, seqlens=seqlens)
    assert np.allclose(O[1:], O2[1:, :, 0], atol=1e-13) and np.allclose(L[1:], L2[1:, :, 0])
    assert np.all(O[0] == 0) and np.all(np.isneginf(L[0]))


@pytest.mark.parametrize("seqlen,capacity,n_sink", [(5, 8, 2), (8, 8, 2), (9, 8, 2),
                                                    (100, 8, 2), (100, 8, 0)])
def test_uniform_scores_give_the_mean_of_the_held_values(seqlen, capacity, n_sink):
    rng = np.random.default_rng(seqlen)
    d = 4
    q = np.zeros((1, 2, d))
    v = rng.standard_normal((1, 1, seqlen, d))
    k = rng.standard_normal((1, 1, seqlen, d))
    O, L = oracle.attention_ring(q, k, v, scale=1.0, seqlens=[seqlen], capacity=capacity,
                                 n_sink=n_sink)
    held = _held_by_eviction_queue(seqlen, capacity, n_sink)
    assert len(held) == min(seqlen, capacity)
    assert np.allclose(O[0, 0], v[0, 0, held].mean(axis=0), atol=1e-14)
    assert math.isclose(L[0, 1], math.log(len(held)), rel_tol=1e-14)


def test_attention_is_over_the_token_set_not_the_slot_order():
    # the window with sinks equals plain attention over the visible tokens laid
    # out contiguously, in any order
    rng = np.random.default_rng(5)
    d, T, cap, ns = 8, 30, 10, 3
    q = rng.standard_normal((1, 4, d))
    k = rng.standard_normal((1, 2, T, d))
    v = rng.standard_normal((1, 2, T, d))
    ids = _held_by_eviction_queue(T, cap, ns)
    perm = rng.permutation(len(ids))
    kk = k[:, :, [ids[i] for i in perm]]
    vv = v[:, :, [ids[i] for i in perm]]
    O, L = oracle.attention_ring(q, k, v, scale=0.3, seqlens=[T], capacity=cap, n_sink=ns)
    O2, L2 = oracle.attention(q[:, :, None], kk, vv, scale=0.3)
    assert np.allclose(O, O2[:, :, 0], atol=1e-13) and np.allclose(L, L2[:, :, 0])
