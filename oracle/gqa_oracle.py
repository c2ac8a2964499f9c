"""fp64 CPU oracle for grouped-query attention (decode split-KV and causal prefill).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The CUDA library never calls it and shares no code with it.

What it follows (page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)",
kernbench2):

* Algorithm lineage: the kernel is FlashAttention (tiled, online softmax),
  its split-and-combine is FlashDecoding; no new mathematics. So where the
  method reaches a result with a plain definition, the oracle is that
  definition: softmax(Q K^T * scale + mask) V, computed in fp64 with explicit
  K/V head repetition (``attention``, ``attention_rows``).
* §0.5 I/O contract: inputs are per-KV-head query groups Q[G, T_q, d] (post-RoPE),
  read-only K/V caches [S, d], softmax_scale = 1/sqrt(d); the output is
  O = O_acc / l_acc. Query head h therefore reads KV head h // G.
* §3 per-tile op sequence (also the TL;DR pseudocode): the running (m, l, O)
  recurrence, written out step by step in ``online_softmax_sweep``.
* §4 reduction: the log-sum-exp merge of two partial triples, ``lse_merge``,
  and normalisation once at the root (``combine_partials``).
* §5.2 decode without sequence parallelism: T_q = 1, every past key visible,
  only the ragged tail masked.
* §5.4 prefill without sequence parallelism: the three tile classes
  (all-past, all-future, partial) of a query block against a KV tile,
  ``tile_class``; future tiles are skipped, partial tiles get a boundary mask.

Readings where the page is silent (each restated in the design notes):

* lse is the natural log of sum(exp(score)) over the visible, scaled scores.
* A decode row with zero visible keys gives O = 0 and lse = -inf.
* Causal visibility with an offset: key j is visible to query t iff
  j <= q_offset + t (the new queries' keys are already in the cache).
* Decode split plan: on one GPU the page's round-robin token placement has
  no counterpart; splits are contiguous chunks of L = ceil(S_max / num_splits)
  keys on the S_max grid, clipped to the row's seqlen.

Every array argument may be any real dtype (bf16 tensors are widened by the
caller via ``to_f64``); all arithmetic here is float64.
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf

# Tile classes of §5.4 (prefill, no SP).
TILE_ALL_PAST = 0
TILE_PARTIAL = 1
TILE_ALL_FUTURE = 2


def to_f64(x) -> np.ndarray:
    """Widen a torch tensor (any float dtype, incl. bf16) or array to float64 exactly."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # local: torch only as a container format here

        return x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# The plain definition (§0.5 contract; lineage: "no new math").
# ---------------------------------------------------------------------------


def visible_count(t: int, S: int, *, seqlen: int | None, causal: bool, q_offset: int) -> int:
    """Number of keys query position t may attend to (keys 0..n-1 are visible).

    decode (§5.2): all keys below the row's seqlen.
    causal prefill (§5.4): key j visible iff j <= q_offset + t.
    non-causal prefill: all S keys.
    """
    if seqlen is not None:
        return int(seqlen)
    if causal:
        return min(S, q_offset + t + 1)
    return S


def _softmax_attend(scores: np.ndarray, V: np.ndarray):
    """Row-wise softmax of ``scores`` [T, n] (entries may be -inf) applied to V [n, d].

    Returns (O [T, d], lse [T], P [T, n]). A row that is entirely -inf gives
    O = 0, lse = -inf and P = 0.
    """
    T, n = scores.shape
    m = scores.max(axis=1) if n > 0 else np.full(T, NEG_INF)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    P = np.exp(scores - safe_m[:, None]) if n > 0 else np.zeros((T, 0))
    l = P.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        W = np.where(l[:, None] > 0, P / np.where(l > 0, l, 1.0)[:, None], 0.0)
        lse = np.where(l > 0, safe_m + np.log(np.where(l > 0, l, 1.0)), NEG_INF)
    O = W @ V if n > 0 else np.zeros((T, V.shape[1]))
    return O, lse, W


def attention(q, k, v, *, scale: float, seqlens=None, causal: bool = False,
              q_offset: int = 0, return_weights: bool = False):
    """softmax(Q K^T * scale + mask) V in fp64, with K/V heads repeated explicitly.

    q: [B, H_q, T_q, d]; k, v: [B, H_kv, S, d]; seqlens: None or [B] ints
    (decode: keys j < seqlens[b] are visible). Returns O [B, H_q, T_q, d],
    lse [B, H_q, T_q] (natural log) and, if asked, the weights [B, H_q, T_q, S].
    Meant for small shapes: it materialises the repeated K/V and all scores.
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    B, H_q, T_q, d = q.shape
    H_kv, S = k.shape[1], k.shape[2]
    assert H_q % H_kv == 0
    G = H_q // H_kv
    # §5.2: the G query heads of one KV head are adjacent, so head h uses KV
    # head h // G. Repeat each KV head G times, explicitly.
    k_rep = np.repeat(k, G, axis=1)
    v_rep = np.repeat(v, G, axis=1)
    O = np.zeros((B, H_q, T_q, d))
    lse = np.zeros((B, H_q, T_q))
    W_all = np.zeros((B, H_q, T_q, S)) if return_weights else None
    for b in range(B):
        sl = None if seqlens is None else int(seqlens[b])
        for h in range(H_q):
            scores = (q[b, h] @ k_rep[b, h].T) * scale  # [T_q, S]
            for t in range(T_q):
                n = visible_count(t, S, seqlen=sl, causal=causal, q_offset=q_offset)
                scores[t, n:] = NEG_INF
            O[b, h], lse[b, h], W = _softmax_attend(scores, v_rep[b, h])
            if return_weights:
                W_all[b, h] = W
    if return_weights:
        return O, lse, W_all
    return O, lse


def attention_rows(q, k, v, rows, *, scale: float, seqlens=None, causal: bool = False,
                   q_offset: int = 0):
    """The same definition, one output row at a time, for sampling large problems.

    rows: iterable of (b, h, t). q: [B, H_q, T_q, d] (decode: T_q = 1);
    k, v: [B, H_kv, S, d] (torch or numpy; only the rows read are widened).
    Returns (O [len(rows), d], lse [len(rows)]).
    """
    rows = list(rows)
    H_q = q.shape[1]
    H_kv, S = k.shape[1], k.shape[2]
    G = H_q // H_kv
    d = q.shape[-1]
    O = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    for i, (b, h, t) in enumerate(rows):
        kv = h // G  # explicit query-head -> KV-head map
        sl = None if seqlens is None else int(seqlens[b])
        n = visible_count(t, S, seqlen=sl, causal=causal, q_offset=q_offset)
        qr = to_f64(q[b, h, t])
        Kr = to_f64(k[b, kv, :n])
        Vr = to_f64(v[b, kv, :n])
        scores = (Kr @ qr)[None, :] * scale
        o, l_, _ = _softmax_attend(scores, Vr)
        O[i], lse[i] = o[0], l_[0]
    return O, lse


# ---------------------------------------------------------------------------
# The tiled recurrence of §3 (and the TL;DR pseudocode), step by step.
# ---------------------------------------------------------------------------


def init_running(rows: int, d: int):
    """Running state (m, l, O) = (-inf, 0, zeros), the persistent arena of §3."""
    return np.full(rows, NEG_INF), np.zeros(rows), np.zeros((rows, d))


def online_softmax_sweep(q_g, K, V, *, scale: float, tile: int, n_valid: int,
                         key_pos0: int = 0, query_pos=None):
    """One rank's sweep over its KV slice, tile by tile, as §3 orders the steps.

    q_g: [M, d] (the G*T_q folded query rows); K, V: [n, d] (the slice);
    keys 0..n_valid-1 of the slice are valid; ``key_pos0`` is the global
    position of the slice's first key. ``query_pos`` (optional, [M]) holds each
    row's last visible global key position for the causal boundary mask; None
    means no causal mask. Returns the unnormalised partial (m, l, O).
    """
    q_g, K, V = to_f64(q_g), to_f64(K), to_f64(V)
    M, d = q_g.shape
    m, l, O = init_running(M, d)
    n_tiles = math.ceil(n_valid / tile)
    for j in range(n_tiles):
        ks, ke = j * tile, min((j + 1) * tile, n_valid)
        # S_j = q_g . K_j^T * scale
        Sj = (q_g @ K[ks:ke].T) * scale
        # additive mask: -inf on keys this row may not see
        mask = np.zeros_like(Sj)
        if query_pos is not None:
            kpos = key_pos0 + np.arange(ks, ke)
            mask[kpos[None, :] > np.asarray(query_pos)[:, None]] = NEG_INF
        Sj = Sj + mask
        # online softmax merge
        m_new = np.maximum(m, Sj.max(axis=1))
        safe = np.where(np.isfinite(m_new), m_new, 0.0)
        P = np.exp(Sj - safe[:, None])
        corr = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
        l = l * corr + P.sum(axis=1)
        Oj = P @ V[ks:ke]
        O = O * corr[:, None] + Oj
        m = m_new
    return m, l, O


# ---------------------------------------------------------------------------
# §4 reduction: log-sum-exp merge, normalise once at the root.
# ---------------------------------------------------------------------------


def lse_merge(m_a, l_a, O_a, m_b, l_b, O_b):
    """Merge two unnormalised partials (§4): m = max, rescale both, add."""
    m_a, l_a, O_a = np.asarray(m_a, float), np.asarray(l_a, float), np.asarray(O_a, float)
    m_b, l_b, O_b = np.asarray(m_b, float), np.asarray(l_b, float), np.asarray(O_b, float)
    m = np.maximum(m_a, m_b)
    safe = np.where(np.isfinite(m), m, 0.0)
    sa = np.where(np.isfinite(m_a), np.exp(m_a - safe), 0.0)
    sb = np.where(np.isfinite(m_b), np.exp(m_b - safe), 0.0)
    return m, l_a * sa + l_b * sb, O_a * sa[..., None] + O_b * sb[..., None]


def finalize(m, l, O):
    """O / l and lse = m + ln l; a row with l = 0 gives O = 0, lse = -inf."""
    m, l, O = np.asarray(m, float), np.asarray(l, float), np.asarray(O, float)
    pos = l > 0
    Of = np.where(pos[..., None], O / np.where(pos, l, 1.0)[..., None], 0.0)
    lse = np.where(pos, m + np.log(np.where(pos, l, 1.0)), NEG_INF)
    return Of, lse


def combine_partials(ms, ls, Os):
    """Fold partials s = 0, 1, ... in order with ``lse_merge``; then ``finalize``.

    ms, ls: [ns, ...]; Os: [ns, ..., d].
    """
    m, l, O = ms[0], ls[0], Os[0]
    for s in range(1, len(ms)):
        m, l, O = lse_merge(m, l, O, ms[s], ls[s], Os[s])
    return finalize(m, l, O)


# ---------------------------------------------------------------------------
# Integer work: decode split plan and prefill tile classes.
# ---------------------------------------------------------------------------


def split_len(S_max: int, num_splits: int) -> int:
    """Keys per split: L = ceil(S_max / num_splits)."""
    return -(-S_max // num_splits)


def split_bounds(S_max: int, num_splits: int, seqlen: int):
    """[start, end) of every split s = 0..num_splits-1 for one row.

    Split s covers [s*L, (s+1)*L) on the S_max grid, clipped to [0, seqlen);
    an empty split has start == end. (Reading: contiguous chunks stand in for
    the page's round-robin placement, §0 / §2.)
    """
    L = split_len(S_max, num_splits)
    out = []
    for s in range(num_splits):
        start = min(s * L, seqlen)
        end = min((s + 1) * L, seqlen)
        out.append((start, end))
    return out


def split_partials(q, k, v, *, scale: float, seqlens, num_splits: int):
    """Per-split unnormalised partials of a decode problem, from the definition.

    q: [B, H_q, d]; k, v: [B, H_kv, S_max, d]. Each split's (m, l, O) is the
    plain softmax restricted to its key range: m = max score, l = sum exp(s - m),
    O = sum exp(s - m) v. Empty splits give (-inf, 0, 0).
    Returns ms, ls [ns, B, H_q] and Os [ns, B, H_q, d].
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    B, H_q, d = q.shape
    H_kv, S_max = k.shape[1], k.shape[2]
    G = H_q // H_kv
    ms = np.full((num_splits, B, H_q), NEG_INF)
    ls = np.zeros((num_splits, B, H_q))
    Os = np.zeros((num_splits, B, H_q, d))
    for b in range(B):
        sl = S_max if seqlens is None else int(seqlens[b])
        for s, (start, end) in enumerate(split_bounds(S_max, num_splits, sl)):
            if end <= start:
                continue
            for h in range(H_q):
                kv = h // G
                sc = (k[b, kv, start:end] @ q[b, h]) * scale
                mx = sc.max()
                p = np.exp(sc - mx)
                ms[s, b, h] = mx
                ls[s, b, h] = p.sum()
                Os[s, b, h] = p @ v[b, kv, start:end]
    return ms, ls, Os


def tile_class(qs: int, qe: int, ks: int, ke: int) -> int:
    """§5.4 classification of query block [qs, qe) against KV tile [ks, ke).

    Positions are global (a chunk at q_offset passes qs + q_offset, qe + q_offset).
    ke <= qs -> all past (no mask); ks >= qe -> all future (skip);
    otherwise partial (boundary mask).
    """
    if ke <= qs:
        return TILE_ALL_PAST
    if ks >= qe:
        return TILE_ALL_FUTURE
    return TILE_PARTIAL


def prefill_tile_classes(T_q: int, S_kv: int, q_offset: int, block_m: int, block_n: int):
    """Class of every (m-tile, n-tile) pair: int array [ceil(T_q/BM), ceil(S_kv/BN)]."""
    nm = -(-T_q // block_m)
    nn = -(-S_kv // block_n)
    out = np.zeros((nm, nn), dtype=np.int64)
    for i in range(nm):
        qs = q_offset + i * block_m
        qe = q_offset + min((i + 1) * block_m, T_q)
        for j in range(nn):
            out[i, j] = tile_class(qs, qe, j * block_n, min((j + 1) * block_n, S_kv))
    return out


# ---------------------------------------------------------------------------
# Hard-capped ring-buffer KV cache with attention sinks.
#
# Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §2 item 4 (the KV
# cache is initialised with a fixed max_tokens and never grows) and §4 item 2
# (once the ring wraps, the oldest entries are overwritten under an
# attention-sink + local-window policy). Readings where the page is silent:
#   * the first n_sink tokens of a row are the sinks and are never
#     overwritten; every later token overwrites the oldest non-sink token, so
#     the cache holds the sinks plus the last (capacity - n_sink) tokens;
#   * a decode step attends to exactly the tokens the cache holds.
# Everything below works at the token level (which token ids are visible,
# which slot a token id lands in), never at the kernel's level.
# ---------------------------------------------------------------------------


def ring_slot(t: int, capacity: int, n_sink: int) -> int:
    """Cache slot of token t: sinks keep their own slot, the rest cycle."""
    assert 0 <= n_sink < capacity and t >= 0
    if t < n_sink:
        return t
    return n_sink + (t - n_sink) % (capacity - n_sink)


def ring_visible_tokens(seqlen: int, capacity: int, n_sink: int):
    """Token ids a row of `seqlen` tokens keeps: the sinks, then the window."""
    assert 0 <= n_sink < capacity and seqlen >= 0
    sinks = list(range(min(seqlen, n_sink)))
    window = capacity - n_sink
    recent_start = max(n_sink, seqlen - window)
    return sinks + list(range(recent_start, seqlen))


def ring_write(stream, seqlen: int, capacity: int, n_sink: int, fill=np.nan):
    """Replays the writes of tokens 0 .. seqlen-1 of `stream` ([T, ...], T >=
    seqlen) into a cache of `capacity` slots, one token at a time in order;
    slots never written hold `fill`. Returns the cache [capacity, ...]."""
    stream = np.asarray(stream)
    cache = np.full((capacity,) + stream.shape[1:], fill, dtype=np.float64)
    for t in range(seqlen):
        cache[ring_slot(t, capacity, n_sink)] = stream[t]
    return cache


def attention_ring(q, k_stream, v_stream, *, scale: float, seqlens, capacity: int,
                   n_sink: int):
    """Decode attention under the sink + window policy, by its definition:
    softmax over the visible tokens of each row's token stream.

    q: [B, H_q, d]; k_stream, v_stream: [B, H_kv, T, d] (every token the row
    has produced, T >= max seqlens). Returns O [B, H_q, d], lse [B, H_q].
    """
    q = to_f64(q)
    B, H_q, d = q.shape
    H_kv = k_stream.shape[1]
    G = H_q // H_kv
    O = np.zeros((B, H_q, d))
    lse = np.zeros((B, H_q))
    for b in range(B):
        ids = ring_visible_tokens(int(seqlens[b]), capacity, n_sink)
        for h in range(H_q):
            kv = h // G
            if not ids:
                O[b, h], lse[b, h] = 0.0, NEG_INF
                continue
            Kr = to_f64(k_stream[b, kv, ids])
            Vr = to_f64(v_stream[b, kv, ids])
            scores = (Kr @ q[b, h])[None, :] * scale
            o, l_, _ = _softmax_attend(scores, Vr)
            O[b, h], lse[b, h] = o[0], l_[0]
    return O, lse


# ---------------------------------------------------------------------------
# INT8 KV cache.
#
# Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §4 item 3:
# optional INT4 / INT8 KV quantisation, recommended for contexts above 4 K.
# The page fixes no scheme. Reading: symmetric, one fp32 scale per (row, KV
# head, token) = max |x| / 127 over the token's d values, codes
# rint(x / scale) (round half to even) in [-127, 127]; an all-zero token gets
# scale 0 and codes 0. Both divisions are single fp32 IEEE divisions, so the
# codes are a deterministic function of the bf16 input. Dequantised values
# are code * scale, exact in fp64.
# ---------------------------------------------------------------------------


def quantize_q8(x):
    """x: [..., d] (any real dtype; bf16 values widen exactly to fp32).
    Returns (codes int8 [..., d], scales float32 [...])."""
    xf = np.asarray(to_f64(x), dtype=np.float32)
    amax = np.max(np.abs(xf), axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    nz = scale > 0
    safe = np.where(nz, scale, np.float32(1.0)).astype(np.float32)
    codes = np.rint(xf / safe[..., None]).astype(np.float32)
    codes = np.clip(codes, -127, 127)
    codes = np.where(nz[..., None], codes, 0)
    return codes.astype(np.int8), scale


def dequantize_q8(codes, scales):
    """codes [..., d] int8, scales [...] -> fp64 values codes * scale."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]


def attention_q8(q, k_codes, k_scales, v_codes, v_scales, *, scale: float, seqlens=None):
    """Decode attention over an INT8 cache, by its definition: the plain
    decode definition applied to the dequantised K and V.

    q: [B, H_q, d]; k_codes, v_codes: [B, H_kv, S, d] int8 (token-major, as
    the tokens were produced); k_scales, v_scales: [B, H_kv, S].
    Returns O [B, H_q, d], lse [B, H_q]."""
    K = dequantize_q8(k_codes, k_scales)
    V = dequantize_q8(v_codes, v_scales)
    O, lse = attention(to_f64(q)[:, :, None, :], K, V, scale=scale, seqlens=seqlens)
    return O[:, :, 0], lse[:, :, 0]


# ---------------------------------------------------------------------------
# INT4 KV cache (the other half of the same recommendation).
#
# Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §4 item 3
# (optional INT4 / INT8 KV quantisation for long contexts; no scheme given).
# Reading: the INT8 scheme above with 4-bit codes: per (batch row, KV head,
# token) one fp32 scale max|x| / 7, codes rint(x / scale) in [-7, 7] with ties
# to even, both divisions single fp32 divisions, an all-zero token with scale
# 0 and codes 0. Dequantised values are code * scale, exact in fp64.
# ---------------------------------------------------------------------------


def quantize_q4(x):
    """x: [..., d] (any real dtype; bf16 values widen exactly to fp32).
    Returns (codes int8 in [-7, 7] [..., d], scales float32 [...])."""
    xf = np.asarray(to_f64(x), dtype=np.float32)
    amax = np.max(np.abs(xf), axis=-1)
    scale = (amax / np.float32(7.0)).astype(np.float32)
    nz = scale > 0
    safe = np.where(nz, scale, np.float32(1.0)).astype(np.float32)
    codes = np.rint(xf / safe[..., None]).astype(np.float32)
    codes = np.clip(codes, -7, 7)
    codes = np.where(nz[..., None], codes, 0)
    return codes.astype(np.int8), scale


def attention_q4(q, k_codes, k_scales, v_codes, v_scales, *, scale: float, seqlens=None):
    """Decode attention over an INT4 cache, by its definition: the plain decode
    definition applied to the dequantised K and V (codes * scale).

    q: [B, H_q, d]; k_codes, v_codes: [B, H_kv, S, d] int8 codes in [-7, 7]
    (token-major); k_scales, v_scales: [B, H_kv, S]. Returns O [B, H_q, d],
    lse [B, H_q]."""
    K = np.asarray(k_codes, dtype=np.float64) * np.asarray(k_scales, dtype=np.float64)[..., None]
    V = np.asarray(v_codes, dtype=np.float64) * np.asarray(v_scales, dtype=np.float64)[..., None]
    O, lse = attention(to_f64(q)[:, :, None, :], K, V, scale=scale, seqlens=seqlens)
    return O[:, :, 0], lse[:, :, 0]
