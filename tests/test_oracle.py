"""Pins for the fp64 oracle against what the mathematics and the page fix.

Page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)". Each test
pins one part of the oracle to something other than itself: closed forms
derived by hand (tests/golden), invariants of softmax attention, library
routines (torch SDPA in fp64, scipy logsumexp), brute force with Python loops,
and enumeration of the integer plans.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _ev(expr):
    return eval(expr, {"__builtins__": {}}, {"log": math.log, "exp": math.exp})


def _ev_tree(x):
    if isinstance(x, list):
        return [_ev_tree(e) for e in x]
    return _ev(x)


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --------------------------------------------------------------------------
# closed forms (tests/golden)
# --------------------------------------------------------------------------


def test_golden_attention_closed_forms():
    cases = json.load(open(GOLDEN))["attention"]
    assert len(cases) >= 4
    for c in cases:
        O, lse = orc.attention(np.array(c["q"]), np.array(c["k"]), np.array(c["v"]),
                               scale=c["scale"], seqlens=c["seqlens"], causal=c["causal"],
                               q_offset=c["q_offset"])
        np.testing.assert_allclose(O, np.array(_ev_tree(c["O"])), rtol=0, atol=1e-12,
                                   err_msg=c["name"])
        np.testing.assert_allclose(lse, np.array(_ev_tree(c["lse"])), rtol=0, atol=1e-12,
                                   err_msg=c["name"])


def test_golden_merge_closed_form():
    c = json.load(open(GOLDEN))["merge"][0]
    a, b = c["a"], c["b"]
    m, l, O = orc.lse_merge(_ev(a["m"]), _ev(a["l"]), np.array(_ev_tree(a["O"])),
                            _ev(b["m"]), _ev(b["l"]), np.array(_ev_tree(b["O"])))
    assert abs(m - _ev(c["m"])) < 1e-12
    assert abs(l - _ev(c["l"])) < 1e-12
    np.testing.assert_allclose(O, _ev_tree(c["O_unnormalised"]), atol=1e-12)
    Of, lse = orc.finalize(m, l, O)
    np.testing.assert_allclose(Of, _ev_tree(c["O"]), atol=1e-12)
    assert abs(lse - _ev(c["lse"])) < 1e-12


# --------------------------------------------------------------------------
# invariants of the definition
# --------------------------------------------------------------------------


@pytest.mark.parametrize("causal,q_offset,seqlens", [(False, 0, None), (True, 0, None),
                                                     (True, 5, None), (False, 0, [3, 11])])
def test_weights_rows_sum_to_one(causal, q_offset, seqlens):
    B, H_q, H_kv, T, S, d = 2, 4, 2, 3 if seqlens is None else 1, 11, 8
    q, k, v = _rand((B, H_q, T, d), 1), _rand((B, H_kv, S, d), 2), _rand((B, H_kv, S, d), 3)
    _, _, W = orc.attention(q, k, v, scale=0.3, seqlens=seqlens, causal=causal,
                            q_offset=q_offset, return_weights=True)
    np.testing.assert_allclose(W.sum(-1), 1.0, atol=1e-13)
    assert (W >= 0).all()
    # masked keys carry exactly zero weight
    for b, h, t in itertools.product(range(B), range(H_q), range(T)):
        n = orc.visible_count(t, S, seqlen=None if seqlens is None else seqlens[b],
                              causal=causal, q_offset=q_offset)
        assert (W[b, h, t, n:] == 0).all()


@pytest.mark.parametrize("causal,q_offset,seqlens", [(False, 0, None), (True, 2, None),
                                                     (False, 0, [1, 7])])
def test_uniform_scores_give_mean_of_visible_v(causal, q_offset, seqlens):
    B, H_q, H_kv, S, d = 2, 4, 2, 9, 5
    T = 1 if seqlens is not None else 4
    q = np.zeros((B, H_q, T, d))
    k, v = _rand((B, H_kv, S, d), 4), _rand((B, H_kv, S, d), 5)
    O, lse = orc.attention(q, k, v, scale=1.0, seqlens=seqlens, causal=causal, q_offset=q_offset)
    for b, h, t in itertools.product(range(B), range(H_q), range(T)):
        n = seqlens[b] if seqlens is not None else (q_offset + t + 1 if causal else S)
        np.testing.assert_allclose(O[b, h, t], v[b, h // 2, :n].mean(0), atol=1e-13)
        assert abs(lse[b, h, t] - math.log(n)) < 1e-13


def test_one_dominant_key_returns_its_value_row():
    S, d = 33, 16
    rng = np.random.default_rng(6)
    k = rng.standard_normal((1, 1, S, d)) * 0.01
    v = rng.standard_normal((1, 1, S, d))
    j = 17
    k[0, 0, j] = 0.0
    k[0, 0, j, 3] = 1.0
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 3] = 40.0  # score_j = 40, every other |score| <= 40 * 0.05
    O, lse = orc.attention(q, k, v, scale=1.0)
    np.testing.assert_allclose(O[0, 0, 0], v[0, 0, j], atol=1e-12)
    assert abs(lse[0, 0, 0] - 40.0) < 1e-12


def test_gqa_equals_mha_with_kv_repeated():
    B, H_kv, G, S, T, d = 2, 3, 4, 10, 2, 8
    H_q = H_kv * G
    q = _rand((B, H_q, T, d), 7)
    k, v = _rand((B, H_kv, S, d), 8), _rand((B, H_kv, S, d), 9)
    k_rep = torch.from_numpy(k).repeat_interleave(G, dim=1).numpy()
    v_rep = torch.from_numpy(v).repeat_interleave(G, dim=1).numpy()
    for causal in (False, True):
        O, lse = orc.attention(q, k, v, scale=0.25, causal=causal, q_offset=3 if causal else 0)
        O2, lse2 = orc.attention(q, k_rep, v_rep, scale=0.25, causal=causal,
                                 q_offset=3 if causal else 0)
        np.testing.assert_allclose(O, O2, atol=1e-14)
        np.testing.assert_allclose(lse, lse2, atol=1e-14)


def test_matches_torch_sdpa_fp64_and_scipy_logsumexp():
    scipy_special = pytest.importorskip("scipy.special")
    B, H_kv, G, T, S, d = 2, 2, 4, 6, 14, 16
    H_q = H_kv * G
    q, k, v = _rand((B, H_q, T, d), 10), _rand((B, H_kv, S, d), 11), _rand((B, H_kv, S, d), 12)
    scale = 1 / math.sqrt(d)
    for q_offset in (0, 8):
        O, lse = orc.attention(q, k, v, scale=scale, causal=True, q_offset=q_offset)
        qt, kt, vt = (torch.from_numpy(x) for x in (q, k, v))
        kt, vt = kt.repeat_interleave(G, 1), vt.repeat_interleave(G, 1)
        mask = torch.arange(S)[None, :] <= (q_offset + torch.arange(T))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                               scale=scale)
        np.testing.assert_allclose(O, ref.numpy(), atol=1e-12)
        scores = (qt @ kt.transpose(-1, -2)).numpy() * scale
        scores = np.where(mask.numpy(), scores, -np.inf)
        np.testing.assert_allclose(lse, scipy_special.logsumexp(scores, axis=-1), atol=1e-12)


def test_causal_row_equals_unmasked_attention_over_prefix():
    B, H_q, H_kv, T, S, d, off = 1, 4, 1, 5, 12, 8, 7
    q, k, v = _rand((B, H_q, T, d), 13), _rand((B, H_kv, S, d), 14), _rand((B, H_kv, S, d), 15)
    O, lse = orc.attention(q, k, v, scale=0.4, causal=True, q_offset=off)
    for t in range(T):
        n = off + t + 1
        Ot, lt = orc.attention(q[:, :, t:t + 1], k[:, :, :n], v[:, :, :n], scale=0.4)
        np.testing.assert_allclose(O[:, :, t], Ot[:, :, 0], atol=1e-14)
        np.testing.assert_allclose(lse[:, :, t], lt[:, :, 0], atol=1e-14)


def _brute(q, k, v, scale, vis):
    """Hand-expanded softmax attention with Python loops and math.exp."""
    B, H_q, T, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    H_kv = len(k[0])
    G = H_q // H_kv
    O = [[[[0.0] * d for _ in range(T)] for _ in range(H_q)] for _ in range(B)]
    L = [[[0.0] * T for _ in range(H_q)] for _ in range(B)]
    for b in range(B):
        for h in range(H_q):
            for t in range(T):
                js = [j for j in range(len(k[b][h // G])) if vis(b, t, j)]
                s = {j: scale * sum(q[b][h][t][c] * k[b][h // G][j][c] for c in range(d))
                     for j in js}
                z = sum(math.exp(s[j]) for j in js)
                for c in range(d):
                    O[b][h][t][c] = sum(math.exp(s[j]) * v[b][h // G][j][c] for j in js) / z
                L[b][h][t] = math.log(z)
    return np.array(O), np.array(L)


def test_brute_force_tiny_shapes():
    B, H_q, H_kv, T, S, d = 2, 2, 1, 2, 4, 3
    q, k, v = _rand((B, H_q, T, d), 16), _rand((B, H_kv, S, d), 17), _rand((B, H_kv, S, d), 18)
    Ob, Lb = _brute(q.tolist(), k.tolist(), v.tolist(), 0.7, lambda b, t, j: j <= 1 + t)
    O, lse = orc.attention(q, k, v, scale=0.7, causal=True, q_offset=1)
    np.testing.assert_allclose(O, Ob, atol=1e-13)
    np.testing.assert_allclose(lse, Lb, atol=1e-13)
    qd = q[:, :, :1]
    Ob, Lb = _brute(qd.tolist(), k.tolist(), v.tolist(), 0.7, lambda b, t, j: j < [3, 1][b])
    O, lse = orc.attention(qd, k, v, scale=0.7, seqlens=[3, 1])
    np.testing.assert_allclose(O, Ob, atol=1e-13)
    np.testing.assert_allclose(lse, Lb, atol=1e-13)


def test_zero_length_decode_row():
    q, k, v = _rand((2, 2, 1, 4), 19), _rand((2, 1, 5, 4), 20), _rand((2, 1, 5, 4), 21)
    O, lse = orc.attention(q, k, v, scale=1.0, seqlens=[0, 5])
    assert (O[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.isfinite(lse[1]).all()
    Or, lr = orc.attention_rows(q, k, v, [(0, 1, 0), (1, 0, 0)], scale=1.0, seqlens=[0, 5])
    assert (Or[0] == 0).all() and np.isneginf(lr[0])
    np.testing.assert_allclose(Or[1], O[1, 0, 0], atol=1e-14)


def test_attention_rows_matches_full():
    B, H_q, H_kv, T, S, d = 2, 8, 2, 3, 20, 8
    q, k, v = _rand((B, H_q, T, d), 22), _rand((B, H_kv, S, d), 23), _rand((B, H_kv, S, d), 24)
    O, lse = orc.attention(q, k, v, scale=0.5, causal=True, q_offset=9)
    rows = list(itertools.product(range(B), range(H_q), range(T)))
    Or, lr = orc.attention_rows(q, k, v, rows, scale=0.5, causal=True, q_offset=9)
    np.testing.assert_allclose(Or, O.reshape(-1, d), atol=1e-14)
    np.testing.assert_allclose(lr, lse.reshape(-1), atol=1e-14)


# --------------------------------------------------------------------------
# the tiled recurrence (§3) and the merge (§4)
# --------------------------------------------------------------------------


@pytest.mark.parametrize("tile", [1, 3, 8, 16, 40])
def test_online_sweep_equals_definition(tile):
    M, n, d = 6, 37, 8
    q, K, V = _rand((M, d), 25), _rand((n, d), 26, 2.0), _rand((n, d), 27)
    m, l, O = orc.online_softmax_sweep(q, K, V, scale=0.5, tile=tile, n_valid=n)
    Of, lse = orc.finalize(m, l, O)
    Oref, lref = orc.attention(q[None, :, None, :], K[None, None], V[None, None], scale=0.5)
    np.testing.assert_allclose(Of, Oref[0, :, 0], atol=1e-13)
    np.testing.assert_allclose(lse, lref[0, :, 0], atol=1e-13)
    # causal boundary mask inside the sweep (rows at positions 20..25)
    pos = np.arange(20, 26)
    m, l, O = orc.online_softmax_sweep(q, K, V, scale=0.5, tile=tile, n_valid=n, query_pos=pos)
    Of, lse = orc.finalize(m, l, O)
    for i in range(M):
        Oi, li = orc.attention(q[None, i:i + 1, None, :], K[None, None, :pos[i] + 1],
                               V[None, None, :pos[i] + 1], scale=0.5)
        np.testing.assert_allclose(Of[i], Oi[0, 0, 0], atol=1e-13)
        assert abs(lse[i] - li[0, 0, 0]) < 1e-13


def test_split_and_merge_equals_single_pass_for_every_split_count():
    B, H_q, H_kv, S, d = 2, 4, 2, 23, 8
    q = _rand((B, H_q, d), 28)
    k, v = _rand((B, H_kv, S, d), 29), _rand((B, H_kv, S, d), 30)
    seqlens = [23, 9]
    O, lse = orc.attention(q[:, :, None], k, v, scale=0.35, seqlens=seqlens)
    for ns in range(1, S + 1):
        ms, ls, Os = orc.split_partials(q, k, v, scale=0.35, seqlens=seqlens, num_splits=ns)
        Oc, lc = orc.combine_partials(ms, ls, Os)
        np.testing.assert_allclose(Oc, O[:, :, 0], atol=1e-13, err_msg=f"ns={ns}")
        np.testing.assert_allclose(lc, lse[:, :, 0], atol=1e-13, err_msg=f"ns={ns}")


def test_merge_is_associative_and_commutative():
    rng = np.random.default_rng(31)
    parts = [(rng.standard_normal(3) * 4, rng.random(3) + 0.1, rng.standard_normal((3, 5)))
             for _ in range(3)]
    a, b, c = parts
    ab_c = orc.lse_merge(*orc.lse_merge(*a, *b), *c)
    a_bc = orc.lse_merge(*a, *orc.lse_merge(*b, *c))
    ba = orc.lse_merge(*b, *a)
    ab = orc.lse_merge(*a, *b)
    for x, y in zip(ab_c, a_bc):
        np.testing.assert_allclose(x, y, rtol=1e-13)
    for x, y in zip(ab, ba):
        np.testing.assert_allclose(x, y, rtol=1e-13)
    # an empty partial (-inf, 0, 0) is the identity
    e = (np.full(3, -np.inf), np.zeros(3), np.zeros((3, 5)))
    for x, y in zip(orc.lse_merge(*a, *e), a):
        np.testing.assert_allclose(x, y, rtol=0, atol=0)


# --------------------------------------------------------------------------
# integer plans
# --------------------------------------------------------------------------


def test_split_bounds_partition_every_row():
    for S_max in (1, 2, 7, 64, 255, 256, 1000):
        for ns in list(range(1, 12)) + [S_max, S_max + 3]:
            L = orc.split_len(S_max, ns)
            assert L * ns >= S_max and (L - 1) * ns < S_max  # L = ceil(S_max / ns)
            for seqlen in sorted({0, 1, S_max // 2, S_max - 1, S_max}):
                if seqlen < 0:
                    continue
                bounds = orc.split_bounds(S_max, ns, seqlen)
                covered = []
                for s, (a, b) in enumerate(bounds):
                    assert 0 <= a <= b <= seqlen and b - a <= L
                    assert a == min(s * L, seqlen)
                    covered.extend(range(a, b))
                assert covered == list(range(seqlen))


def test_tile_class_matches_elementwise_visibility():
    # brute force: a tile is past iff every (query, key) pair is visible, future iff none is.
    for qs, qe, ks, ke in itertools.product(range(0, 9), range(1, 10), range(0, 9), range(1, 10)):
        if qe <= qs or ke <= ks:
            continue
        vis = [[j <= i for j in range(ks, ke)] for i in range(qs, qe)]
        all_vis = all(all(r) for r in vis)
        none_vis = not any(any(r) for r in vis)
        c = orc.tile_class(qs, qe, ks, ke)
        if c == orc.TILE_ALL_PAST:
            assert all_vis
        elif c == orc.TILE_ALL_FUTURE:
            assert none_vis
        else:
            assert not none_vis  # a partial tile always holds a visible pair
        assert (c == orc.TILE_ALL_FUTURE) == none_vis


@pytest.mark.parametrize("T_q,S_kv,off,bm,bn", [(8192, 8192, 0, 128, 128),
                                                (2048, 32768, 30720, 128, 128),
                                                (300, 300, 0, 128, 64), (17, 50, 33, 16, 16)])
def test_prefill_tile_counts_equal_lower_triangle(T_q, S_kv, off, bm, bn):
    cls = orc.prefill_tile_classes(T_q, S_kv, off, bm, bn)
    computed = int((cls != orc.TILE_ALL_FUTURE).sum())
    # lower-triangle tile count by direct reasoning: m-tile i needs n-tiles up to the one
    # holding its last row's last visible key, q_off + min((i+1)*bm, T_q) - 1.
    nm = -(-T_q // bm)
    expect = sum((off + min((i + 1) * bm, T_q) - 1) // bn + 1 for i in range(nm))
    assert computed == expect
    assert ((cls == orc.TILE_PARTIAL).sum(axis=1) >= 1).all()
