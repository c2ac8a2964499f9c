"""C ABI: the library loads, exports every declared symbol, its integer plan
matches independent derivations bit for bit, and bad arguments come back as
error codes before anything reaches a GPU. No GPU needed."""

import ctypes
import itertools
import os
import re

import pytest

import oracle as orc
from gqa_attention_split_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_attn.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return api.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_attn_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported_and_bound(L):
    declared = _declared_functions()
    assert "gqa_attn_decode" in declared and "gqa_attn_prefill" in declared
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(api.symbols()) == declared


def test_version_and_strerror(L):
    assert api.gqa_attn_version() >= 100
    for code in range(0, -8, -1):
        assert api.strerror(code) and api.strerror(code) != "unknown error code"
    assert api.strerror(-99) == "unknown error code"


def test_split_bounds_bit_exact_vs_oracle(L):
    for S_max in (1, 2, 7, 64, 255, 256, 1000, 8192):
        for ns in (1, 2, 3, 4, 7, 19, S_max):
            for seqlen in sorted({0, 1, S_max // 3, S_max - 1, S_max}):
                if seqlen < 0:
                    continue
                rc, got = api.gqa_attn_split_bounds(S_max, ns, seqlen)
                assert rc == 0
                assert got == orc.split_bounds(S_max, ns, seqlen), (S_max, ns, seqlen)


def test_split_bounds_rejects_bad_args(L):
    assert api.gqa_attn_split_bounds(10, 0, 5)[0] == api.GQA_ERR_INVALID_ARG
    assert api.gqa_attn_split_bounds(10, 2, 11)[0] == api.GQA_ERR_INVALID_ARG
    assert api.gqa_attn_split_bounds(10, 2, -1)[0] == api.GQA_ERR_INVALID_ARG


def test_tile_class_bit_exact_vs_oracle(L):
    for qs, qe, ks, ke in itertools.product(range(0, 7), range(1, 8), range(0, 7), range(1, 8)):
        if qe > qs and ke > ks:
            assert api.gqa_attn_tile_class(qs, qe, ks, ke) == orc.tile_class(qs, qe, ks, ke)


@pytest.mark.parametrize("T_q,S_kv,off,causal", [(8192, 8192, 0, 1), (2048, 32768, 30720, 1),
                                                 (300, 300, 0, 1), (17, 50, 33, 1),
                                                 (1000, 1000, 0, 0), (0, 10, 0, 1)])
def test_prefill_tile_counts_bit_exact_vs_oracle(L, T_q, S_kv, off, causal):
    bm, bn = api.gqa_attn_prefill_block_m(), api.gqa_attn_prefill_block_n()
    rc, past, part, fut = api.gqa_attn_prefill_tile_counts(T_q, S_kv, off, causal)
    assert rc == 0
    if T_q == 0:
        assert past == part == fut == 0
        return
    cls = orc.prefill_tile_classes(T_q, S_kv, off, bm, bn)
    if not causal:
        assert (past, part, fut) == (cls.size, 0, 0)
    else:
        assert past == int((cls == orc.TILE_ALL_PAST).sum())
        assert part == int((cls == orc.TILE_PARTIAL).sum())
        assert fut == int((cls == orc.TILE_ALL_FUTURE).sum())


def _pick_reference(B, H_kv, S, sms, one_row=16384):
    # The rule stated in include/gqa_attn.h, restated independently
    # (one_row: the one-wave split bound for B = 1; 2048 for the INT8 rule).
    cdiv = lambda a, b: -(-a // b)
    fits = [n for n in (16, 8, 4, 2) if B * H_kv * n <= sms]
    if fits:   # one wave of whole-row clusters, if it is busy enough
        n = fits[0]
        keys = cdiv(S, n)
        busy = B * H_kv * n >= 0.8 * sms and keys <= (one_row if B == 1 else 2048)
        if keys >= 256 and (busy or keys <= 512):
            return n
    n = cdiv(sms, B * H_kv)
    if n > 16 and B * H_kv * 16 * (n // 16) >= 0.8 * sms:
        n = 16 * (n // 16)
    n = max(n, cdiv(S, 1024))
    if n > 16:
        n = 16 * cdiv(n, 16)
    return max(1, min(n, max(1, S // 256), 8192))


def test_pick_num_splits_bit_exact_and_properties(L):
    assert api.gqa_attn_pick_num_splits(1, 8, 8192, 152) == 16       # 8K decode: 8 clusters
    assert api.gqa_attn_pick_num_splits(4, 8, 131072, 152) == 128    # 128K ragged decode
    assert api.gqa_attn_pick_num_splits(1, 1, 256, 152) == 1         # tiny decode
    assert api.gqa_attn_pick_num_splits(2, 8, 8192, 152) == 8        # one wave, 8 clusters of 8
    assert api.gqa_attn_pick_num_splits(1, 8, 32768, 152) == 16      # one wave, 2048-key splits
    assert api.gqa_attn_pick_num_splits(1, 8, 131072, 152) == 16     # one row: up to 16384 keys
    assert api.gqa_attn_pick_num_splits(1, 8, 524288, 152) == 512    # 32768-key splits: no
    assert api.gqa_attn_pick_num_splits(2, 8, 65536, 152) == 64      # a batch: 2048 at most
    assert api.gqa_attn_pick_num_splits(1, 4, 8192, 152) == 16       # short splits, 64 CTAs
    assert api.gqa_attn_pick_num_splits(1, 4, 32768, 152) == 32      # 2048-key splits: no
    for B, H_kv, S, sms in itertools.product((1, 2, 3, 4, 8, 64), (1, 2, 4, 6, 8),
                                             (1, 255, 256, 1000, 2048, 4096, 8192, 16384,
                                              32768, 65536, 100000, 131072, 262144, 300000),
                                             (1, 148, 152)):
        ns = api.gqa_attn_pick_num_splits(B, H_kv, S, sms)
        assert ns == _pick_reference(B, H_kv, S, sms), (B, H_kv, S, sms)
        assert 1 <= ns <= max(1, S // 256)
        # the blocks cover at least 80% of the SMs whenever the length allows,
        # unless short splits (<= 512 keys) fit in one wave of whole-row clusters
        short_wave = ns in (16, 8, 4, 2) and B * H_kv * ns <= sms and -(-S // ns) <= 512
        if S // 256 >= -(-sms // (B * H_kv)) and not short_wave:
            assert B * H_kv * ns >= 0.8 * sms
    assert api.gqa_attn_pick_num_splits(0, 8, 8192, 152) == api.GQA_ERR_INVALID_ARG


def test_pick_num_splits_q8_plans_half_the_keys(L):
    # an INT8 token is about half the bytes of a bf16 one
    assert api.gqa_attn_pick_num_splits_q8(1, 8, 8192, 152) == 16     # 8K decode: unchanged
    assert api.gqa_attn_pick_num_splits_q8(4, 8, 131072, 152) == 64   # 128K ragged: half
    assert api.gqa_attn_pick_num_splits_q8(1, 8, 131072, 152) == 64   # one row: bound 2048
    for B, H_kv, S, sms in itertools.product((1, 4, 64), (1, 8),
                                             (1, 2, 255, 513, 8192, 65536, 131072), (1, 152)):
        assert api.gqa_attn_pick_num_splits_q8(B, H_kv, S, sms) == \
            _pick_reference(B, H_kv, -(-S // 2), sms, one_row=2048), (B, H_kv, S, sms)
    assert api.gqa_attn_pick_num_splits_q8(1, 8, 0, 152) == api.GQA_ERR_INVALID_ARG


def test_decode_cluster_size(L):
    # largest of 16, 8, 4, 2 dividing the split count; at most 8 once the grid
    # (splits x KV heads x batch) has more CTAs than SMs
    cases = [((1, 8, 16, 152), 16),    # 8K decode: 128 CTAs, one wave
             ((1, 8, 19, 152), 1),     # prime split count: no clusters
             ((1, 8, 6, 152), 2),
             ((1, 8, 12, 152), 4),
             ((1, 8, 24, 152), 8),     # 192 CTAs: more than one wave
             ((4, 8, 128, 152), 8),    # ragged 128K batch
             ((3, 2, 32, 152), 8),
             ((1, 2, 64, 152), 16),    # exactly 128 CTAs
             ((1, 19, 8, 152), 8),     # exactly 152 CTAs
             ((1, 1, 1, 152), 1)]
    for args, cs in cases:
        assert api.gqa_attn_decode_cluster_size(*args) == cs, args
    for bad in ((0, 8, 16, 152), (1, 0, 16, 152), (1, 8, 0, 152), (1, 8, 16, 0)):
        assert api.gqa_attn_decode_cluster_size(*bad) == api.GQA_ERR_INVALID_ARG


def test_workspace_size(L):
    assert api.gqa_attn_decode_workspace_size(1, 64, 128, 1) == 0
    n = api.gqa_attn_decode_workspace_size(1, 64, 128, 19)
    assert n >= 64 * 19 * (128 + 2) * 4 and n % 256 == 0
    assert api.gqa_attn_decode_workspace_size(1, 64, 96, 19) == 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case fails host checks first


@pytest.mark.parametrize("args,code", [
    # q,k,v,o null
    ((0, FAKE, FAKE, FAKE, 0, 0, 1, 8, 1, 64, 256, 0.125, 0), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, 0, 0, 0, 1, 8, 1, 64, 256, 0.125, 0), api.GQA_ERR_INVALID_ARG),
    # H_q % H_kv != 0
    ((FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 6, 4, 64, 256, 0.125, 0), api.GQA_ERR_INVALID_ARG),
    # bad sizes
    ((FAKE, FAKE, FAKE, FAKE, 0, 0, -1, 8, 1, 64, 256, 0.125, 0), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 8, 1, 64, 0, 0.125, 0), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 8, 1, 64, 256, 0.125, -2), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 8, 1, 64, 256, float("nan"), 0), api.GQA_ERR_INVALID_ARG),
    # unsupported head dim / group size
    ((FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 8, 1, 96, 256, 0.125, 0), api.GQA_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 17, 1, 64, 256, 0.125, 0), api.GQA_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 32, 1, 64, 256, 0.125, 0), api.GQA_ERR_UNSUPPORTED),
    # misaligned pointer
    ((FAKE + 2, FAKE, FAKE, FAKE, 0, 0, 1, 8, 1, 64, 256, 0.125, 0), api.GQA_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE + 8, FAKE, 0, 0, 1, 8, 1, 64, 256, 0.125, 0), api.GQA_ERR_MISALIGNED),
])
def test_decode_bad_args_return_codes_without_launch(L, args, code):
    assert api.gqa_attn_decode(*args, None) == code


def test_decode_ws_rejects_auto_split_count(L):
    rc = api.gqa_attn_decode_ws(FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 8, 1, 64, 256, 0.125, 0,
                                FAKE, 1 << 20, None)
    assert rc == api.GQA_ERR_INVALID_ARG


def test_decode_empty_batch_is_a_no_op(L):
    assert api.gqa_attn_decode(FAKE, FAKE, FAKE, FAKE, 0, 0, 0, 8, 1, 64, 256, 0.125, 0,
                               None) == 0


@pytest.mark.parametrize("args,code", [
    ((0, FAKE, FAKE, FAKE, 0, 1, 64, 8, 128, 128, 128, 0, 1, 0.1), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 7, 128, 128, 128, 0, 1, 0.1), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 8, 128, 128, 128, -1, 1, 0.1), api.GQA_ERR_INVALID_ARG),
    # the scale must be finite and > 0 (the kernels scale each row's raw maximum)
    ((FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 8, 128, 128, 128, 0, 1, 0.0), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 8, 128, 128, 128, 0, 1, -0.1), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 8, 128, 128, 128, 0, 0, -0.1), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 8, 128, 128, 128, 0, 1, float("inf")),
     api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 8, 128, 128, 128, 0, 1, float("nan")),
     api.GQA_ERR_INVALID_ARG),
    # prefill runs d = 64 and 128
    ((FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 8, 96, 128, 128, 0, 1, 0.1), api.GQA_ERR_UNSUPPORTED),
])
def test_prefill_bad_args_return_codes_without_launch(L, args, code):
    assert api.gqa_attn_prefill_ex(*args, None) == code


@pytest.mark.parametrize("args,code", [
    # k_cache, v_cache, k_new, v_new, positions, B, H_kv, d, capacity, n_sink
    ((0, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 8, 2), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, 1, 1, 64, 8, 2), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 8, 8), api.GQA_ERR_INVALID_ARG),   # no window
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 8, -1), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 0, 0), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 96, 8, 2), api.GQA_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE + 8, FAKE, FAKE, 1, 1, 64, 8, 2), api.GQA_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 64, 8, 2), 0),                         # empty batch
])
def test_ring_append_bad_args_return_codes_without_launch(L, args, code):
    assert api.gqa_attn_ring_append(*args, None) == code


@pytest.mark.parametrize("args,code", [
    # q, k, v, o, lse, seqlens, B, H_q, H_kv, d, capacity, n_sink, scale, num_splits
    ((FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 8, 1, 64, 256, 2, 0.125, 0), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 8, 1, 64, 256, 256, 0.125, 0), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 8, 1, 64, 256, -1, 0.125, 0), api.GQA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 8, 1, 96, 256, 2, 0.125, 0), api.GQA_ERR_UNSUPPORTED),
    ((FAKE + 2, FAKE, FAKE, FAKE, 0, FAKE, 1, 8, 1, 64, 256, 2, 0.125, 0),
     api.GQA_ERR_MISALIGNED),
    ((FAKE, FAKE, FAKE, FAKE, 0, FAKE, 0, 8, 1, 64, 256, 2, 0.125, 0), 0),        # empty batch
])
def test_decode_ring_bad_args_return_codes_without_launch(L, args, code):
    assert api.gqa_attn_decode_ring(*args, None) == code


def test_debug_tile_counts_need_the_debug_build(L):
    # the product library has no tile counters: the call reports that and
    # touches nothing (no device work either)
    rc, counts = api.gqa_attn_debug_tile_counts(clear=True)
    assert rc == api.GQA_ERR_UNSUPPORTED and counts == [0, 0, 0]


def test_merge_and_partial_bad_args_return_codes_without_launch(L):
    st = None
    # o_parts, lse_parts, o, lse, R, rows, d
    assert api.gqa_attn_merge(FAKE, FAKE, FAKE, FAKE, 0, 8, 64, st) == api.GQA_ERR_INVALID_ARG
    assert api.gqa_attn_merge(0, FAKE, FAKE, FAKE, 2, 8, 64, st) == api.GQA_ERR_INVALID_ARG
    assert api.gqa_attn_merge(FAKE, FAKE, FAKE, FAKE, 2, -1, 64, st) == api.GQA_ERR_INVALID_ARG
    assert api.gqa_attn_merge(FAKE, FAKE, FAKE, FAKE, 2, 8, 96, st) == api.GQA_ERR_UNSUPPORTED
    assert api.gqa_attn_merge(FAKE + 4, FAKE, FAKE, FAKE, 2, 8, 64, st) == api.GQA_ERR_MISALIGNED
    assert api.gqa_attn_merge(FAKE, FAKE, FAKE, FAKE, 2, 0, 64, st) == 0  # nothing to merge
    # q, k, v, o_part, lse_part, seqlens, B, H_q, H_kv, d, S_max, scale, num_splits
    assert api.gqa_attn_decode_partial(FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 8, 1, 64, 256, 0.125, 0,
                                       st) == api.GQA_ERR_INVALID_ARG      # lse is required
    assert api.gqa_attn_decode_partial(FAKE, FAKE, FAKE, FAKE + 8, FAKE, 0, 1, 8, 1, 64, 256,
                                       0.125, 0, st) == api.GQA_ERR_MISALIGNED
    assert api.gqa_attn_decode_partial(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 8, 1, 64, 256, 0.125,
                                       0, st) == 0                         # empty batch


def test_pick_num_splits_q4_takes_the_int8_rule(L):
    # both quantised decodes are issue-bound: INT4 plans like INT8 (half the row)
    assert api.gqa_attn_pick_num_splits_q4(1, 8, 8192, 152) == 16     # 8K decode
    assert api.gqa_attn_pick_num_splits_q4(4, 8, 131072, 152) == 64   # 128K ragged
    for B, H_kv, S, sms in itertools.product((1, 4, 64), (1, 8),
                                             (1, 2, 255, 513, 8192, 65536, 131072), (1, 152)):
        assert api.gqa_attn_pick_num_splits_q4(B, H_kv, S, sms) == \
            _pick_reference(B, H_kv, -(-S // 2), sms, one_row=2048), (B, H_kv, S, sms)
    assert api.gqa_attn_pick_num_splits_q4(1, 8, 0, 152) == api.GQA_ERR_INVALID_ARG


def test_q4_bad_args_return_codes_without_launch(L):
    st = None
    # k, v, k_codes, v_codes, k_scales, v_scales, B, H_kv, S, d
    assert api.gqa_attn_quantize_kv_q4(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1, 1, 64, 128,
                                       st) == api.GQA_ERR_INVALID_ARG
    assert api.gqa_attn_quantize_kv_q4(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 48, 128,
                                       st) == api.GQA_ERR_UNSUPPORTED    # S % 32 != 0
    assert api.gqa_attn_quantize_kv_q4(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64,
                                       st) == api.GQA_ERR_UNSUPPORTED    # d != 128
    assert api.gqa_attn_quantize_kv_q4(FAKE, FAKE, FAKE + 4, FAKE, FAKE, FAKE, 1, 1, 64, 128,
                                       st) == api.GQA_ERR_MISALIGNED
    # q, k_codes, v_codes, k_scales, v_scales, o, lse, seqlens, B, H_q, H_kv, d, S_max, scale, ns
    assert api.gqa_attn_decode_q4(FAKE, FAKE, FAKE, 0, FAKE, FAKE, 0, 0, 1, 8, 1, 128, 64, 0.1,
                                  0, st) == api.GQA_ERR_INVALID_ARG
    assert api.gqa_attn_decode_q4(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 1, 8, 1, 128, 48,
                                  0.1, 0, st) == api.GQA_ERR_UNSUPPORTED
    assert api.gqa_attn_decode_q4(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 0, 0, 8, 1, 128, 64,
                                  0.1, 0, st) == 0                       # empty batch


def test_only_the_c_abi_is_exported(L):
    # The library is built with hidden visibility: its C++ internals (launch
    # helpers, their per-device "attributes set" statics, template kernels)
    # are private to each build, so the product library and the -DGQA_DEBUG
    # build can live in one process. Process-unique symbols would be merged
    # across the two by the dynamic linker.
    import shutil
    import subprocess

    if shutil.which("nm") is None:
        pytest.skip("nm not available")
    out = subprocess.run(["nm", "-D", "--defined-only", api.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    syms = [ln.split() for ln in out.splitlines() if len(ln.split()) == 3]
    assert not [s for s in syms if s[1] == "u"], "process-unique symbols exported"
    ours = sorted(s[2] for s in syms if s[2].startswith("gqa_attn_"))
    assert ours == sorted(api.symbols())
    assert not [s for s in syms if "gqa" in s[2] and not s[2].startswith("gqa_attn_")]


def test_prefill_partial_bad_args_return_codes_without_launch(L):
    st = None
    # q, k, v, o_part, lse_part, B, H_q, H_kv, d, T_q, S_kv, q_offset, key_offset, causal, scale
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 128, 64, 64, 0, 0, 1, 0.1)
    bad = [((FAKE, FAKE, FAKE, FAKE, 0) + ok[5:], api.GQA_ERR_INVALID_ARG),        # lse required
           (ok[:12] + (-1,) + ok[13:], api.GQA_ERR_INVALID_ARG),                  # key_offset
           (ok[:11] + (-1,) + ok[12:], api.GQA_ERR_INVALID_ARG),                  # q_offset
           (ok[:14] + (0.0,), api.GQA_ERR_INVALID_ARG),                           # scale
           (ok[:8] + (96,) + ok[9:], api.GQA_ERR_UNSUPPORTED),                    # head dim
           ((FAKE, FAKE, FAKE, FAKE + 8) + ok[4:], api.GQA_ERR_MISALIGNED),
           (ok[:5] + (0,) + ok[6:], 0)]                                            # empty batch
    for args, code in bad:
        assert api.gqa_attn_prefill_partial(*args, st) == code, args
    # queries past the slice's last key are allowed (the rest of the keys are
    # in later slices); the whole-cache prefill rejects them
    assert api.gqa_attn_prefill_ex(FAKE, FAKE, FAKE, FAKE, 0, 1, 8, 2, 128, 64, 64, 10, 1, 0.1,
                                   st) == api.GQA_ERR_INVALID_ARG
