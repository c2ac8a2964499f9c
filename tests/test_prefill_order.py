"""Host plan of the prefill work order (gqa_attn_prefill_schedule), on the CPU.

Page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)", §5.4 (prefill
scheduling of query blocks against KV tiles, heaviest first). The persistent
kernel numbers its work items heaviest query block first; the host may hand
it an order instead, grouped by (batch, KV head) so that concurrently running
CTAs share their keys in L2. The checks restate the item numbering and the
tile counts independently and test the plan's properties: every item exactly
once, super-groups whose K/V fits the budget and that no CTA revisits,
heaviest first within a super-group, and the list-scheduling bound on the
most loaded CTA.
"""

import math

import pytest

from gqa_attention_split_gb300 import api

BM = BN = 128
BUDGET = 48 << 20


@pytest.fixture(autouse=True)
def _default_budget():
    api.gqa_attn_debug_prefill_order(-1)
    yield
    api.gqa_attn_debug_prefill_order(-1)


def visible_tiles(row0, T_q, S_kv, q_offset, causal):
    """KV tiles a query block starting at row0 reads (0 past the last query)."""
    if row0 >= T_q:
        return 0
    if not causal:
        return math.ceil(S_kv / BN)
    last_key = q_offset + min(row0 + BM, T_q)   # one past the block's last visible key
    return math.ceil(min(S_kv, last_key) / BN)


def items_of(B, H_q, H_kv, T_q, S_kv, q_offset, causal):
    """[(group, tiles)] in the kernel's item numbering: even G, one query block
    of a head pair per item, blocks from the last down, (batch, pair) fastest;
    odd G, two consecutive blocks of one head, block pairs from the last down,
    (batch, head) fastest."""
    G = H_q // H_kv
    nmb = math.ceil(T_q / BM)
    out = []
    if G % 2 == 0:
        for m in reversed(range(nmb)):
            for b in range(B):
                for pair in range(H_q // 2):
                    kvh = (2 * pair) // G
                    out.append((b * H_kv + kvh, visible_tiles(m * BM, T_q, S_kv, q_offset,
                                                              causal)))
    else:
        for bp in reversed(range((nmb + 1) // 2)):
            for b in range(B):
                for h in range(H_q):
                    n = max(visible_tiles(2 * bp * BM, T_q, S_kv, q_offset, causal),
                            visible_tiles((2 * bp + 1) * BM, T_q, S_kv, q_offset, causal))
                    out.append((b * H_kv + h // G, n))
    return out


def super_groups(B, H_kv, S_kv, d, budget=BUDGET):
    """Super-group of each (batch, KV head) group: n_sg nearly equal runs of
    consecutive groups, each holding at most budget bytes of K/V (one group if a
    single group is larger)."""
    groups = B * H_kv
    per = S_kv * d * 4
    n_sg = math.ceil(groups / max(1, budget // per))
    of = [g * n_sg // groups for g in range(groups)]
    sizes = [of.count(i) for i in range(n_sg)]
    assert max(sizes) - min(sizes) <= 1
    assert max(sizes) == 1 or max(sizes) * per <= budget
    return of


def check_plan(shape, ctas, budget=BUDGET):
    B, H_q, H_kv, d, T_q, S_kv, off, causal = shape
    rc, lists = api.gqa_attn_prefill_schedule(B, H_q, H_kv, d, T_q, S_kv, off, int(causal),
                                              ctas)
    items = items_of(B, H_q, H_kv, T_q, S_kv, off, causal)
    assert rc == len(items)
    flat = sorted(i for lst in lists for i in lst)
    assert flat == list(range(len(items)))                 # every item exactly once
    sg = super_groups(B, H_kv, S_kv, d, budget)
    costs = [n + 1 for _, n in items]
    loads = []
    for lst in lists:
        s = [sg[items[i][0]] for i in lst]
        assert s == sorted(s)                               # no super-group revisited
        for a, b in zip(lst, lst[1:]):
            if sg[items[a][0]] == sg[items[b][0]]:
                assert items[a][1] >= items[b][1]           # heaviest first within one
        loads.append(sum(costs[i] for i in lst))
    # greedy list scheduling: the most loaded CTA is within one item of the mean
    assert max(loads) <= sum(costs) / ctas + max(costs)
    return lists, items


def test_l2_resident_problems_keep_the_closed_form_order():
    # 8K causal, 64/8 heads: K/V of all groups is 33.5 MB
    rc, lists = api.gqa_attn_prefill_schedule(1, 64, 8, 128, 8192, 8192, 0, 1, 152)
    assert rc == 0 and lists == []


def test_chunked_32k_prefill_plan():
    # 2 x 8 groups of 16.8 MB: six super-groups of 2 or 3 groups
    lists, items = check_plan((2, 64, 8, 128, 2048, 32768, 30720, True), 152)
    assert sorted(set(super_groups(2, 8, 32768, 128))) == list(range(6))
    assert len(items) == 1024


@pytest.mark.parametrize("shape", [
    (1, 64, 64, 128, 8192, 8192, 0, True),      # G = 1: block pairs, 64 groups of 4.2 MB
    (1, 64, 8, 128, 32768, 32768, 0, True),     # 32K causal: 8192 items
    (4, 64, 8, 128, 8192, 8192, 0, True),       # four batch rows
    (2, 48, 16, 64, 3000, 20000, 17000, True),  # G = 3, d = 64, chunk at an offset
    (1, 16, 2, 128, 1000, 70000, 0, False),     # full attention over long keys
])
def test_plans_of_larger_than_l2_problems(shape):
    check_plan(shape, 152)


def test_small_budget_orders_tiny_problems_one_group_at_a_time():
    api.gqa_attn_debug_prefill_order(1)
    lists, items = check_plan((2, 8, 2, 128, 300, 300, 0, True), 6, budget=1)
    groups_seen = [[items[i][0] for i in lst] for lst in lists]
    for g in groups_seen:
        assert g == sorted(g)
    api.gqa_attn_debug_prefill_order(0)         # closed form for everything
    assert api.gqa_attn_prefill_schedule(2, 64, 8, 128, 2048, 32768, 30720, 1, 152)[0] == 0


def test_limits_and_errors():
    # more items than the table holds: closed form
    assert api.gqa_attn_prefill_schedule(8, 64, 8, 128, 32768, 32768, 0, 1, 152)[0] == 0
    # more CTAs than the table holds: closed form
    assert api.gqa_attn_prefill_schedule(2, 64, 8, 128, 2048, 32768, 30720, 1, 200)[0] == 0
    assert api.gqa_attn_prefill_schedule(1, 64, 6, 128, 128, 128, 0, 1, 8)[0] \
        == api.GQA_ERR_INVALID_ARG                     # H_q not a multiple of H_kv
    assert api.gqa_attn_prefill_schedule(1, 64, 8, 128, 128, 128, 0, 1, 0)[0] \
        == api.GQA_ERR_INVALID_ARG
    assert api.gqa_attn_prefill_schedule(1, 64, 8, 96, 2048, 32768, 0, 1, 152)[0] \
        == api.GQA_ERR_UNSUPPORTED                     # d not 64 or 128
    assert api.gqa_attn_prefill_schedule(1, 64, 8, 128, 2048, 1 << 29, 0, 1, 152)[0] \
        == api.GQA_ERR_UNSUPPORTED                     # B * H_kv * S_kv >= 2^31
    assert api.gqa_attn_prefill_schedule(1, 64, 8, 128, 2048, 32768, -1, 1, 152)[0] \
        == api.GQA_ERR_INVALID_ARG
    # an item_cap smaller than the plan
    assert api.gqa_attn_prefill_schedule(2, 64, 8, 128, 2048, 32768, 30720, 1, 152,
                                         item_cap=100)[0] == api.GQA_ERR_INVALID_ARG
