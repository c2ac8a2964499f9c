// Integer planning for the decode split-KV sweep and the causal prefill tile
// schedule. Host only; the kernels recompute the same quantities with the
// device-side mirrors in plan.cuh, and tests compare both against independent
// derivations.
//
// Page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)".
//   §2.2 valid-length arithmetic  -> split bounds (contiguous chunks here)
//   §5.4 prefill tile classes     -> gqa_attn_tile_class
//   §9 tuning (split/tile sizes)  -> gqa_attn_pick_num_splits
//   §5.4 prefill scheduling       -> plan_prefill_order (work order of the
//                                    persistent prefill kernel)

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <functional>
#include <memory>
#include <queue>
#include <utility>
#include <vector>

#include "gqa_attn.h"
#include "plan.cuh"

namespace {

constexpr int kMinKeysPerSplit = 256;   // below this a split is mostly ramp-up
constexpr int kMaxKeysPerSplit = 1024;  // long rows spread over many blocks
// split bounds of the one-wave plan below: a batch of rows may be ragged (a long
// row's splits would then set the time), a single row cannot
constexpr int kMaxKeysPerWaveSplit = 2048;
constexpr int kMaxKeysPerWaveSplitOneRow = 16384;
// splits this short take the one-wave plan even with fewer than 80% of the SMs
// busy: a combine launch costs more than the idle SMs
constexpr int kShortSplitKeys = 512;
constexpr int kMaxSplits = 8192;
constexpr int kClusterSplits = 16;      // splits merged on chip by one thread-block cluster

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The split rule; one_row: the one-wave split bound for B == 1.
int pick_splits(int B, int H_kv, int S_max, int num_sms, int64_t one_row);

}  // namespace

// The bf16 decode streams a single row best in one wave even with long
// splits; the INT8 / INT4 decodes are bound by issue per SM and keep the
// batch bound (their rule below).
extern "C" int gqa_attn_pick_num_splits(int B, int H_kv, int S_max, int num_sms) {
    return pick_splits(B, H_kv, S_max, num_sms, kMaxKeysPerWaveSplitOneRow);
}

namespace {

int pick_splits(int B, int H_kv, int S_max, int num_sms, int64_t one_row) {
    if (B <= 0 || H_kv <= 0 || S_max <= 0 || num_sms <= 0) return GQA_ERR_INVALID_ARG;
    const int64_t pairs = int64_t(B) * H_kv;
    // One wave of whole-row clusters: the largest ns of 16, 8, 4, 2 whose
    // grid fits on the SMs, if it keeps >= 80% of them busy and its splits
    // hold 256..2048 keys (`one_row` for a single row), or if its splits hold
    // 256..512 keys however many SMs it uses. Each row then merges on chip in
    // one cluster and no combine kernel runs (GB300, 64/8 heads: B = 2 at 8K
    // 13.9 us with 8 splits against 19.6 with 10; B = 1 at 32K 24.3 us with
    // 16 against 28.0 with 32, at 128K 82.4 against 89.2 with 128; 28/4 heads,
    // B = 1 at 8K: 7.6 us with 16 splits on 64 CTAs against 8.9 with 32).
    const int64_t wave_max = B == 1 ? one_row : kMaxKeysPerWaveSplit;
    for (int ns : {16, 8, 4, 2}) {
        if (pairs * ns > num_sms) continue;
        const int64_t keys = ceil_div(S_max, ns);
        const bool busy = 5 * pairs * ns >= 4 * int64_t(num_sms) && keys <= wave_max;
        if (keys >= kMinKeysPerSplit && (busy || keys <= kShortSplitKeys)) return ns;
        break;
    }
    // Otherwise enough blocks to cover the SMs at low batch, in whole clusters of
    // kClusterSplits splits once a row gets that many (the decode kernel
    // merges one cluster's splits on chip).
    int64_t ns = ceil_div(num_sms, pairs);
    if (ns > kClusterSplits) {
        const int64_t whole = kClusterSplits * (ns / kClusterSplits);
        if (5 * pairs * whole >= 4 * int64_t(num_sms)) ns = whole;  // keeps >= 80% of the SMs
    }
    // Long rows spread over many blocks.
    ns = std::max<int64_t>(ns, ceil_div(S_max, kMaxKeysPerSplit));
    if (ns > kClusterSplits) ns = kClusterSplits * ceil_div(ns, kClusterSplits);
    // But no split shorter than kMinKeysPerSplit keys.
    ns = std::min<int64_t>(ns, std::max(1, S_max / kMinKeysPerSplit));
    ns = std::max<int64_t>(1, std::min<int64_t>(ns, kMaxSplits));
    return int(ns);
}

}  // namespace

// An INT8 token carries about half the bytes of a bf16 one, and the bounds
// above are per-split byte budgets written in bf16 keys; the one-wave bound
// stays 2048 for a single row too (a CTA's issue rate, not HBM, bounds these
// decodes).
extern "C" int gqa_attn_pick_num_splits_q8(int B, int H_kv, int S_max, int num_sms) {
    if (S_max <= 0) return GQA_ERR_INVALID_ARG;
    return pick_splits(B, H_kv, int((int64_t(S_max) + 1) / 2), num_sms, kMaxKeysPerWaveSplit);
}

// INT4 takes the INT8 rule. Its token is about a quarter of a bf16 one in
// bytes, but the decode over it is bound by issue, not bytes, like the INT8
// one (GB300: 8K decode 9.35 us at 16 splits vs 10.0 at 8; ragged 128K 80.4 us
// at 64 vs 89.0 at 32).
extern "C" int gqa_attn_pick_num_splits_q4(int B, int H_kv, int S_max, int num_sms) {
    return gqa_attn_pick_num_splits_q8(B, H_kv, S_max, num_sms);
}

extern "C" int gqa_attn_decode_cluster_size(int B, int H_kv, int num_splits, int num_sms) {
    if (B <= 0 || H_kv <= 0 || num_splits <= 0 || num_sms <= 0) return GQA_ERR_INVALID_ARG;
    return gqa::decode_cluster_size(num_splits, int64_t(num_splits) * H_kv * B, num_sms);
}

extern "C" int gqa_attn_split_bounds(int S_max, int num_splits, int seqlen, int32_t* starts,
                                     int32_t* ends) {
    if (S_max <= 0 || num_splits <= 0 || seqlen < 0 || seqlen > S_max || !starts || !ends)
        return GQA_ERR_INVALID_ARG;
    const int L = gqa::split_len(S_max, num_splits);
    for (int s = 0; s < num_splits; ++s) {
        gqa::SplitRange r = gqa::split_range(L, s, seqlen);
        starts[s] = r.start;
        ends[s] = r.end;
    }
    return GQA_OK;
}

extern "C" int gqa_attn_tile_class(int qs, int qe, int ks, int ke) {
    return gqa::tile_class(qs, qe, ks, ke);
}

extern "C" int gqa_attn_prefill_block_m(void) { return gqa::kPrefillBlockM; }
extern "C" int gqa_attn_prefill_block_n(void) { return gqa::kPrefillBlockN; }

extern "C" int gqa_attn_prefill_tile_counts(int T_q, int S_kv, int q_offset, int causal,
                                            int64_t* n_past, int64_t* n_partial,
                                            int64_t* n_future) {
    if (T_q < 0 || S_kv < 0 || q_offset < 0 || !n_past || !n_partial || !n_future)
        return GQA_ERR_INVALID_ARG;
    int64_t c[3] = {0, 0, 0};
    const int nm = int(ceil_div(T_q, gqa::kPrefillBlockM));
    const int nn = int(ceil_div(S_kv, gqa::kPrefillBlockN));
    for (int i = 0; i < nm; ++i) {
        const int qs = q_offset + i * gqa::kPrefillBlockM;
        const int qe = q_offset + std::min((i + 1) * gqa::kPrefillBlockM, T_q);
        for (int j = 0; j < nn; ++j) {
            const int ks = j * gqa::kPrefillBlockN;
            const int ke = std::min((j + 1) * gqa::kPrefillBlockN, S_kv);
            c[causal ? gqa::tile_class(qs, qe, ks, ke) : gqa::kTileAllPast]++;
        }
    }
    *n_past = c[gqa::kTileAllPast];
    *n_partial = c[gqa::kTilePartial];
    *n_future = c[gqa::kTileAllFuture];
    return GQA_OK;
}

namespace gqa {

namespace {

std::atomic<int64_t> g_order_budget{-1};  // < 0: kPrefillL2Budget

// The prefill kernel's item numbering (pair_item in prefill.cu), host side:
// item L's (batch, KV head) group and the KV tiles it runs.
struct ItemShape {
    int group;
    int n;
};

ItemShape prefill_item(int B, int H_q, int H_kv, int T_q, int S_kv, int q_offset, bool causal,
                       bool partial, bool blocks, int64_t L) {
    const int G = H_q / H_kv, BM = kPrefillBlockM, BN = kPrefillBlockN;
    const int tiles = int(ceil_div(S_kv, BN)), n_mblocks = int(ceil_div(T_q, BM));
    auto block_tiles = [&](int row0) {
        if (row0 >= T_q) return 0;
        const int qe = q_offset + std::min(row0 + BM, T_q);
        if (!causal) return tiles;
        if (partial && qe <= 0) return 0;  // the slice starts past these queries
        return std::min(tiles, (qe - 1) / BN + 1);
    };
    ItemShape r{};
    if (blocks) {  // two consecutive query blocks of one head
        const int64_t bh_count = int64_t(B) * H_q;
        const int bpi = int((n_mblocks + 1) / 2 - 1 - L / bh_count);
        const int bh = int(L % bh_count), b = bh / H_q, h = bh % H_q;
        r.group = b * H_kv + h / G;
        r.n = std::max(block_tiles(2 * bpi * BM), block_tiles((2 * bpi + 1) * BM));
    } else {  // one query block of two heads
        const int pairs = H_q / 2;
        const int64_t bp_count = int64_t(B) * pairs;
        const int m = int(n_mblocks - 1 - L / bp_count), bp = int(L % bp_count);
        const int b = bp / pairs, h = (bp % pairs) * 2;
        r.group = b * H_kv + h / G;
        r.n = block_tiles(m * BM);
    }
    return r;
}

}  // namespace

int64_t prefill_order_budget() {
    const int64_t b = g_order_budget.load(std::memory_order_relaxed);
    return b < 0 ? kPrefillL2Budget : b;
}

bool plan_prefill_order(PrefillSched& s, int B, int H_q, int H_kv, int d, int T_q, int S_kv,
                        int q_offset, bool causal, bool partial, int ctas, int64_t items,
                        int64_t l2_budget) {
    s.on = 0;
    if (l2_budget <= 0 || ctas <= 0 || ctas > kPrefillSchedCtas || items <= 0 ||
        items > kPrefillSchedItems || B <= 0 || H_kv <= 0 || H_q % H_kv != 0 || S_kv <= 0)
        return false;
    const int64_t group_bytes = int64_t(S_kv) * d * 2 * 2;  // K and V rows, bf16
    const int64_t groups = int64_t(B) * H_kv;
    if (group_bytes * groups <= l2_budget) return false;  // all of K/V stays in L2
    // n_sg super-groups whose sizes differ by at most one group (a small last
    // one would end the launch on its heaviest items): group g is in
    // super-group g * n_sg / groups
    const int64_t sg_max = std::max<int64_t>(1, l2_budget / group_bytes);
    const int64_t n_sg = ceil_div(groups, sg_max);
    const bool blocks = (H_q / H_kv) % 2 != 0;
    struct Key {
        int64_t sg;
        int n;
        int L;
    };
    std::vector<Key> keys(static_cast<size_t>(items));
    for (int64_t L = 0; L < items; ++L) {
        const ItemShape it = prefill_item(B, H_q, H_kv, T_q, S_kv, q_offset, causal, partial,
                                          blocks, L);
        keys[size_t(L)] = Key{int64_t(it.group) * n_sg / groups, it.n, int(L)};
    }
    std::sort(keys.begin(), keys.end(), [](const Key& a, const Key& b) {
        if (a.sg != b.sg) return a.sg < b.sg;
        if (a.n != b.n) return a.n > b.n;
        return a.L < b.L;
    });
    // greedy: the next item to the CTA with the least work so far (ties: the
    // lowest CTA index); an item costs its KV tiles plus about one tile of
    // Q load and epilogue
    using Load = std::pair<int64_t, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> free_at;
    for (int c = 0; c < ctas; ++c) free_at.push({0, c});
    std::vector<std::vector<uint16_t>> per(static_cast<size_t>(ctas));
    for (const Key& k : keys) {
        const Load t = free_at.top();
        free_at.pop();
        per[size_t(t.second)].push_back(uint16_t(k.L));
        free_at.push({t.first + k.n + 1, t.second});
    }
    int at = 0;
    for (int c = 0; c < ctas; ++c) {
        s.off[c] = uint16_t(at);
        for (uint16_t L : per[size_t(c)]) s.item[at++] = L;
    }
    s.off[ctas] = uint16_t(at);
    s.on = 1;
    return true;
}

}  // namespace gqa

extern "C" int gqa_attn_prefill_schedule(int B, int H_q, int H_kv, int d, int T_q, int S_kv,
                                         int q_offset, int causal, int num_ctas, int32_t* off,
                                         int32_t* items, int item_cap) {
    // the prefill entry points' own limits
    if (B <= 0 || B > 65535 || H_q <= 0 || H_kv <= 0 || H_q % H_kv != 0 || T_q < 0 ||
        S_kv <= 0 || q_offset < 0 || num_ctas <= 0 || !off || !items || item_cap < 0)
        return GQA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GQA_ERR_UNSUPPORTED;
    if (int64_t(B) * H_q * T_q >= (int64_t(1) << 31) ||
        int64_t(B) * H_kv * S_kv >= (int64_t(1) << 31))
        return GQA_ERR_UNSUPPORTED;
    const bool blocks = (H_q / H_kv) % 2 != 0;
    const int64_t n_mblocks = ceil_div(T_q, gqa::kPrefillBlockM);
    const int64_t n_items = blocks ? (n_mblocks + 1) / 2 * B * H_q : n_mblocks * B * (H_q / 2);
    auto s = std::make_unique<gqa::PrefillSched>();
    if (!gqa::plan_prefill_order(*s, B, H_q, H_kv, d, T_q, S_kv, q_offset, causal != 0, false,
                                 num_ctas, n_items, gqa::prefill_order_budget()))
        return 0;
    const int n = s->off[num_ctas];
    if (n > item_cap) return GQA_ERR_INVALID_ARG;
    for (int c = 0; c <= num_ctas; ++c) off[c] = s->off[c];
    for (int i = 0; i < n; ++i) items[i] = s->item[i];
    return n;
}

extern "C" int gqa_attn_debug_prefill_order(int64_t budget_bytes) {
    gqa::g_order_budget.store(budget_bytes < 0 ? -1 : budget_bytes, std::memory_order_relaxed);
    return GQA_OK;
}
