// Integer planning for the decode split-KV sweep and the causal prefill tile
// schedule. Host only; the kernels recompute the same quantities with the
// device-side mirrors in plan.cuh, and tests compare both against independent
// derivations.
//
// Page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)".
//   §2.2 valid-length arithmetic  -> split bounds (contiguous chunks here)
//   §5.4 prefill tile classes     -> gqa_attn_tile_class
//   §9 tuning (split/tile sizes)  -> gqa_attn_pick_num_splits

#include <algorithm>
#include <cstdint>

#include "gqa_attn.h"
#include "plan.cuh"

namespace {

constexpr int kMinKeysPerSplit = 256;   // below this a split is mostly ramp-up
constexpr int kMaxKeysPerSplit = 1024;  // long rows spread over many blocks
constexpr int kMaxSplits = 8192;
constexpr int kClusterSplits = 16;      // splits merged on chip by one thread-block cluster

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" int gqa_attn_pick_num_splits(int B, int H_kv, int S_max, int num_sms) {
    if (B <= 0 || H_kv <= 0 || S_max <= 0 || num_sms <= 0) return GQA_ERR_INVALID_ARG;
    const int64_t pairs = int64_t(B) * H_kv;
    // Enough blocks to cover the SMs at low batch, in whole clusters of
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

// An INT8 token carries about half the bytes of a bf16 one, and the bounds
// above are per-split byte budgets written in bf16 keys.
extern "C" int gqa_attn_pick_num_splits_q8(int B, int H_kv, int S_max, int num_sms) {
    if (S_max <= 0) return GQA_ERR_INVALID_ARG;
    return gqa_attn_pick_num_splits(B, H_kv, int((int64_t(S_max) + 1) / 2), num_sms);
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
