// Integer plan shared by the host library and the kernels (host + device).
// Page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)", §2.2
// (valid-length arithmetic) and §5.4 (query block vs KV tile classes).
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define GQA_HD __host__ __device__ __forceinline__
#else
#define GQA_HD inline
#endif

namespace gqa {

constexpr int kPrefillBlockM = 128;  // query rows per prefill work item
constexpr int kPrefillBlockN = 128;  // keys per prefill KV tile

constexpr int kTileAllPast = 0;
constexpr int kTilePartial = 1;
constexpr int kTileAllFuture = 2;

struct SplitRange {
    int start;
    int end;
};

// Keys per decode split: L = ceil(S_max / num_splits).
GQA_HD int split_len(int S_max, int num_splits) {
    return int((int64_t(S_max) + num_splits - 1) / num_splits);
}

// Split s covers [s*L, (s+1)*L) on the S_max grid, clipped to [0, seqlen).
GQA_HD SplitRange split_range(int L, int s, int seqlen) {
    int64_t a = int64_t(s) * L, b = a + L;
    SplitRange r;
    r.start = int(a < seqlen ? a : seqlen);
    r.end = int(b < seqlen ? b : seqlen);
    return r;
}

// Number of non-empty splits of a row: ceil(seqlen / L).
GQA_HD int active_splits(int L, int seqlen) { return seqlen <= 0 ? 0 : (seqlen + L - 1) / L; }

// §5.4: ke <= qs -> all past; ks >= qe -> all future (skip); else partial.
GQA_HD int tile_class(int qs, int qe, int ks, int ke) {
    if (ke <= qs) return kTileAllPast;
    if (ks >= qe) return kTileAllFuture;
    return kTilePartial;
}

// Cluster size of a decode launch with ns splits per row and `ctas` CTAs in
// all: the largest of 16, 8, 4, 2 dividing ns, else 1; at most 8 when the
// grid needs more than one wave (more CTAs than the num_sms SMs), because
// smaller clusters fill the SMs that finished CTAs free more evenly.
inline int decode_cluster_size(int ns, int64_t ctas, int num_sms) {
    const int max_cs = ctas <= int64_t(num_sms) ? 16 : 8;
    for (int cs : {16, 8, 4, 2})
        if (cs <= max_cs && ns % cs == 0) return cs;
    return 1;
}

// Work order of the persistent prefill kernel, passed as a kernel parameter.
// With on == 0 the kernel walks its closed-form order (heaviest query blocks
// first over every batch and KV head, snake order over the CTAs). When the
// K/V of all (batch, KV head) groups is larger than L2 that order streams
// every group's keys from DRAM again in each round of items; the host then
// orders the items by super-groups of (batch, KV head) whose K/V fits in an
// L2 budget, heaviest first within a super-group, and gives each item to the
// CTA with the least work so far. CTA c runs item[off[c]] .. item[off[c+1]-1]
// (the kernel's own item numbers). The order changes no result: items are
// independent and each is computed the same way wherever it runs.
constexpr int kPrefillSchedCtas = 160;
constexpr int kPrefillSchedItems = 12288;
// K/V bytes per super-group: two neighbouring super-groups (the CTAs move
// from one to the next at different times) stay within the 129 MB L2
constexpr int64_t kPrefillL2Budget = int64_t(48) << 20;

struct PrefillSched {
    int on;
    uint16_t off[kPrefillSchedCtas + 1];
    uint16_t item[kPrefillSchedItems];
};

// Fills `s` for a launch of `ctas` CTAs over `items` work items (s.on = 0 and
// false when the closed-form order is kept). q_offset is relative to the first
// key of the launch; partial: a slice launch, whose blocks may see no key.
// l2_budget: K/V bytes per super-group (<= 0: always the closed-form order).
bool plan_prefill_order(PrefillSched& s, int B, int H_q, int H_kv, int d, int T_q, int S_kv,
                        int q_offset, bool causal, bool partial, int ctas, int64_t items,
                        int64_t l2_budget);

// The budget the library uses (test hook: gqa_attn_debug_prefill_order).
int64_t prefill_order_budget();

}  // namespace gqa
