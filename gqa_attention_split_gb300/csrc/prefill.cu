// Causal GQA prefill for sm_103a on the 5th-generation tensor cores.
//
// Page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)".
//   §3 per-tile op sequence: S_j = Q K_j^T * scale (+ boundary mask),
//        m_new = max(m, rowmax S_j), P = exp(S_j - m_new), corr = exp(m - m_new),
//        l = l*corr + rowsum P, O = O*corr + P V_j; normalise O / l at the end.
//   §5.4 prefill, no SP: a query block [qs, qe) against KV tile [ks, ke) is
//        all-past (ke <= qs: no mask), all-future (ks >= qe: skipped) or
//        partial (masked), in global positions (chunked prefill at q_offset).
//
// GB300 mapping (prefill_pair_kernel below): a persistent kernel, one CTA per
// SM, walks work items heaviest first. A work item is two groups of 128
// query rows that read the same K/V tiles: one query block of two heads of a
// KV group (even G, the page's GQA lever of folding a group's heads together
// applied to prefill), or two consecutive query blocks of one head (odd G).
// A TMA warp streams Q and the K/V tiles, one thread issues every tcgen05.mma
// (S = Q K^T into tensor memory, O += P V with P read from tensor memory),
// and one softmax warpgroup per group runs the online softmax row by row
// (one query row per thread) and the epilogue.
// Every wait is bounded and reports a timeout in the status word.

#include <cuda_runtime.h>
#include <math.h>

#include <array>
#include <memory>
#include <mutex>
#include <utility>
#include <vector>

#include "gqa_attn.h"
#include "plan.cuh"
#include "ptx.cuh"
#include "runtime.cuh"
#include "tcgen05.cuh"
#include "trace.cuh"

namespace gqa {
namespace prefill {

constexpr int BM = kPrefillBlockM;  // 128 query rows per work item
constexpr int BN = kPrefillBlockN;  // 128 keys per KV tile
constexpr uint32_t kBoxBytes = 128 * 128;        // [128 rows][64 bf16]: one TMA box
constexpr uint32_t kTmemCols = 512;  // S_0, S_1, O_0, O_1: 128 columns each
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units: rescale O when max grows by > 256x

struct Params {
    uint16_t* o;        // [B, H_q, T_q, d]
    float* o32;         // partial prefill: O in fp32 instead of o
    float* lse;         // [B, H_q, T_q] or null
    unsigned* status;
    int B, H_q, H_kv, G, T_q, S_kv, q_offset, causal, n_mblocks;
    float scale_log2;
    int inject_timeout;  // test hook: block 0 withholds its (first) Q copy
};

#ifdef GQA_DEBUG
// Debug builds only: S = Q K^T tiles the MMA issuers actually issued, per
// (batch, query head, query block, KV tile), split by the §5.4 class of the
// tile (all past, partial, all future). A correct schedule issues no
// all-future tile and exactly the all-past and partial ones.
static __device__ unsigned long long g_dbg_tiles[3];

__device__ __forceinline__ void dbg_count_tile(unsigned long long (&cnt)[3], const Params& p,
                                               int qs, int qe, int j, int heads) {
    const int ks = j * BN, ke = min(ks + BN, p.S_kv);
    cnt[p.causal ? tile_class(qs, qe, ks, ke) : kTileAllPast] += heads;
}
__device__ __forceinline__ void dbg_flush_tiles(const unsigned long long (&cnt)[3]) {
    for (int c = 0; c < 3; ++c)
        if (cnt[c]) atomicAdd(&g_dbg_tiles[c], cnt[c]);
}
#define GQA_DBG(...) __VA_ARGS__
#else
#define GQA_DBG(...)
#endif

__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, int x, int y,
                                         int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// MMAs with the descriptors given as 32-bit halves: the k-steps of one
// operand differ only in the start-address field of the low word, so each
// step adds to the low word alone; kAcc fixed at compile time needs no flag.
template <int kAcc>
__device__ __forceinline__ void mma_ss_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                          uint32_t b_lo, uint32_t b_hi, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "mov.b64 da, {%1, %2};\n\t"
        "mov.b64 db, {%3, %4};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "n"(kAcc)
        : "memory");
}
__device__ __forceinline__ void mma_ts_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                          uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}


// ---------------------------------------------------------------------------
// The prefill kernel. A work item is two groups of 128 query rows that read
// the same K/V tiles: with an even G, one query block of two query heads of a
// KV group (the page's GQA lever, §5.2, fold the G heads into the matmul M
// dimension, applied to prefill); with an odd G, two consecutive query blocks
// of one head. Every K/V tile loaded into shared memory serves 2 x 128 query
// rows. P stays in tensor memory (written over its own S columns) and feeds the
// P.V MMA as the A operand, so shared memory only carries Q, K, V.
//
// Persistent: one CTA per SM walks the work items heaviest first (snake order
// over the CTAs), so the next item's Q load and first S overlap the previous
// item's epilogue, and the tensor memory is allocated once.
//   warpgroup 0 (104 registers/thread): warp 0 TMA (per item: Q of both
//               groups, then K_j, V_j through a 4-slot ring); warp 1 owns the
//               tensor memory and one thread of it issues every MMA, per KV
//               tile j: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1), each only while
//               its group has tiles (the groups of a block pair have different
//               causal extents). An S MMA overwrites the P the previous PV of
//               its group read; the tcgen05.mma operations of one thread
//               execute and complete in issue order. Warps 2 and 3 only wait.
//   warpgroups 1 and 2 (200 registers/thread): softmax of group A and of
//               group B, then that group's epilogue (O through TMA stores);
//               while one group computes, the tensor core runs the other
//               group's MMAs.
// Register split: 128 x 104 + 256 x 200 = 64512 = 384 threads x 168 at launch.
// Every barrier phase is counted across items: the k-th completion of a
// barrier has parity k & 1 (per group for the S, P and O barriers).

constexpr int kPairThreads = 384;
// Four slots of one tile each: ring item r (K_j or V_j of some work item)
// reuses the slot of item r - 4; the loads land well before their MMAs.
constexpr int kRingSlots = 4;
// O leaves through TMA stores: each softmax warp owns two 2 KB buffers, each
// one [32 rows][32 bf16] box in the 64-byte swizzle (16-byte chunk k of row
// r at r * 64 + ((k ^ ((r >> 1) & 3)) << 4), so a warp's row-per-lane writes
// hit distinct banks).
constexpr uint32_t kStageBoxBytes = 32 * 32 * 2;

// Shared-memory layout for head dim D (64 or 128): a tile of 128 rows is D/64
// boxes of 64 columns.
template <int D>
struct PairGeo {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kBoxes = D / 64;
    static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;
    static constexpr uint32_t kQOff = 0;                                  // Q_A, then Q_B
    static constexpr uint32_t kRingOff = 2 * kTileBytes;                  // kRingSlots tiles
    static constexpr uint32_t kStageOff = kRingOff + kRingSlots * kTileBytes;
    static constexpr uint32_t kBarOff = kStageOff + 8 * 2 * kStageBoxBytes;
    static constexpr int kSmemBytes = 1024 + kBarOff + 256;
    static_assert(kSmemBytes <= 232448, "more dynamic shared memory than one CTA may have");
};
// S_g (and P_g over its first 64 columns) at g*128; O_g at 256 + g*128.
__device__ __forceinline__ uint32_t col_s_of(int g) { return uint32_t(g) * 128u; }
__device__ __forceinline__ uint32_t col_o_of(int g) { return 256u + uint32_t(g) * 128u; }

enum PairBar {
    pQFull = 0,                        // Q of both groups landed (per item)
    pQEmpty = 1,                       // the item's last S MMAs have completed
    pSlotFull = 2,                     // x kRingSlots
    pSlotEmpty = pSlotFull + kRingSlots,  // x kRingSlots, released by the MMA thread's commits
    pSFull = pSlotEmpty + kRingSlots,  // x2: S_g ready (per tile)
    pPFull = pSFull + 2,               // x2: P_g ready (4 softmax warps)
    pODone = pPFull + 2,               // x2: O_g final (per item)
    pDrain = pODone + 2,               // the MMA issuer's last commit
    pNumBars = pDrain + 1
};
static_assert(pNumBars * 8 + 4 <= 256, "barrier area");

// One work item: two groups of 128 query rows that read the same K/V tiles.
// Even G: one query block of two adjacent query heads of a KV group. Odd G
// (pair_blocks): two consecutive query blocks of one head. Items are numbered
// heaviest first (query blocks from the last one down), and a CTA takes items
// c, 2G-1-c, 2G+c, ... (snake order), or the items a host-made order
// (PrefillSched, plan.cuh) lists for it. Each group has its own KV tile count
// (causal: up to its own last query), possibly 0 (the second block of a head
// with an odd block count); the item runs the larger one.
struct PairItem {
    int b, kvh;
    int head[2];   // query head of group g
    int row0[2];   // first query row of group g (row0 >= T_q: an empty group)
    int qs[2];     // global position of that row
    int qe[2];     // one past the group's last query (global); qe <= qs when empty
    int n[2];      // KV tiles of group g
    int n_tiles;   // max(n[0], n[1])
    // (head pairs set only the [0] fields and n_tiles: head[1] = head[0] + 1,
    // the rest equal)
};

// kBlocks: the groups are two query blocks of one head (odd G), else one
// block of two heads (even G; then both groups share row0, qs, qe and n).
// kPartial: a prefill over one slice of the keys, where the query offset
// relative to the slice may be negative and a block may see no key (n = 0).
template <bool kBlocks, bool kPartial>
__device__ __forceinline__ bool pair_item(const Params& p, const PrefillSched& sch, int it,
                                          PairItem& w) {
    const int G = gridDim.x, c = blockIdx.x;
    int L;
    if (sch.on) {
        const int i = sch.off[c] + it;
        if (i >= sch.off[c + 1]) return false;
        L = sch.item[i];
    } else {
        L = it * G + ((it & 1) ? G - 1 - c : c);
    }
    int h;
    if constexpr (kBlocks) {
        const int tiles = (p.S_kv + BN - 1) / BN;
        int mb[2];
        const int n_bpairs = (p.n_mblocks + 1) / 2, bh_count = p.B * p.H_q;
        if (L >= n_bpairs * bh_count) return false;
        const int bpi = n_bpairs - 1 - L / bh_count, bh = L % bh_count;
        w.b = bh / p.H_q;
        h = bh % p.H_q;
        w.head[0] = w.head[1] = h;
        mb[0] = 2 * bpi;
        mb[1] = 2 * bpi + 1;
        w.kvh = h / p.G;
        for (int g = 0; g < 2; ++g) {
            w.row0[g] = mb[g] * BM;
            w.qs[g] = p.q_offset + w.row0[g];
            w.qe[g] = p.q_offset + min(w.row0[g] + BM, p.T_q);
            int n = w.row0[g] < p.T_q ? tiles : 0;
            if (p.causal && n > 0) {
                if (kPartial && w.qe[g] <= 0) n = 0;  // the slice starts past these queries
                else n = min(n, (w.qe[g] - 1) / BN + 1);  // all-future tiles skipped
            }
            w.n[g] = n;
        }
        w.n_tiles = max(w.n[0], w.n[1]);
    } else {
        const int pairs = p.H_q / 2, bp_count = p.B * pairs;
        if (L >= p.n_mblocks * bp_count) return false;
        const int m = p.n_mblocks - 1 - L / bp_count, bp = L % bp_count;
        // only the [0] fields and n_tiles: head pairs never read the others
        w.b = bp / pairs;
        h = (bp % pairs) * 2;
        w.head[0] = h;
        w.kvh = h / p.G;
        w.row0[0] = m * BM;
        w.qs[0] = p.q_offset + m * BM;
        w.qe[0] = p.q_offset + min(m * BM + BM, p.T_q);
        w.n_tiles = (p.S_kv + BN - 1) / BN;
        if (p.causal) w.n_tiles = min(w.n_tiles, (w.qe[0] - 1) / BN + 1);  // all-future skipped
        if constexpr (kPartial) {  // the per-group path reads every field
            if (p.causal && w.qe[0] <= 0) w.n_tiles = 0;
            w.head[1] = h + 1;
            w.row0[1] = w.row0[0];
            w.qs[1] = w.qs[0];
            w.qe[1] = w.qe[0];
            w.n[0] = w.n[1] = w.n_tiles;
        }
    }
    return true;
}

template <bool kBlocks, int D, bool kPartial = false>
__global__ void __launch_bounds__(kPairThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ CUtensorMap tmap_o, const Params p,
                        const __grid_constant__ PrefillSched sched) {
    using Gm = PairGeo<D>;
    constexpr uint32_t kTileBytes = Gm::kTileBytes;
    // per-group bookkeeping: block pairs, or slices where a group may see no key
    constexpr bool kGen = kBlocks || kPartial;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Gm::kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Gm::kBarOff + pNumBars * 8);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar(pQFull), 1);
        mbar_init(bar(pQEmpty), 1);
        for (int s = 0; s < kRingSlots; ++s) {
            mbar_init(bar(pSlotFull + s), 1);
            mbar_init(bar(pSlotEmpty + s), 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(bar(pSFull + g), 1);
            mbar_init(bar(pPFull + g), 4);
            mbar_init(bar(pODone + g), 1);
        }
        mbar_init(bar(pDrain), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int wg = warp >> 2;
    PairItem w;

    if (wg == 0) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 104;" ::: "memory");
      if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ TMA producer
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
        bool alive = true;
        int r = 0;        // ring items issued so far, over all work items
        int q_loads = 0;  // Q loads issued (one per work item)
        for (int it = 0; alive && pair_item<kBlocks, kPartial>(p, sched, it, w); ++it) {
            // Q of both heads; the previous item's last S MMAs must be done.
            if (it > 0) alive = mbar_wait_bounded(bar(pQEmpty), (it - 1) & 1, p.status);
            if (!alive) break;
            // Test hook: block 0 withholds its first Q copy, so every wait on
            // it runs out and reports kStatusTimeout (nothing faults or hangs).
            if (!(p.inject_timeout && blockIdx.x == 0 && it == 0)) {
                // (an empty group's rows lie past T_q: the copy reads zero fill)
                mbar_arrive_expect_tx(bar(pQFull), 2 * kTileBytes);
                for (int g = 0; g < 2; ++g)
                    for (int hh = 0; hh < Gm::kBoxes; ++hh)
                        tma_load(smem_u32(smem + Gm::kQOff + g * kTileBytes) + hh * kBoxBytes,
                                 &tmap_q, hh * 64, kBlocks ? w.row0[g] : w.row0[0],
                                 w.b * p.H_q + (kBlocks ? w.head[g] : w.head[0] + g),
                                 bar(pQFull));
                q_loads = it + 1;
            }
            for (int i = 0; i < 2 * w.n_tiles; ++i, ++r) {  // K_0, V_0, K_1, V_1, ...
                const int s = r % kRingSlots;
                if (r >= kRingSlots)
                    alive = mbar_wait_bounded(bar(pSlotEmpty + s), ((r / kRingSlots) - 1) & 1,
                                              p.status);
                if (!alive) break;
                const CUtensorMap* map = (i & 1) ? &tmap_v : &tmap_k;
                const uint32_t dst = smem_u32(smem + Gm::kRingOff + s * kTileBytes);
                mbar_arrive_expect_tx(bar(pSlotFull + s), kTileBytes);
                for (int hh = 0; hh < Gm::kBoxes; ++hh)
                    tma_load(dst + hh * kBoxBytes, map, hh * 64, (i >> 1) * BN,
                             w.b * p.H_kv + w.kvh, bar(pSlotFull + s));
            }
        }
        // Every copy still in flight lands before the CTA exits (only the
        // last kRingSlots ring items and the last Q can be outstanding).
        if (q_loads > 0) mbar_wait_bounded(bar(pQFull), (q_loads - 1) & 1, p.status);
        for (int i = max(0, r - kRingSlots); i < r; ++i)
            mbar_wait_bounded(bar(pSlotFull + i % kRingSlots), (i / kRingSlots) & 1, p.status);
      } else if (warp == 1 && lane == 0) {
        // -------------------------------------------------------- MMA issuer
        // Per KV tile j: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1); S_A(0), S_B(0)
        // of an item follow the previous item's last PV MMAs.
        const uint32_t idesc_s = tc::idesc_bf16_f32(BM, BN, false);
        const uint32_t idesc_pv = tc::idesc_bf16_f32(BM, D, true);
        auto slot_addr = [&](int i) {
            return smem_u32(smem + Gm::kRingOff + (i % kRingSlots) * kTileBytes);
        };
        auto wait_item = [&](int i) {
            return mbar_wait_bounded(bar(pSlotFull + i % kRingSlots), (i / kRingSlots) & 1, p.status);
        };
        // Descriptors are built once per operand; each k-step adds its byte
        // offset >> 4 to the 14-bit start-address field (shared addresses
        // stay below 256 KB, so the field never carries out).
        const uint64_t qdesc0 = tc::sdesc_sw128(smem_u32(smem + Gm::kQOff), 16, 1024);
        const uint64_t qdesc1 = tc::sdesc_sw128(smem_u32(smem + Gm::kQOff + kTileBytes), 16, 1024);
        auto issue_s = [&](int g, int ri) {  // S_g = Q_g K^T, K in ring item ri
            const uint64_t qdesc = g ? qdesc1 : qdesc0;
            const uint64_t kdesc = tc::sdesc_sw128(slot_addr(ri), 16, 1024);
            const uint32_t qlo = uint32_t(qdesc), qhi = uint32_t(qdesc >> 32);
            const uint32_t klo = uint32_t(kdesc), khi = uint32_t(kdesc >> 32);
            const uint32_t dst = tmem + col_s_of(g);
            mma_ss_lo<0>(dst, qlo, qhi, klo, khi, idesc_s);
#pragma unroll
            for (int kk = 1; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
                mma_ss_lo<1>(dst, qlo + off, qhi, klo + off, khi, idesc_s);
            }
            tc::commit(bar(pSFull + g));
        };
        auto issue_pv = [&](int g, int ri, bool first) {  // O_g (+)= P_g V, V in ring item ri
            const uint64_t vdesc = tc::sdesc_sw128(slot_addr(ri), kBoxBytes, 1024);
            const uint32_t vlo = uint32_t(vdesc), vhi = uint32_t(vdesc >> 32);
            const uint32_t dst = tmem + col_o_of(g), src = tmem + col_s_of(g);
            mma_ts_lo(dst, src, vlo, vhi, idesc_pv, first ? 0u : 1u);
#pragma unroll
            for (int ks = 1; ks < BN / 16; ++ks)
                mma_ts_lo(dst, src + ks * 8, vlo + uint32_t((ks * 2048) >> 4), vhi, idesc_pv, 1u);
        };
        bool alive = true;
        int r = 0;                // ring items consumed so far
        int tt[2] = {0, 0};       // KV tiles group g finished so far (its S and P phases)
        GQA_DBG(unsigned long long dbg[3] = {0, 0, 0};)
        for (int it = 0; alive && pair_item<kBlocks, kPartial>(p, sched, it, w); ++it) {
            const int n = w.n_tiles;
            if constexpr (kPartial) {
                if (n == 0) {  // no group sees a key of this slice: Q is free again
                    alive = mbar_wait_bounded(bar(pQFull), it & 1, p.status);
                    tc::commit(bar(pQEmpty));
                    continue;
                }
            }
            alive = mbar_wait_bounded(bar(pQFull), it & 1, p.status) && wait_item(r);
            if (!alive) break;
            tc::fence_after_sync();
            if constexpr (!kGen) {
                // two heads, one query block: both groups run every tile
                issue_s(0, r);
                issue_s(1, r);
                GQA_DBG(dbg_count_tile(dbg, p, w.qs[0], w.qe[0], 0, 2);)
                tc::commit(bar(pSlotEmpty + r % kRingSlots));  // K_0 read by both S MMAs
                if (n == 1) tc::commit(bar(pQEmpty));
                for (int j = 0; j < n && alive; ++j) {
                    const bool more = j + 1 < n;
                    const int rv = r + 2 * j + 1;  // V_j; K_{j+1} follows it
                    // the loads first (they land early), so that once P is ready
                    // only the fence and the issue remain
                    alive = wait_item(rv);
                    if (alive && more) alive = wait_item(rv + 1);
                    for (int g = 0; g < 2 && alive; ++g) {
                        // P_g(0) of an item is written after the softmax threads
                        // have read the previous item's O_g, so PV_g(0) may
                        // overwrite it.
                        alive = mbar_wait_bounded(bar(pPFull + g), (tt[0] + j) & 1, p.status);
                        if (!alive) break;
                        tc::fence_after_sync();
                        issue_pv(g, rv, j == 0);
                        if (g == 1) tc::commit(bar(pSlotEmpty + rv % kRingSlots));  // V_j done
                        if (more) {
                            issue_s(g, rv + 1);
                            GQA_DBG(dbg_count_tile(dbg, p, w.qs[0], w.qe[0], j + 1, 1);)
                            if (g == 1) {
                                tc::commit(bar(pSlotEmpty + (rv + 1) % kRingSlots));  // K_{j+1}
                                if (j + 2 == n) tc::commit(bar(pQEmpty));  // last S of the item
                            }
                        } else {
                            tc::commit(bar(pODone + g));
                        }
                    }
                }
                tt[0] += n;
                tt[1] += n;
            } else {
                // two query blocks of one head: group g runs its own n[g] tiles
                // (possibly 0). The last group that reads K_t / V_t (t < n) is
                // group 1 while it has tiles, else group 0.
                auto last_user = [&](int t) { return t < w.n[1] ? 1 : 0; };
                if (w.n[0] > 0) {
                    issue_s(0, r);
                    GQA_DBG(dbg_count_tile(dbg, p, w.qs[0], w.qe[0], 0, 1);)
                }
                if (w.n[1] > 0) {
                    issue_s(1, r);
                    GQA_DBG(dbg_count_tile(dbg, p, w.qs[1], w.qe[1], 0, 1);)
                }
                tc::commit(bar(pSlotEmpty + r % kRingSlots));  // K_0 read by the S MMAs
                if (n == 1) tc::commit(bar(pQEmpty));
                for (int j = 0; j < n && alive; ++j) {
                    const int rv = r + 2 * j + 1;  // V_j; K_{j+1} follows it
                    alive = wait_item(rv);
                    if (alive && j + 1 < n) alive = wait_item(rv + 1);
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        if (!alive) break;
                        const int n_g = g ? w.n[1] : w.n[0];
                        if (j >= n_g) continue;  // this group has no tile j
                        alive = mbar_wait_bounded(bar(pPFull + g),
                                                  ((g ? tt[1] : tt[0]) + j) & 1, p.status);
                        if (!alive) break;
                        tc::fence_after_sync();
                        issue_pv(g, rv, j == 0);
                        if (g == last_user(j)) tc::commit(bar(pSlotEmpty + rv % kRingSlots));
                        if (j + 1 < n_g) {
                            issue_s(g, rv + 1);
                            GQA_DBG(dbg_count_tile(dbg, p, g ? w.qs[1] : w.qs[0],
                                                   g ? w.qe[1] : w.qe[0], j + 1, 1);)
                            if (g == last_user(j + 1)) {
                                tc::commit(bar(pSlotEmpty + (rv + 1) % kRingSlots));  // K_{j+1}
                                if (j + 2 == n) tc::commit(bar(pQEmpty));  // last S of the item
                            }
                        } else {
                            tc::commit(bar(pODone + g));
                        }
                    }
                }
                tt[0] += w.n[0];
                tt[1] += w.n[1];
            }
            r += 2 * n;
        }
        GQA_DBG(dbg_flush_tiles(dbg);)
        // No MMA may still run when the tensor memory is freed.
        tc::commit(bar(pDrain));
        mbar_wait_bounded(bar(pDrain), 0, p.status);
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 200;" ::: "memory");
        // ------------------------------------------------ softmax warpgroups
        const int g = wg - 1;                 // the item's group 0 or 1
        const int quad = warp & 3;            // tensor-memory lanes 32*quad .. +31
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);
        const uint32_t col_s = col_s_of(g), col_o = col_o_of(g);
        const uint32_t stage = smem_u32(smem + Gm::kStageOff + (g * 4 + quad) * 2 * kStageBoxBytes);
        const uint64_t c2 = f2pack(p.scale_log2, p.scale_log2);
        bool alive = true;
        int tt = 0;   // KV tiles this group finished so far, over all work items
        [[maybe_unused]] int itg = 0;  // block pairs: items in which this group had tiles
        for (int it = 0; alive && pair_item<kBlocks, kPartial>(p, sched, it, w); ++it) {
            // this group's fields (selected, not indexed: they stay in registers)
            const int ng = kGen ? (g ? w.n[1] : w.n[0]) : w.n_tiles;
            if constexpr (kGen) {
                if (ng == 0) {  // past the last query, or (slices) no key visible: no MMAs
                    if constexpr (kPartial) {  // these rows' result: O = 0, lse = -inf
                        const int row0_z = kBlocks && g ? w.row0[1] : w.row0[0];
                        const int head_z = kBlocks ? w.head[0] : w.head[0] + g;
                        if (row0_z + row < p.T_q) {
                            const size_t orow =
                                (size_t(w.b) * p.H_q + head_z) * p.T_q + row0_z + row;
                            float4* dst = reinterpret_cast<float4*>(p.o32 + orow * D);
#pragma unroll
                            for (int i = 0; i < D / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                            p.lse[orow] = -INFINITY;
                        }
                    }
                    continue;
                }
            }
            const int qs_g = kBlocks && g ? w.qs[1] : w.qs[0];
            const int qe_g = kBlocks && g ? w.qe[1] : w.qe[0];
            const int qg = qs_g + row;
            float m_run = -INFINITY, l_run = 0.f, lb_run = 0.f;
            for (int j = 0; j < ng && alive; ++j) {
                alive = __all_sync(0xffffffffu,
                                   mbar_wait_bounded(bar(pSFull + g), (tt + j) & 1, p.status));
                if (!alive) break;
                tc::fence_after_sync();
                float sv[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tc::tmem_ld32(lane_base + col_s + c * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(r[i]);
                }
                tc::tmem_wait_ld();

                const int ks = j * BN, ke = min(ks + BN, p.S_kv);
                const bool masked =
                    (p.causal && tile_class(qs_g, qe_g, ks, ke) == kTilePartial) ||
                    (ke - ks < BN);
                if (masked) {
                    const int lim = (p.causal ? min(qg, p.S_kv - 1) : p.S_kv - 1) - ks;
#pragma unroll
                    for (int c = 0; c < BN; ++c) sv[c] = c <= lim ? sv[c] : -INFINITY;
                }
                float mx;
                {
                    float mm[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mm[i] = fmaxf(sv[i], sv[8 + i]);
#pragma unroll
                    for (int c = 16; c < BN; c += 16)
#pragma unroll
                        for (int i = 0; i < 8; ++i) mm[i] = fmax3(mm[i], sv[c + i], sv[c + 8 + i]);
                    mx = fmax3(fmax3(mm[0], mm[1], mm[2]), fmax3(mm[3], mm[4], mm[5]),
                               fmaxf(mm[6], mm[7]));
                }
                const float m_new = fmaxf(m_run, mx * p.scale_log2);
                const bool need = m_new > m_run + kRescaleThreshold;
                const float corr = need ? fast_exp2(m_run - m_new) : 1.f;
                const float m_use = need ? m_new : m_run;
                m_run = m_use;
                // p = 2^(s*scale - m): sums of p and of bf16(p); P (bf16 pairs,
                // lower key in the low half) over the first 64 columns of S.
                // (slices: a row that has seen no visible key keeps m = -inf; its
                // p must come out 0, not NaN, so it subtracts 0 instead)
                const float m_sub = (kPartial && m_use == -INFINITY) ? 0.f : m_use;
                const uint64_t n2 = f2pack(-m_sub, -m_sub);
                uint64_t s2[4];
                float bl[4], bh[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    s2[u] = 0ull;
                    bl[u] = bh[u] = 0.f;
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int c = half * 64 + 2 * i;
                        float x0, x1;
                        f2unpack(ffma2(f2pack(sv[c], sv[c + 1]), c2, n2), x0, x1);
                        const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
                        s2[i & 3] = fadd2(s2[i & 3], f2pack(e0, e1));
                        pk[i] = pack_bf16x2(e0, e1);
                        bl[i & 3] = add_f32_bf16_lo(bl[i & 3], pk[i]);
                        bh[i & 3] = add_f32_bf16_hi(bh[i & 3], pk[i]);
                    }
                    tc::tmem_st32(lane_base + col_s + half * 32, pk);
                }
                {
                    float t[8], tb[8];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        f2unpack(s2[u], t[2 * u], t[2 * u + 1]);
                        tb[2 * u] = bl[u];
                        tb[2 * u + 1] = bh[u];
                    }
                    l_run = l_run * corr +
                            (((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7])));
                    lb_run = lb_run * corr + (((tb[0] + tb[1]) + (tb[2] + tb[3])) +
                                              ((tb[4] + tb[5]) + (tb[6] + tb[7])));
                }
                // O is complete here: this tile's S MMA was issued after the
                // previous P.V, and tcgen05 MMAs complete in order. Done after
                // the exponentials, when the scores no longer hold registers.
                if (j > 0 && __any_sync(0xffffffffu, need)) {
                    const uint64_t corr2 = f2pack(corr, corr);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tc::tmem_ld32(lane_base + col_o + c * 32, r);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float a0, a1;
                            f2unpack(fmul2(f2pack(__uint_as_float(r[2 * i]),
                                                  __uint_as_float(r[2 * i + 1])),
                                           corr2),
                                     a0, a1);
                            r[2 * i] = __float_as_uint(a0);
                            r[2 * i + 1] = __float_as_uint(a1);
                        }
                        tc::tmem_st32(lane_base + col_o + c * 32, r);
                    }
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(pPFull + g));
            }
            if (!alive) break;

            // ---- epilogue: O / l -> bf16, lse = (m + log2 l) * ln 2. Every
            // read of O_g completes (wait::ld) before this warp's next P
            // arrive, which is what lets the next item's PV_g(0) overwrite O_g.
            alive = __all_sync(0xffffffffu, mbar_wait_bounded(bar(pODone + g),
                                                              (kGen ? itg : it) & 1, p.status));
            if (!alive) break;
            tc::fence_after_sync();
            const int row0_g = kBlocks && g ? w.row0[1] : w.row0[0];
            const int head_g = kBlocks ? w.head[0] : w.head[0] + g;
            const bool valid = row0_g + row < p.T_q;
            const size_t orow = (size_t(w.b) * p.H_q + head_g) * p.T_q + row0_g + row;
            if constexpr (kPartial) {
                // fp32 O for the merge, through the same staging buffers and TMA
                // stores as bf16: a chunk is 16 fp32 columns, 64 B per row like
                // 32 bf16 columns. A row that saw no key of the slice gets O = 0
                // and lse = -inf.
                const float inv = lb_run > 0.f ? 1.f / lb_run : 0.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tc::tmem_ld32(lane_base + col_o + c * 32, r);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int chunk = 2 * c + h;
                        // buffer chunk & 1 was last read by the store two chunks back
                        const uint32_t buf = stage + (chunk & 1) * kStageBoxBytes;
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            const int i = h * 16 + v4 * 4;
                            uint4 o4;
                            o4.x = __float_as_uint(__uint_as_float(r[i]) * inv);
                            o4.y = __float_as_uint(__uint_as_float(r[i + 1]) * inv);
                            o4.z = __float_as_uint(__uint_as_float(r[i + 2]) * inv);
                            o4.w = __float_as_uint(__uint_as_float(r[i + 3]) * inv);
                            st_shared_v4(buf + lane * 64 + ((v4 ^ ((lane >> 1) & 3)) << 4), o4);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            // rows at or past T_q fall outside the tensor, not written
                            tma_store_3d(&tmap_o, buf, chunk * 16, row0_g + quad * 32,
                                         w.b * p.H_q + head_g);
                            bulk_commit_group();
                        }
                    }
                }
                if (valid)
                    p.lse[orow] = lb_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
                tt += ng;
                ++itg;
                continue;
            }
            const float inv = 1.f / lb_run;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tc::tmem_ld32(lane_base + col_o + c * 32, r);
                tc::tmem_wait_ld();
                // buffer c & 1 was last read by the store two chunks back
                const uint32_t buf = stage + (c & 1) * kStageBoxBytes;
                if (lane == 0) bulk_wait_group_read<1>();
                __syncwarp();
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                    uint4 o4;
                    o4.x = pack_bf16x2(__uint_as_float(r[v4 * 8 + 0]) * inv,
                                       __uint_as_float(r[v4 * 8 + 1]) * inv);
                    o4.y = pack_bf16x2(__uint_as_float(r[v4 * 8 + 2]) * inv,
                                       __uint_as_float(r[v4 * 8 + 3]) * inv);
                    o4.z = pack_bf16x2(__uint_as_float(r[v4 * 8 + 4]) * inv,
                                       __uint_as_float(r[v4 * 8 + 5]) * inv);
                    o4.w = pack_bf16x2(__uint_as_float(r[v4 * 8 + 6]) * inv,
                                       __uint_as_float(r[v4 * 8 + 7]) * inv);
                    st_shared_v4(buf + lane * 64 + ((v4 ^ ((lane >> 1) & 3)) << 4), o4);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    // rows at or past T_q fall outside the tensor and are not written
                    tma_store_3d(&tmap_o, buf, c * 32, row0_g + quad * 32, w.b * p.H_q + head_g);
                    bulk_commit_group();
                }
            }
            if (valid && p.lse) p.lse[orow] = (m_run + __log2f(l_run)) * kLn2;
            tt += ng;
            if constexpr (kGen) ++itg;
        }
        // the O stores finish before the CTA (and its shared memory) does
        if (lane == 0) bulk_wait_group_all();
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

int check_args(const void* q, const void* k, const void* v, const void* o, int B, int H_q,
               int H_kv, int d, int T_q, int S_kv, int q_offset, float scale) {
    if (!q || !k || !v || !o) return GQA_ERR_INVALID_ARG;
    if (B < 0 || B > 65535 || H_q <= 0 || H_kv <= 0 || T_q < 0 || S_kv < 1 || q_offset < 0)
        return GQA_ERR_INVALID_ARG;
    // scale > 0: the kernels take each row's maximum over the raw scores and
    // scale it, which is the maximum of the scaled scores only for scale > 0
    if (H_q % H_kv != 0 || !isfinite(scale) || !(scale > 0.f)) return GQA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GQA_ERR_UNSUPPORTED;
    if (int64_t(B) * H_q * T_q >= (int64_t(1) << 31) ||
        int64_t(B) * H_kv * S_kv >= (int64_t(1) << 31))
        return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return GQA_ERR_MISALIGNED;
    return GQA_OK;
}

// One launch of the pair kernel for head dim D; function attributes once per
// device.
template <bool kBlocks, int D, bool kPartial>
int launch_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                const CUtensorMap& to, const Params& prm, const PrefillSched& sched, int ctas,
                cudaStream_t stream) {
    auto kern = prefill_pair_kernel<kBlocks, D, kPartial>;
    static std::atomic<uint64_t> attr_done{0};
    const int dev = current_device();
    if (device_attrs_pending(attr_done, dev)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PairGeo<D>::kSmemBytes) != cudaSuccess)
            return GQA_ERR_CUDA;
        device_attrs_mark(attr_done, dev);
    }
    kern<<<dim3(unsigned(ctas)), kPairThreads, PairGeo<D>::kSmemBytes, stream>>>(tq, tk, tv, to,
                                                                                prm, sched);
    return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

// The work order of a launch (plan_prefill_order), cached per shape: a
// model's layers repeat a few shapes, and the plan sorts every item. The
// kernel parameter is copied at launch, so a plan only has to outlive the
// launch call.
std::shared_ptr<const PrefillSched> work_order(int B, int H_q, int H_kv, int d, int T_q,
                                               int S_kv, int q_offset, bool causal, bool partial,
                                               int ctas, int64_t items) {
    // (no make_shared: its type tag is a process-unique symbol that the
    // dynamic linker would merge across libraries)
    static const std::shared_ptr<const PrefillSched> closed_form(new PrefillSched{});
    const int64_t budget = prefill_order_budget();
    const int64_t groups = int64_t(B) * H_kv, group_bytes = int64_t(S_kv) * d * 4;
    if (budget <= 0 || group_bytes * groups <= budget || items > kPrefillSchedItems ||
        ctas > kPrefillSchedCtas)
        return closed_form;
    using Key = std::array<int64_t, 12>;
    const Key key{B, H_q, H_kv, d, T_q, S_kv, q_offset, causal, partial, ctas, items, budget};
    static std::mutex mu;
    static std::vector<std::pair<Key, std::shared_ptr<const PrefillSched>>> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const auto& e : cache)
            if (e.first == key) return e.second;
    }
    std::shared_ptr<PrefillSched> s(new PrefillSched{});
    if (!plan_prefill_order(*s, B, H_q, H_kv, d, T_q, S_kv, q_offset, causal, partial, ctas,
                            items, budget))
        return closed_form;
    std::shared_ptr<const PrefillSched> plan(std::move(s));
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() >= 16) cache.erase(cache.begin());  // oldest first
    cache.emplace_back(key, plan);
    return plan;
}

// Both entry points: queries at global positions q_offset + t against keys
// at key_offset + j (key_offset = 0 for a whole cache); o32 set: the fp32
// partial output of one slice.
int run(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, float* o32,
        float* lse, int B, int H_q, int H_kv, int d, int T_q, int S_kv, int q_offset,
        int key_offset, int causal, float scale, cudaStream_t stream) {
    const bool partial = o32 != nullptr;
    unsigned* status = status_word();
    if (!status) return GQA_ERR_CUDA;
    CUtensorMap tq, tk, tv, to;
    if (encode_tmap_3d_bf16(&tq, q, d, T_q, uint64_t(B) * H_q, 64, BM,
                            CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
        encode_tmap_3d_bf16(&tk, k, d, S_kv, uint64_t(B) * H_kv, 64, BN,
                            CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
        encode_tmap_3d_bf16(&tv, v, d, S_kv, uint64_t(B) * H_kv, 64, BN,
                            CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
        return GQA_ERR_CUDA;
    Params prm{};
    prm.o = o;
    prm.o32 = o32;
    prm.lse = lse;
    prm.status = status;
    prm.B = B;
    prm.H_q = H_q;
    prm.H_kv = H_kv;
    prm.G = H_q / H_kv;
    prm.T_q = T_q;
    prm.S_kv = S_kv;
    // the kernels see the queries' offset relative to the first key (may be
    // negative for a slice that starts past some queries)
    prm.q_offset = causal ? q_offset - key_offset : 0;
    prm.causal = causal ? 1 : 0;
    prm.n_mblocks = (T_q + BM - 1) / BM;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.inject_timeout = take_injected_timeout() ? 1 : 0;
    // Even group sizes pair two heads of a KV group per work item; odd ones pair
    // two consecutive query blocks of one head.
    const bool blocks = prm.G % 2 != 0;
    const int64_t items = blocks ? int64_t((prm.n_mblocks + 1) / 2) * B * H_q
                                 : int64_t(prm.n_mblocks) * B * (H_q / 2);
    if (items > 0x7fffffff) return GQA_ERR_UNSUPPORTED;
    // persistent: one CTA per SM (at most one per work item)
    const int sms = num_sms();
    if (sms <= 0) return GQA_ERR_CUDA;
    const int ctas = int(items < int64_t(sms) ? items : int64_t(sms));
    const std::shared_ptr<const PrefillSched> sched =
        work_order(B, H_q, H_kv, d, T_q, S_kv, prm.q_offset, causal != 0, partial, ctas, items);
    if (!sched) return GQA_ERR_CUDA;
    const PrefillSched& ord = *sched;
    if (partial) {  // fp32 O: boxes of 16 columns x 32 rows (64 B rows, as bf16's 32 columns)
        const uint64_t od[3] = {uint64_t(d), uint64_t(T_q), uint64_t(B) * H_q};
        const uint32_t ob[3] = {16, 32, 1};
        if (encode_tmap(&to, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 3, o32, od, ob,
                        CU_TENSOR_MAP_SWIZZLE_64B) != cudaSuccess)
            return GQA_ERR_CUDA;
        if (d == 128)
            return blocks ? launch_pair<true, 128, true>(tq, tk, tv, to, prm, ord, ctas, stream)
                          : launch_pair<false, 128, true>(tq, tk, tv, to, prm, ord, ctas, stream);
        return blocks ? launch_pair<true, 64, true>(tq, tk, tv, to, prm, ord, ctas, stream)
                      : launch_pair<false, 64, true>(tq, tk, tv, to, prm, ord, ctas, stream);
    }
    if (encode_tmap_3d_bf16(&to, o, d, T_q, uint64_t(B) * H_q, 32, 32,
                            CU_TENSOR_MAP_SWIZZLE_64B) != cudaSuccess)
        return GQA_ERR_CUDA;
    if (d == 128)
        return blocks ? launch_pair<true, 128, false>(tq, tk, tv, to, prm, ord, ctas, stream)
                      : launch_pair<false, 128, false>(tq, tk, tv, to, prm, ord, ctas, stream);
    return blocks ? launch_pair<true, 64, false>(tq, tk, tv, to, prm, ord, ctas, stream)
                  : launch_pair<false, 64, false>(tq, tk, tv, to, prm, ord, ctas, stream);
}

}  // namespace prefill
}  // namespace gqa

using namespace gqa;

extern "C" int gqa_attn_prefill_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   uint16_t* o, float* lse, int B, int H_q, int H_kv, int d,
                                   int T_q, int S_kv, int q_offset, int causal, float scale,
                                   cudaStream_t stream) {
    int rc = prefill::check_args(q, k, v, o, B, H_q, H_kv, d, T_q, S_kv, q_offset, scale);
    if (rc != GQA_OK) return rc;
    if (causal && int64_t(q_offset) + T_q > S_kv) return GQA_ERR_INVALID_ARG;
    if (B == 0 || T_q == 0) return GQA_OK;
    return prefill::run(q, k, v, o, nullptr, lse, B, H_q, H_kv, d, T_q, S_kv, q_offset, 0,
                        causal, scale, stream);
}

extern "C" int gqa_attn_prefill_partial(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                        float* o_part, float* lse_part, int B, int H_q, int H_kv,
                                        int d, int T_q, int S_kv, int q_offset, int key_offset,
                                        int causal, float scale, cudaStream_t stream) {
    if (!lse_part || (reinterpret_cast<uintptr_t>(lse_part) & 3u) || key_offset < 0)
        return GQA_ERR_INVALID_ARG;
    int rc = prefill::check_args(q, k, v, o_part, B, H_q, H_kv, d, T_q, S_kv, q_offset, scale);
    if (rc != GQA_OK) return rc;
    if (B == 0 || T_q == 0) return GQA_OK;
    return prefill::run(q, k, v, nullptr, o_part, lse_part, B, H_q, H_kv, d, T_q, S_kv, q_offset,
                        key_offset, causal, scale, stream);
}

extern "C" int gqa_attn_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                uint16_t* o, float* lse, int B, int T_q, int S_kv, int q_offset,
                                int causal, float scale, cudaStream_t stream) {
    return gqa_attn_prefill_ex(q, k, v, o, lse, B, 64, 8, 128, T_q, S_kv, q_offset, causal,
                               scale, stream);
}

extern "C" int gqa_attn_debug_tile_counts(int64_t* counts, int clear) {
#ifdef GQA_DEBUG
    if (!counts) return GQA_ERR_INVALID_ARG;
    unsigned long long c[3] = {0, 0, 0};
    if (cudaDeviceSynchronize() != cudaSuccess) return GQA_ERR_CUDA;
    if (cudaMemcpyFromSymbol(c, gqa::prefill::g_dbg_tiles, sizeof(c)) != cudaSuccess)
        return GQA_ERR_CUDA;
    for (int i = 0; i < 3; ++i) counts[i] = int64_t(c[i]);
    if (clear) {
        const unsigned long long z[3] = {0, 0, 0};
        if (cudaMemcpyToSymbol(gqa::prefill::g_dbg_tiles, z, sizeof(z)) != cudaSuccess)
            return GQA_ERR_CUDA;
    }
    return GQA_OK;
#else
    (void)counts;
    (void)clear;
    return GQA_ERR_UNSUPPORTED;
#endif
}

#ifdef GQA_TRACE
extern "C" GQA_API int gqa_attn_trace_dump_prefill(void* host, size_t bytes, int clear) {
    if (bytes > sizeof(gqa::g_trace)) bytes = sizeof(gqa::g_trace);
    if (cudaDeviceSynchronize() != cudaSuccess) return GQA_ERR_CUDA;
    if (cudaMemcpyFromSymbol(host, gqa::g_trace, bytes) != cudaSuccess) return GQA_ERR_CUDA;
    if (clear) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, gqa::g_trace) != cudaSuccess) return GQA_ERR_CUDA;
        if (cudaMemset(p, 0, sizeof(gqa::g_trace)) != cudaSuccess) return GQA_ERR_CUDA;
    }
    return GQA_OK;
}
#endif
