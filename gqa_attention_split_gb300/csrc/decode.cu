// Split-KV GQA decode for sm_103a: a KV-bandwidth-bound sweep over key
// splits, merged with the log-sum-exp rule in two levels.
//
// Page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)".
//   §5.2 decode, no SP: T_q = 1, the G query heads of one KV head are folded
//        into the matmul M dimension, so every K/V tile is read from HBM once
//        for all G heads; only the ragged tail is masked.
//   §3 per-tile op sequence: S_j = q_g K_j^T * scale, m_new = max(m, rowmax),
//        P = exp(S_j - m_new), corr = exp(m - m_new), l = l*corr + rowsum P,
//        O = O*corr + P V_j.
//   §4 reduction: partials (m, l, O) merge with the log-sum-exp rule as a
//        2-level reduce-to-root (level 2 inside a CUBE, level 1 across the
//        CUBE group), normalised once at the root.
//
// GB300 mapping.
// * One CTA per (split, KV head, batch row). Each warp owns a ring of STAGES
//   shared-memory stages of TILE_T keys of K and V, filled by TMA with
//   128-byte swizzle (bank-conflict-free ldmatrix). Warps take the split's
//   tiles round-robin.
// * Tensor cores run "swapped": S^T = K_j q^T (M = 16 keys, N = 8 query heads)
//   and O^T += V_j^T P^T (M = 16 dims, N = 8 heads), so the 8 heads of a group
//   fill the N = 8 side of mma.m16n8k16 (a group of 9-16 heads runs as two
//   CTAs over the same K/V tiles); movmatrix turns the P^T accumulator
//   into the B operand. Exponentials run in base 2 with log2(e)*scale folded
//   into the scores.
// * Level 2 of the reduction: the warps of a CTA merge in shared memory, then
//   the CS CTAs of a thread-block cluster (consecutive splits of one KV head)
//   store one record per head into the shared memory of that head's owner
//   CTA (distributed shared memory), a cluster barrier makes the records
//   visible, and the owner folds them in cluster-rank order. If one cluster
//   spans the whole row it writes O and lse directly.
// * Level 1 (only when a row spans several clusters): each cluster writes a
//   partial to the workspace and a PDL-launched combine kernel merges them in
//   group order.
// * A split's last, ragged tile is loaded shifted back to end at the split's
//   last key, so every row TMA brings in is a real cache entry of this row or
//   zero fill; keys outside the tile's own range are masked by selection
//   (-inf), never by arithmetic on padding.
// All merges use a fixed order, so results are bitwise deterministic.

#include <cuda_runtime.h>
#include <stdint.h>
#include <math.h>

#include <atomic>
#include <type_traits>

#include "gqa_attn.h"
#include "plan.cuh"
#include "ptx.cuh"
#include "runtime.cuh"
#include "trace.cuh"

namespace gqa {
namespace decode {

constexpr int kMaxG = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

#ifndef GQA_DEC_WARM_TILES
#define GQA_DEC_WARM_TILES 3  // tiles per warp warmed in L2 before griddepcontrol.wait
#endif

struct SplitParams {
    const uint16_t* q;        // [B, H_q, D]
    const int32_t* seqlens;   // [B] or null
    uint16_t* o;              // [B, H_q, D]   (written when n_groups == 1)
    float* o32;               // [B, H_q, D] fp32 instead of o (partial decode), or null
    float* lse;               // [B, H_q] or null
    float* part_o;            // [B, H_q, n_groups, D]  unnormalised group partials
    float* part_m;            // [B, H_q, n_groups]     base-2 running max
    float* part_l;            // [B, H_q, n_groups]
    unsigned* status;
    int B, H_q, H_kv, G, S_max, ns, L, n_groups;
    int hgroups;              // CTAs per (split, KV head): 1, or 2 when G > 8 (heads in groups of 8)
    float scale_log2;         // scale * log2(e)
    int inject_timeout;       // test hook: block (0,0,0) withholds its first copy
    int trace_row0;           // first timeline row of this launch (trace builds only)
    int warm_l2;              // the grid fits in one wave: warm L2 before griddepcontrol.wait
    int ring;                 // ring-buffer cache: a row longer than S_max keeps S_max slots
};

// Q8: the cache holds int8 codes, K token-major [S][D] and V dim-major
// [D][S], with one fp32 scale per token for each (see gqa_attn_decode_q8).
// Q4: int4 codes, two per byte, K token-major [S][D/2] and V dim-major
// [D][S/2], scales as Q8 (see gqa_attn_decode_q4).
template <int D, int TILE_T, int STAGES, int WARPS, bool Q8 = false, bool Q4 = false>
struct SplitCfg {
    static constexpr bool kQuant = Q8 || Q4;
    static constexpr int kThreads = WARPS * 32;
    static constexpr int kBoxes = D / 64;               // bf16: 128-byte column boxes per row
    static constexpr int kBoxBytes = TILE_T * 128;      // bf16: one box, TILE_T rows x 128 B
    static constexpr int kKBytes = Q4   ? TILE_T * D / 2
                                   : Q8 ? TILE_T * D
                                        : kBoxes * kBoxBytes;  // K part of a stage
    static constexpr int kVBytes = kKBytes;  // V (or V^T) part: the same size
    static constexpr int kStageBytes = kKBytes + kVBytes;
    static constexpr int kRingBytes = WARPS * STAGES * kStageBytes;
    // int8 / int4: per-token scales of K and V for every stage, [WARPS][STAGES][2][TILE_T]
    static constexpr int kScaleOffset = kRingBytes;
    static constexpr int kScaleBytes = kQuant ? WARPS * STAGES * 2 * TILE_T * 4 : 0;
    static constexpr int kTxBytes = kStageBytes + (kQuant ? 2 * TILE_T * 4 : 0);  // per stage
    // Per-head record a CTA sends to the head's owner in the cluster:
    // {m, l, 0, 0, O[0..D)} as floats (16 + 4*D bytes, a multiple of 16).
    static constexpr int kRec = 4 + D;
    static constexpr int kRecBytes = kRec * 4;
    static constexpr int kWarpMergeFloats = (WARPS - 1) * (D / 16 * 4 + 4) * 32;
    static constexpr int kMergeBytes = kWarpMergeFloats * 4;
    static constexpr int kDataBytes = kRingBytes + kScaleBytes > kMergeBytes
                                          ? kRingBytes + kScaleBytes
                                          : kMergeBytes;
    // Inbound records: [heads per rank][CS][kRec]. A rank owns ceil(8 / CS)
    // heads, so it receives at most 16 records for any CS <= 16.
    static constexpr int kRecvOffset = kDataBytes;
    static constexpr int kRecvBytes = 2 * kMaxG * kRecBytes;
    static constexpr int kBarOffset = kRecvOffset + kRecvBytes;
    static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kBarOffset + WARPS * STAGES * 8;
    static constexpr int kMT = TILE_T / 16;             // 16-key m-tiles per stage
    static constexpr int kKC = D / 16;                  // 16-wide k-chunks of a head dim
    static_assert(TILE_T % 16 == 0 && TILE_T <= 256, "tile");
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(!Q8 || (D == 128 && (TILE_T == 32 || TILE_T == 64 || TILE_T == 128)),
                  "int8 tiles: 32, 64 or 128 tokens of a 128-dim head");
    static_assert(!Q4 || (D == 128 && TILE_T == 64 && !Q8), "int4 tiles: 64 tokens, d = 128");
    static_assert(kStageBytes % 1024 == 0, "stages stay aligned for the TMA swizzle");
};

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ int load_seqlen(const int32_t* seqlens, int b, int S_max,
                                           unsigned* status, bool report, bool ring) {
    int sl = seqlens ? seqlens[b] : S_max;
    if (ring && sl > S_max) return S_max;  // every slot of a wrapped ring is live
    if (sl < 0 || sl > S_max) {
        if (report) atomicOr(status, kStatusBadSeqlen);
        sl = sl < 0 ? 0 : S_max;
    }
    return sl;
}

__device__ __forceinline__ uint16_t to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Writes one merged (m, l, O) element: the final normalised output when the
// row has a single group, else the group's partial for the combine kernel.
__device__ __forceinline__ void emit(const SplitParams& p, size_t row, int gi, int dim, int D,
                                     float m, float l, float o) {
    if (p.n_groups == 1) {
        if (p.o32)
            p.o32[row * D + dim] = l > 0.f ? o / l : 0.f;
        else
            p.o[row * D + dim] = to_bf16_bits(l > 0.f ? o / l : 0.f);
        if (dim == 0 && p.lse) p.lse[row] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
    } else {
        const size_t pr = row * p.n_groups + gi;
        p.part_o[pr * D + dim] = o;
        if (dim == 0) {
            p.part_m[pr] = m;
            p.part_l[pr] = l;
        }
    }
}

template <int D, int TILE_T, int STAGES, int WARPS, int CS, bool Q8, bool Q4 = false>
__global__ void __launch_bounds__(WARPS * 32, 1)
    split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v,
                 const __grid_constant__ CUtensorMap tmap_ks,
                 const __grid_constant__ CUtensorMap tmap_vs, const SplitParams p) {
    using C = SplitCfg<D, TILE_T, STAGES, WARPS, Q8, Q4>;
    constexpr bool kQ = C::kQuant;  // int8 or int4 codes with per-token scales
    const int s = blockIdx.x, b = blockIdx.z;
    // KV head, and this CTA's query heads of its group: at most kMaxG, the
    // MMA's N; a larger group runs as several CTAs over the same K/V tiles
    const int kv = p.hgroups == 2 ? int(blockIdx.y >> 1) : int(blockIdx.y);  // 1 or 2 groups
    const int hsub = p.hgroups == 2 ? int(blockIdx.y & 1u) : 0;
    const int Gc = min(kMaxG, p.G - hsub * kMaxG);      // heads of this CTA
    const int head0 = kv * p.G + hsub * kMaxG;           // its first query head
    const int gi = s / CS;         // cluster (group) index within the row
    const int rank = s % CS;       // == %cluster_ctarank for a (CS, 1, 1) cluster
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;

    [[maybe_unused]] const int blin = p.trace_row0 + (b * gridDim.y + blockIdx.y) * gridDim.x + s;
    if (threadIdx.x == 0) {
        GQA_TRACE_STAMP(blin, 0);
        unsigned smid;
        asm("mov.u32 %0, %%smid;" : "=r"(smid));
        GQA_TRACE_VALUE(blin, 6, smid);
    }

    // With more than one group per row the combine kernel follows: let it be
    // scheduled now (it waits for this grid before reading anything).
    if (p.n_groups > 1) pdl_launch_dependents();

    // ---- set-up that touches no global memory: it may overlap the previous
    // kernel in the stream (programmatic dependent launch).
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset) + warp * STAGES;
    uint8_t* ring = smem + size_t(warp) * STAGES * C::kStageBytes;
    // Heads whose cluster merge this CTA owns: h = rank, rank + CS, ... < G.
    const int n_own = CS > 1 && rank < Gc ? (Gc - rank + CS - 1) / CS : 0;
    float* recv = reinterpret_cast<float*>(smem + C::kRecvOffset);  // [n_own][CS][kRec]
    if (lane == 0) {
        for (int i = 0; i < STAGES; ++i) mbar_init(smem_u32(&bars[i]), 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
        if constexpr (kQ) {
            tma_prefetch_desc(&tmap_ks);
            tma_prefetch_desc(&tmap_vs);
        }
    }
    __syncwarp();
    // Cluster barrier, phase 0: every CTA of the cluster is running before any
    // of them stores into another's shared memory (arrive now, wait later).
    if constexpr (CS > 1) cluster_arrive_release();

    // Warm L2 with this warp's first tiles while the previous kernel in
    // the stream finishes its merge (that kernel lets this grid launch once
    // its own K/V streams are done). The row length read here may be stale:
    // it only chooses what to warm, and every load below uses the length
    // read after griddepcontrol.wait.
    if (p.warm_l2 && s < p.ns) {
        int hint = p.seqlens ? *reinterpret_cast<const volatile int32_t*>(p.seqlens + b) : p.S_max;
        hint = hint < 0 ? 0 : (hint > p.S_max ? p.S_max : hint);
        const SplitRange rh = split_range(p.L, s, hint);
        // bf16 tiles start at the split's first key; int8 / int4 tiles sit
        // on TILE_T-aligned keys (see below)
        const int hbase = kQ ? rh.start - rh.start % TILE_T : rh.start;
        const int nt = rh.end > rh.start ? (rh.end - hbase + TILE_T - 1) / TILE_T : 0;
        const int mine = warp < nt ? (nt - warp + WARPS - 1) / WARPS : 0;
        constexpr int kPf = kQ ? 4 : 2 * C::kBoxes;  // the copies of one tile
        static_assert(GQA_DEC_WARM_TILES * kPf <= 32, "one lane per prefetch");
        if (lane < min(GQA_DEC_WARM_TILES, mine) * kPf) {
            const int i = lane / kPf, j = lane % kPf;
            const int tok0 = hbase + (warp + i * WARPS) * TILE_T;
            const int z = b * p.H_kv + kv;
            if constexpr (kQ) {
                if (j == 0)
                    tma_prefetch_l2_3d(&tmap_k, 0, tok0, z);
                else if (j == 1)  // int4: two tokens per byte of a V row
                    tma_prefetch_l2_3d(&tmap_v, Q4 ? tok0 / 2 : tok0, 0, z);
                else
                    tma_prefetch_l2_2d(j == 2 ? &tmap_ks : &tmap_vs, tok0, z);
            } else {
                const int y = tok0 + TILE_T <= rh.end ? tok0 : rh.end - TILE_T;
                tma_prefetch_l2_3d((j & 1) ? &tmap_v : &tmap_k, (j >> 1) * 64, y, z);
            }
        }
    }

    pdl_wait_primary();  // everything below may read what earlier kernels wrote
    if (threadIdx.x == 0) GQA_TRACE_STAMP(blin, 1);

    const int seqlen = load_seqlen(p.seqlens, b, p.S_max, p.status,
                                   s == 0 && kv == 0 && threadIdx.x == 0, p.ring != 0);
    // A whole group beyond the row's end does nothing (uniform over the
    // cluster, so no CTA waits at a cluster barrier for one that left). With a
    // single group this can only be a row of length 0: O = 0, lse = -inf.
    if (int64_t(gi) * CS * p.L >= seqlen) {
        if (p.n_groups == 1 && rank == 0) {
            for (int i = threadIdx.x; i < Gc * D; i += C::kThreads) {
                const size_t row = size_t(b) * p.H_q + head0 + i / D;
                emit(p, row, 0, i % D, D, -INFINITY, 0.f, 0.f);
            }
        }
        return;
    }
    const SplitRange r = s < p.ns ? split_range(p.L, s, seqlen) : SplitRange{seqlen, seqlen};
    const int len = r.end - r.start;
    // bf16 tiles start at r.start (the last one shifted back to end at
    // r.end, so only real rows load). int8 tiles sit on TILE_T-aligned keys
    // (a TMA box of the dim-major V codes must start on a 16-byte boundary);
    // keys of a tile outside [r.start, r.end) are masked, and padding codes are
    // finite, so no P = 0 row can turn into NaN.
    const int base = kQ ? r.start - r.start % TILE_T : r.start;
    const int n_tiles = len > 0 ? (r.end - base + TILE_T - 1) / TILE_T : 0;
    const int my_n = warp < n_tiles ? (n_tiles - warp + WARPS - 1) / WARPS : 0;
    const int zc = b * p.H_kv + kv;  // outer TMA coordinate: (batch, KV head)

    const uint64_t policy = l2_policy_evict_first();
    // Row of the first key TMA brings in for this warp's i-th tile.
    auto tile_y = [&](int i) {
        const int tok0 = r.start + (warp + i * WARPS) * TILE_T;
        return tok0 + TILE_T <= r.end ? tok0 : r.end - TILE_T;
    };
    float* scales = reinterpret_cast<float*>(smem + C::kScaleOffset);  // int8 only
    // A bf16 stage is 2 * kBoxes copies (K and V, 64 columns each); an int8
    // or int4 stage is K codes, V codes, K scales, V scales. Lane 0 arms the
    // stage's barrier, then each copy goes out from its own lane.
    constexpr int kCopies = kQ ? 4 : 2 * C::kBoxes;
    static_assert(STAGES * kCopies <= 32, "one lane per copy of the first stages");
    auto copy = [&](int i, int j) {
        const int slot = i % STAGES;
        const uint32_t bar = smem_u32(&bars[slot]);
        const uint32_t stage = smem_u32(ring + slot * C::kStageBytes);
        if constexpr (kQ) {
            const int t0 = base + (warp + i * WARPS) * TILE_T;
            if (j == 0)
                tma_load_3d(stage, &tmap_k, 0, t0, zc, bar, policy);
            else if (j == 1)  // int4: the V row's x coordinate is in bytes, t0 / 2
                tma_load_3d(stage + C::kKBytes, &tmap_v, Q4 ? t0 / 2 : t0, 0, zc, bar, policy);
            else
                tma_load_2d(smem_u32(scales + ((warp * STAGES + slot) * 2 + (j - 2)) * TILE_T),
                            j == 2 ? &tmap_ks : &tmap_vs, t0, zc, bar, policy);
        } else {  // K or V (j & 1), box j >> 1
            tma_load_3d(stage + (j & 1) * C::kKBytes + (j >> 1) * C::kBoxBytes,
                        (j & 1) ? &tmap_v : &tmap_k, (j >> 1) * 64, tile_y(i), zc, bar, policy);
        }
    };
    auto issue = [&](int i) {  // the whole warp
        if (lane == 0) mbar_arrive_expect_tx(smem_u32(&bars[i % STAGES]), C::kTxBytes);
        __syncwarp();
        if (lane < kCopies) copy(i, lane);
    };

    // Test hook: the first block withholds its first copy, so its first wait
    // runs out and reports kStatusTimeout (nothing faults, nothing hangs).
    const bool withhold = p.inject_timeout && s == 0 && kv == 0 && b == 0 && warp == 0;
    const int issued0 = min(STAGES, my_n);
    if (lane == 0)
        for (int i = withhold ? 1 : 0; i < issued0; ++i)
            mbar_arrive_expect_tx(smem_u32(&bars[i]), C::kTxBytes);
    __syncwarp();
    if (lane < issued0 * kCopies && !(withhold && lane < kCopies)) copy(lane / kCopies, lane % kCopies);
    int issued = issued0;
    bool triggered = false;

    // q^T as the B operand (k = head dim, n = query head g of this group).
    // int8: f16 pairs, with the head dims in the order the K words are read
    // (k step kc of lane c takes dims 32c + 4kc .. +3; see the S MMA below).
    // int4: k step kc of lane c takes dims 32c + 8(kc/2) + 2(kc%2) + {0, 4}
    // (first pair) and + {1, 5} (second pair, divided by 16: those K codes
    // come out of nib_pair_hi as 16 x code).
    // Before the conversion each head is scaled by a power of two 2^e that puts
    // its largest |q| in [2^14, 2^15): the f16 operands then hold every bf16 bit
    // of q whatever its magnitude (unscaled, |q| > 65504 would overflow f16 and
    // tiny q would fall into its subnormals). 2^-e comes off with the K scale.
    uint32_t qf[C::kKC][2];
    // int8 / int4: this lane's share of sum_d offset_d * q'[g][d] over the f16
    // values q' the MMA sees, where offset_d is what the K code of dim d
    // carries on top of the code (see qoff below)
    float qsum = 0.f;
    [[maybe_unused]] float hs0 = p.scale_log2, hs1 = p.scale_log2;  // quantised: heads 2c, 2c+1
    {
        const bool has = g < Gc;
        const uint16_t* qh = p.q + (size_t(b) * p.H_q + head0 + (has ? g : 0)) * D;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qh);
        if constexpr (kQ) {
            uint2 w[C::kKC];  // dims 32c + 4j .. +3 in w[j]
            float amax = 0.f;
#pragma unroll
            for (int kc = 0; kc < C::kKC; ++kc) {
                w[kc] = has ? *reinterpret_cast<const uint2*>(qh + 32 * c + 4 * kc)
                            : make_uint2(0u, 0u);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(__uint_as_float(w[kc].x << 16)),
                                               fabsf(__uint_as_float(w[kc].x & 0xFFFF0000u))),
                                         fmaxf(fabsf(__uint_as_float(w[kc].y << 16)),
                                               fabsf(__uint_as_float(w[kc].y & 0xFFFF0000u)))));
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));  // head g's max |q|
            // amax in [2^(E-127), 2^(E-126)) for a normal amax with exponent field E
            const int ebits = int((__float_as_uint(amax) >> 23) & 0xffu);
            const int e = amax > 0.f ? min(max(141 - ebits, -126), 126) : 0;
            const float up = __uint_as_float(uint32_t(e + 127) << 23);    // 2^e
            const float down = __uint_as_float(uint32_t(127 - e) << 23);  // 2^-e
            if constexpr (Q8) {
#pragma unroll
                for (int kc = 0; kc < C::kKC; ++kc) {
                    qf[kc][0] = pack_f16x2(__uint_as_float(w[kc].x << 16) * up,
                                           __uint_as_float(w[kc].x & 0xFFFF0000u) * up);
                    qf[kc][1] = pack_f16x2(__uint_as_float(w[kc].y << 16) * up,
                                           __uint_as_float(w[kc].y & 0xFFFF0000u) * up);
                    const float2 f0 =
                        __half22float2(*reinterpret_cast<const __half2*>(&qf[kc][0]));
                    const float2 f1 =
                        __half22float2(*reinterpret_cast<const __half2*>(&qf[kc][1]));
                    qsum += (f0.x + f0.y) + (f1.x + f1.y);
                }
            } else {
                const float up16 = up * 0.0625f;
                // word m of the lane's dims: dims 32c + 2m (low half), 32c + 2m + 1
                auto qw = [&](int m) { return (m & 1) ? w[m >> 1].y : w[m >> 1].x; };
#pragma unroll
                for (int kc = 0; kc < C::kKC; ++kc) {
                    const uint32_t wa = qw(4 * (kc >> 1) + (kc & 1));  // dims +0, +1
                    const uint32_t wb = qw(4 * (kc >> 1) + (kc & 1) + 2);  // dims +4, +5
                    qf[kc][0] = pack_f16x2(__uint_as_float(wa << 16) * up,
                                           __uint_as_float(wb << 16) * up);
                    qf[kc][1] = pack_f16x2(__uint_as_float(wa & 0xFFFF0000u) * up16,
                                           __uint_as_float(wb & 0xFFFF0000u) * up16);
                    const float2 f0 =
                        __half22float2(*reinterpret_cast<const __half2*>(&qf[kc][0]));
                    const float2 f1 =
                        __half22float2(*reinterpret_cast<const __half2*>(&qf[kc][1]));
                    qsum += kQ4OffsetLo * (f0.x + f0.y) + kQ4OffsetHi * (f1.x + f1.y);
                }
            }
            hs0 = p.scale_log2 * __shfl_sync(0xffffffffu, down, 8 * c);      // head 2c
            hs1 = p.scale_log2 * __shfl_sync(0xffffffffu, down, 8 * c + 4);  // head 2c + 1
        } else {
#pragma unroll
            for (int kc = 0; kc < C::kKC; ++kc) {
                qf[kc][0] = has ? qrow[(kc * 16 + 2 * c) / 2] : 0u;
                qf[kc][1] = has ? qrow[(kc * 16 + 8 + 2 * c) / 2] : 0u;
            }
        }
    }

    // int8: the f16 codes are code + 1152, so the S MMA adds 1152 * sum_d q'[h][d]
    // to head h's scores (qoff, taken off before scaling) and the P.V MMA adds
    // 1152 * sum_k P'[h][k] to every dim of head h (poff, this lane's share of
    // the running sum of the f16 P' it fed the MMA; taken off at the end).
    // int4: the same with the offsets of its conversions, 1032 and 1152
    // (16 x 72) per K position and 1152 for every V value, which qsum and poff
    // already carry.
    float qoff0 = 0.f, qoff1 = 0.f, poff0 = 0.f, poff1 = 0.f;
    if constexpr (kQ) {
        constexpr float kQScale = Q8 ? kQ8Offset : 1.f;
        qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
        qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);  // lanes 4g .. 4g+3: head g
        qoff0 = kQScale * __shfl_sync(0xffffffffu, qsum, 8 * c);
        qoff1 = kQScale * __shfl_sync(0xffffffffu, qsum, 8 * c + 4);
    }
    float m0 = -INFINITY, m1 = -INFINITY;  // heads 2c, 2c+1 (base-2 domain)
    float l0 = 0.f, l1 = 0.f;               // this lane's share of the row sums
    float acc[C::kKC][4];                   // O^T: rows = dims, cols = heads
#pragma unroll
    for (int i = 0; i < C::kKC; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    bool alive = true;
    int waited = 0;
    for (int i = 0; i < my_n; ++i) {
        const int slot = i % STAGES;
        if (alive) {
            alive = mbar_wait_bounded(smem_u32(&bars[slot]), (i / STAGES) & 1, p.status);
            alive = __all_sync(0xffffffffu, alive);  // keep the warp's control flow uniform
            if (alive) waited = i + 1;                // copies observed complete so far
        }
        if (i == 0 && threadIdx.x == 0) GQA_TRACE_STAMP(blin, 2);
        if constexpr (!kQ) {
            const uint32_t kbase = smem_u32(ring + slot * C::kStageBytes);
            const uint32_t vbase = kbase + C::kKBytes;
            const int tok0 = r.start + (warp + i * WARPS) * TILE_T;
            const int y = tile_y(i);
            const int lo = tok0, hi = min(tok0 + TILE_T, r.end);

            // ---- S^T = K_j q^T  (per 16-key m-tile, accumulate over the head dim)
            float sc[C::kMT][4];
    #pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
                sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
    #pragma unroll
                for (int kc = 0; kc < C::kKC; ++kc) {
                    const int mi = lane >> 3;
                    const int row = mt * 16 + (mi & 1) * 8 + (lane & 7);
                    const int ch = kc * 2 + (mi >> 1);
                    uint32_t a[4];
                    ldmatrix_x4(a, kbase + (ch >> 3) * C::kBoxBytes + swz128(row, ch & 7));
                    mma_bf16_16816(sc[mt], a, qf[kc][0], qf[kc][1]);
                }
            }

            // ---- scale, mask (select), running max over keys for heads 2c, 2c+1
            float mx0 = -INFINITY, mx1 = -INFINITY;
    #pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
    #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int pos = y + mt * 16 + g + (e >> 1) * 8;
                    const bool ok = pos >= lo && pos < hi;
                    sc[mt][e] = ok ? sc[mt][e] * p.scale_log2 : -INFINITY;
                }
                mx0 = fmaxf(mx0, fmaxf(sc[mt][0], sc[mt][2]));
                mx1 = fmaxf(mx1, fmaxf(sc[mt][1], sc[mt][3]));
            }
    #pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: >= 1 key valid
            const float corr0 = fast_exp2(m0 - mn0), corr1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            float ps0 = 0.f, ps1 = 0.f;
    #pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
                sc[mt][0] = fast_exp2(sc[mt][0] - mn0);
                sc[mt][1] = fast_exp2(sc[mt][1] - mn1);
                sc[mt][2] = fast_exp2(sc[mt][2] - mn0);
                sc[mt][3] = fast_exp2(sc[mt][3] - mn1);
                ps0 += sc[mt][0] + sc[mt][2];
                ps1 += sc[mt][1] + sc[mt][3];
            }
            l0 = l0 * corr0 + ps0;
            l1 = l1 * corr1 + ps1;
    #pragma unroll
            for (int md = 0; md < C::kKC; ++md) {
                acc[md][0] *= corr0;
                acc[md][1] *= corr1;
                acc[md][2] *= corr0;
                acc[md][3] *= corr1;
            }

            // ---- O^T += V_j^T P^T  (k = keys, 16 per step)
    #pragma unroll
            for (int kt = 0; kt < C::kMT; ++kt) {
                const uint32_t b_lo = movmatrix_trans(pack_bf16x2(sc[kt][0], sc[kt][1]));
                const uint32_t b_hi = movmatrix_trans(pack_bf16x2(sc[kt][2], sc[kt][3]));
    #pragma unroll
                for (int md = 0; md < C::kKC; ++md) {
                    const int mi = lane >> 3;
                    const int tok = kt * 16 + (mi >> 1) * 8 + (lane & 7);
                    const int ch = md * 2 + (mi & 1);
                    uint32_t a[4];
                    ldmatrix_x4_trans(a, vbase + (ch >> 3) * C::kBoxBytes + swz128(tok, ch & 7));
                    mma_bf16_16816(acc[md], a, b_lo, b_hi);
                }
            }

        } else if constexpr (Q8) {
            // int8 codes: K rows are tokens [TILE_T][128 B] (128-byte swizzle),
            // V rows are head dims [D][TILE_T B] (64-byte swizzle). m-tile mt of
            // the MMAs takes logical key m = 2c' + h (+8) to tile key
            // 16c' + 4mt + h (+2), so that a lane's B-operand keys of the P.V
            // step in every m-tile (logical 2c, 2c+1, 2c+8, 2c+9) are codes
            // 16c + 4mt .. +3 of a V row: one 16-byte load serves all four
            // m-tiles. The sum over keys does not depend on their order. Scores
            // and P are scaled per token after the MMAs (K) and before them (V).
            static_assert(TILE_T == 64, "the key order below covers 64-token tiles");
            const uint32_t kbase = smem_u32(ring + slot * C::kStageBytes);
            const uint32_t vbase = kbase + C::kKBytes;
            const float* ksc = scales + (warp * STAGES + slot) * 2 * TILE_T;
            const float* vsc = ksc + TILE_T;
            const int tok0 = base + (warp + i * WARPS) * TILE_T;
            const int lo = max(tok0, r.start), hi = min(tok0 + TILE_T, r.end);
            const int kr0 = 16 * (g >> 1) + (g & 1);  // tile key of logical row g in m-tile 0;
                                                      // row g + 8: + 2; m-tile mt: + 4 mt

            // ---- S^T = K_j q^T: lane c reads dims [32c, 32c + 32) of its two
            // key rows (two 16-byte chunks each) and converts them to f16.
            float sc[C::kMT][4];
            bool ok[C::kMT][2];
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
                sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
                uint32_t w[2][8];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int row = 4 * mt + kr0 + 2 * rr;
#pragma unroll
                    for (int hc = 0; hc < 2; ++hc) {
                        const uint4 v4 = ld_shared_v4(kbase + row * 128 +
                                                      (((2 * c + hc) ^ (row & 7)) << 4));
                        w[rr][hc * 4 + 0] = v4.x;
                        w[rr][hc * 4 + 1] = v4.y;
                        w[rr][hc * 4 + 2] = v4.z;
                        w[rr][hc * 4 + 3] = v4.w;
                    }
                }
#pragma unroll
                for (int kc = 0; kc < C::kKC; ++kc) {
                    uint32_t a[4];
                    u8x4_to_f16x4_biased(w[0][kc], a[0], a[2]);
                    u8x4_to_f16x4_biased(w[1][kc], a[1], a[3]);
                    mma_f16_16816(sc[mt], a, qf[kc][0], qf[kc][1]);
                }
            }

            // ---- scale by the token's K scale, mask (select), running max
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int key = 4 * mt + kr0 + 2 * rr;
                    const int pos = tok0 + key;
                    ok[mt][rr] = pos >= lo && pos < hi;
                    const float kq = ksc[key];  // the token's K scale
                    sc[mt][2 * rr] =
                        ok[mt][rr] ? (sc[mt][2 * rr] - qoff0) * (kq * hs0) : -INFINITY;
                    sc[mt][2 * rr + 1] =
                        ok[mt][rr] ? (sc[mt][2 * rr + 1] - qoff1) * (kq * hs1) : -INFINITY;
                }
                mx0 = fmaxf(mx0, fmaxf(sc[mt][0], sc[mt][2]));
                mx1 = fmaxf(mx1, fmaxf(sc[mt][1], sc[mt][3]));
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: >= 1 key valid
            const float corr0 = fast_exp2(m0 - mn0), corr1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
                sc[mt][0] = fast_exp2(sc[mt][0] - mn0);
                sc[mt][1] = fast_exp2(sc[mt][1] - mn1);
                sc[mt][2] = fast_exp2(sc[mt][2] - mn0);
                sc[mt][3] = fast_exp2(sc[mt][3] - mn1);
                ps0 += sc[mt][0] + sc[mt][2];
                ps1 += sc[mt][1] + sc[mt][3];
                // P times the token's V scale; a masked key gives exactly 0
                // whatever scale its (padding) slot holds
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const float f = vsc[4 * mt + kr0 + 2 * rr];
                    sc[mt][2 * rr] = ok[mt][rr] ? sc[mt][2 * rr] * f : 0.f;
                    sc[mt][2 * rr + 1] = ok[mt][rr] ? sc[mt][2 * rr + 1] * f : 0.f;
                }
            }
            l0 = l0 * corr0 + ps0;
            l1 = l1 * corr1 + ps1;
#pragma unroll
            for (int md = 0; md < C::kKC; ++md) {
                acc[md][0] *= corr0;
                acc[md][1] *= corr1;
                acc[md][2] *= corr0;
                acc[md][3] *= corr1;
            }
            // P' as the MMA will see it (f16), and its per-head sums: the V
            // codes carry the 1152 offset, removed once at the end
            uint32_t pp[C::kMT][2];
            float pv0 = 0.f, pv1 = 0.f;
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
                pp[mt][0] = pack_f16x2(sc[mt][0], sc[mt][1]);
                pp[mt][1] = pack_f16x2(sc[mt][2], sc[mt][3]);
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&pp[mt][0]));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&pp[mt][1]));
                pv0 += f0.x + f1.x;
                pv1 += f0.y + f1.y;
            }
            poff0 = poff0 * corr0 + pv0;
            poff1 = poff1 * corr1 + pv1;

            // ---- O^T += V_j^T P^T: lane (g, c) reads codes 16c .. 16c+15 of dims
            // md*16 + g and + 8 (16-byte chunk c of the 64-byte row, swizzled);
            // word mt of each is m-tile mt's operand.
            uint32_t b_lo[C::kMT], b_hi[C::kMT];
#pragma unroll
            for (int kt = 0; kt < C::kMT; ++kt) {
                b_lo[kt] = movmatrix_trans(pp[kt][0]);
                b_hi[kt] = movmatrix_trans(pp[kt][1]);
            }
#pragma unroll
            for (int md = 0; md < C::kKC; ++md) {
                const int d0 = md * 16 + g, d1 = d0 + 8;
                const uint4 v0 = ld_shared_v4(vbase + d0 * TILE_T + ((c ^ ((d0 >> 1) & 3)) << 4));
                const uint4 v1 = ld_shared_v4(vbase + d1 * TILE_T + ((c ^ ((d1 >> 1) & 3)) << 4));
                const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
                const uint32_t w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int kt = 0; kt < C::kMT; ++kt) {
                    uint32_t a[4];
                    u8x4_to_f16x4_biased(w0[kt], a[0], a[2]);
                    u8x4_to_f16x4_biased(w1[kt], a[1], a[3]);
                    mma_f16_16816(acc[md], a, b_lo[kt], b_hi[kt]);
                }
            }
        } else {
            // int4 codes, two per byte (the lower token or dim in the low
            // nibble): K rows are tokens [TILE_T][64 B], V rows are head dims
            // [D][32 B], both unswizzled. m-tile mt of the MMAs takes logical key
            // m = 2c' + h (+8) from tile key 16c' + mt + 4h (+8): then a lane's
            // P.V operand keys (logical 2c, 2c+1, 2c+8, 2c+9) in m-tile mt are
            // nibbles mt and mt + 4 of the two words holding keys 16c .. 16c+15
            // of a V row, one 8-byte load per dim row for all four m-tiles.
            // Every V nibble is shifted to bits 4-7 and read by nib_pair_hi as
            // 1152 + 16 x code, so P is divided by 16 throughout: the offset the
            // P.V sums carry is then 72 per code step, near the int8 path's
            // ratio, where nib_pair_lo's 1032 per step would leave too little
            // of the result once the fp32 sums over thousands of keys cancel it.
            // The K side keeps the mixed form: its offset is one constant per
            // head and key row, and what its rounding leaves is nearly the same
            // for every key of a row, which the softmax takes out.
            static_assert(TILE_T == 64, "the key order below covers 64-token tiles");
            const uint32_t kbase = smem_u32(ring + slot * C::kStageBytes);
            const uint32_t vbase = kbase + C::kKBytes;
            const float* ksc = scales + (warp * STAGES + slot) * 2 * TILE_T;
            const float* vsc = ksc + TILE_T;
            const int tok0 = base + (warp + i * WARPS) * TILE_T;
            const int lo = max(tok0, r.start), hi = min(tok0 + TILE_T, r.end);
            const int kr0 = 16 * (g >> 1) + 4 * (g & 1);  // tile key of logical row g in
                                                          // m-tile 0; row g + 8: + 8;
                                                          // m-tile mt: + mt

            // ---- S^T = K_j q^T: lane c reads dims [32c, 32c + 32) of its two
            // key rows (one 16-byte chunk each); k step kc takes word kc / 2,
            // shifted by 8 for odd kc.
            float sc[C::kMT][4];
            bool ok[C::kMT][2];
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
                sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
                const uint4 r0 = ld_shared_v4(kbase + (kr0 + mt) * 64 + c * 16);
                const uint4 r1 = ld_shared_v4(kbase + (kr0 + mt + 8) * 64 + c * 16);
                const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w};
                const uint32_t w1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
                for (int kc = 0; kc < C::kKC; ++kc) {
                    const int sh = (kc & 1) * 8;
                    const uint32_t x0 = w0[kc >> 1] >> sh, x1 = w1[kc >> 1] >> sh;
                    const uint32_t a[4] = {nib_pair_lo(x0), nib_pair_lo(x1), nib_pair_hi(x0),
                                           nib_pair_hi(x1)};
                    mma_f16_16816(sc[mt], a, qf[kc][0], qf[kc][1]);
                }
            }

            // ---- scale by the token's K scale, mask (select), running max
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int key = kr0 + mt + 8 * rr;
                    const int pos = tok0 + key;
                    ok[mt][rr] = pos >= lo && pos < hi;
                    const float kq = ksc[key];  // the token's K scale
                    sc[mt][2 * rr] =
                        ok[mt][rr] ? (sc[mt][2 * rr] - qoff0) * (kq * hs0) : -INFINITY;
                    sc[mt][2 * rr + 1] =
                        ok[mt][rr] ? (sc[mt][2 * rr + 1] - qoff1) * (kq * hs1) : -INFINITY;
                }
                mx0 = fmaxf(mx0, fmaxf(sc[mt][0], sc[mt][2]));
                mx1 = fmaxf(mx1, fmaxf(sc[mt][1], sc[mt][3]));
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: >= 1 key valid
            const float corr0 = fast_exp2(m0 - mn0), corr1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
                sc[mt][0] = fast_exp2(sc[mt][0] - mn0);
                sc[mt][1] = fast_exp2(sc[mt][1] - mn1);
                sc[mt][2] = fast_exp2(sc[mt][2] - mn0);
                sc[mt][3] = fast_exp2(sc[mt][3] - mn1);
                ps0 += sc[mt][0] + sc[mt][2];
                ps1 += sc[mt][1] + sc[mt][3];
                // P times the token's V scale and 1/16; a masked key gives
                // exactly 0 whatever scale its slot holds
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const float f = vsc[kr0 + mt + 8 * rr] * 0.0625f;
                    sc[mt][2 * rr] = ok[mt][rr] ? sc[mt][2 * rr] * f : 0.f;
                    sc[mt][2 * rr + 1] = ok[mt][rr] ? sc[mt][2 * rr + 1] * f : 0.f;
                }
            }
            l0 = l0 * corr0 + ps0;
            l1 = l1 * corr1 + ps1;
#pragma unroll
            for (int md = 0; md < C::kKC; ++md) {
                acc[md][0] *= corr0;
                acc[md][1] *= corr1;
                acc[md][2] *= corr0;
                acc[md][3] *= corr1;
            }
            // P' as the MMA will see it (f16), and its per-head sums times the
            // 1152 offset of every V value, removed at the end
            uint32_t pp[C::kMT][2];
            float pv0 = 0.f, pv1 = 0.f;
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
                pp[mt][0] = pack_f16x2(sc[mt][0], sc[mt][1]);
                pp[mt][1] = pack_f16x2(sc[mt][2], sc[mt][3]);
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&pp[mt][0]));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&pp[mt][1]));
                pv0 += f0.x + f1.x;
                pv1 += f0.y + f1.y;
            }
            pv0 *= kQ4OffsetHi;
            pv1 *= kQ4OffsetHi;
            poff0 = poff0 * corr0 + pv0;
            poff1 = poff1 * corr1 + pv1;

            // ---- O^T += V_j^T P^T: lane (g, c) reads keys 16c .. 16c+15 of
            // dims md*16 + g and + 8 (8 bytes each); m-tile kt takes nibbles
            // kt, kt + 4 of each word (low word: keys 16c .. +7, high word:
            // keys 16c + 8 .. +15), moved to bits 4-7 and 20-23 first.
            uint32_t b_lo[C::kMT], b_hi[C::kMT];
#pragma unroll
            for (int kt = 0; kt < C::kMT; ++kt) {
                b_lo[kt] = movmatrix_trans(pp[kt][0]);
                b_hi[kt] = movmatrix_trans(pp[kt][1]);
            }
#pragma unroll
            for (int md = 0; md < C::kKC; ++md) {
                const int d0 = md * 16 + g, d1 = d0 + 8;
                const uint2 v0 = ld_shared_v2(vbase + d0 * (TILE_T / 2) + c * 8);
                const uint2 v1 = ld_shared_v2(vbase + d1 * (TILE_T / 2) + c * 8);
#pragma unroll
                for (int kt = 0; kt < C::kMT; ++kt) {
                    auto at4 = [&](uint32_t u) {  // nibbles kt, kt + 4 -> bits 4-7, 20-23
                        return kt == 0 ? u << 4 : u >> (4 * (kt - 1));
                    };
                    const uint32_t a[4] = {nib_pair_hi(at4(v0.x)), nib_pair_hi(at4(v1.x)),
                                           nib_pair_hi(at4(v0.y)), nib_pair_hi(at4(v1.y))};
                    mma_f16_16816(acc[md], a, b_lo[kt], b_hi[kt]);
                }
            }
        }

        __syncwarp();
        if (alive && issued < my_n) issue(issued);
        if (alive && issued < my_n) ++issued;
        // The warp's last K/V copy is issued: the next kernel in the stream may
        // launch now and warm L2 behind the copies still in flight (it reads
        // nothing this grid writes before its griddepcontrol.wait). GB300,
        // 8K decode: 8.80-8.83 us per call in an 80-layer graph against
        // 9.04-9.07 with the trigger after the stream; 9-call graphs lose
        // ~1.5% (9.17-9.20 against 9.02-9.06 us).
        if (p.n_groups == 1 && !triggered && issued == my_n) {
            pdl_launch_dependents();
            triggered = true;
        }
    }
    // A wait that ran out may leave copies in flight: wait for them (bounded)
    // before the shared memory is reused or released. A withheld copy was
    // never issued, so there is nothing of it to wait for.
    for (int i = waited; i < issued; ++i)
        if (!(withhold && i == 0))
            mbar_wait_bounded(smem_u32(&bars[i % STAGES]), (i / STAGES) & 1, p.status);

#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    if constexpr (kQ) {
        constexpr float kPScale = Q8 ? kQ8Offset : 1.f;  // int4's sums carry their offsets
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            poff0 += __shfl_xor_sync(0xffffffffu, poff0, off);
            poff1 += __shfl_xor_sync(0xffffffffu, poff1, off);
        }
#pragma unroll
        for (int md = 0; md < C::kKC; ++md) {
            acc[md][0] -= kPScale * poff0;
            acc[md][1] -= kPScale * poff1;
            acc[md][2] -= kPScale * poff0;
            acc[md][3] -= kPScale * poff1;
        }
    }
    if (threadIdx.x == 0) GQA_TRACE_STAMP(blin, 3);
    // A warp without tiles (or whose wait ran out) lets the next kernel
    // launch here. A combine kernel that follows was allowed to launch at the
    // start.
    if (p.n_groups == 1 && !triggered) pdl_launch_dependents();

    // ---- level 2a: the other warps hand their partials to warp 0, which
    // merges them fragment by fragment in registers (warp order fixed).
    constexpr int kFrag = C::kKC * 4 + 4;  // accumulators, then m0, m1, l0, l1
    float* wbuf = reinterpret_cast<float*>(smem);  // [WARPS-1][kFrag][32]
    if constexpr (CS > 1) cluster_wait_acquire();  // phase 0 (long complete by now)
    __syncthreads();  // every warp is done with its ring
    if (warp > 0) {
        float* dst = wbuf + (warp - 1) * kFrag * 32 + lane;
#pragma unroll
        for (int md = 0; md < C::kKC; ++md)
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[(md * 4 + e) * 32] = acc[md][e];
        dst[(C::kKC * 4 + 0) * 32] = m0;
        dst[(C::kKC * 4 + 1) * 32] = m1;
        dst[(C::kKC * 4 + 2) * 32] = l0;
        dst[(C::kKC * 4 + 3) * 32] = l1;
    }
    __syncthreads();
    if (warp == 0) {
        float ms0 = m0, ms1 = m1;
#pragma unroll
        for (int w = 1; w < WARPS; ++w) {
            const float* src = wbuf + (w - 1) * kFrag * 32 + lane;
            ms0 = fmaxf(ms0, src[(C::kKC * 4 + 0) * 32]);
            ms1 = fmaxf(ms1, src[(C::kKC * 4 + 1) * 32]);
        }
        // An empty CTA keeps (-inf, 0, 0); -inf - -inf never reaches exp2.
        auto weight = [](float m, float mstar) {
            return m == -INFINITY ? 0.f : fast_exp2(m - mstar);
        };
        const float f0 = weight(m0, ms0), f1 = weight(m1, ms1);
        l0 *= f0;
        l1 *= f1;
#pragma unroll
        for (int md = 0; md < C::kKC; ++md) {
            acc[md][0] *= f0;
            acc[md][1] *= f1;
            acc[md][2] *= f0;
            acc[md][3] *= f1;
        }
#pragma unroll
        for (int w = 1; w < WARPS; ++w) {
            const float* src = wbuf + (w - 1) * kFrag * 32 + lane;
            const float g0 = weight(src[(C::kKC * 4 + 0) * 32], ms0);
            const float g1 = weight(src[(C::kKC * 4 + 1) * 32], ms1);
            l0 += g0 * src[(C::kKC * 4 + 2) * 32];
            l1 += g1 * src[(C::kKC * 4 + 3) * 32];
#pragma unroll
            for (int md = 0; md < C::kKC; ++md) {
                acc[md][0] += g0 * src[(md * 4 + 0) * 32];
                acc[md][1] += g1 * src[(md * 4 + 1) * 32];
                acc[md][2] += g0 * src[(md * 4 + 2) * 32];
                acc[md][3] += g1 * src[(md * 4 + 3) * 32];
            }
        }
        // Warp 0 now holds the CTA partial: lane (g, c) has heads 2c, 2c+1 at
        // dims md*16 + g (+8). Without a cluster it is the result (or this
        // split's partial). With one, each head's record {m, l, 0, 0, O[D]}
        // goes straight from registers into slot [h / CS][rank] of the head's
        // owner, rank h % CS, as plain distributed-shared-memory stores.
        uint32_t rbase[2] = {0u, 0u};
        if constexpr (CS > 1) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = 2 * c + e;
                rbase[e] = map_to_rank(smem_u32(recv + ((h / CS) * CS + rank) * C::kRec),
                                       uint32_t(h % CS));
            }
        }
#pragma unroll
        for (int md = 0; md < C::kKC; ++md) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int dim = md * 16 + g + (e >> 1) * 8;
                const int head = 2 * c + (e & 1);
                const float mm = (e & 1) ? ms1 : ms0, ll = (e & 1) ? l1 : l0;
                if (head < Gc) {
                    if constexpr (CS == 1)
                        emit(p, size_t(b) * p.H_q + head0 + head, gi, dim, D, mm, ll,
                             acc[md][e]);
                    else
                        st_dsmem(rbase[e & 1] + (4 + dim) * 4, acc[md][e]);
                }
            }
        }
        if (CS > 1 && g == 0) {
            if (2 * c < Gc) {
                st_dsmem(rbase[0] + 0, ms0);
                st_dsmem(rbase[0] + 4, l0);
            }
            if (2 * c + 1 < Gc) {
                st_dsmem(rbase[1] + 0, ms1);
                st_dsmem(rbase[1] + 4, l1);
            }
        }
    }

    if constexpr (CS > 1) {
        // ---- level 2b. Cluster barrier, phase 1: each thread's stores are
        // released by its arrive and acquired by every wait, so all records
        // are in their owners' shared memory. No CTA touches another's shared
        // memory after this point, so none can outlive a store aimed at it.
        cluster_arrive_release();
        cluster_wait_acquire();
        if (threadIdx.x == 0) GQA_TRACE_STAMP(blin, 4);
        // Per owned head, warp 0 alone: lane q holds sender q's (m, l), the
        // weights come from two warp reductions, and each lane folds the CS
        // records over its D/32 dims with vector loads (rank order fixed).
        if (warp == 0) {
            constexpr int kPer = D / 32;
            using VecT = typename std::conditional<kPer == 4, float4, float2>::type;
            for (int j = 0; j < n_own; ++j) {
                const float* r0 = recv + j * CS * C::kRec;
                const float mq = lane < CS ? r0[lane * C::kRec + 0] : -INFINITY;
                const float lq = lane < CS ? r0[lane * C::kRec + 1] : 0.f;
                const float mstar = warp_max(mq);
                const float f = mq == -INFINITY ? 0.f : fast_exp2(mq - mstar);
                const float lsum = warp_sum(f * lq);
                float o[kPer];
#pragma unroll
                for (int e = 0; e < kPer; ++e) o[e] = 0.f;
#pragma unroll
                for (int q2 = 0; q2 < CS; ++q2) {
                    const VecT v =
                        *reinterpret_cast<const VecT*>(r0 + q2 * C::kRec + 4 + lane * kPer);
                    const float fq = __shfl_sync(0xffffffffu, f, q2);
                    const float* fv = reinterpret_cast<const float*>(&v);
#pragma unroll
                    for (int e = 0; e < kPer; ++e) o[e] += fq * fv[e];
                }
                const size_t row = size_t(b) * p.H_q + head0 + rank + j * CS;
#pragma unroll
                for (int e = 0; e < kPer; ++e) emit(p, row, gi, lane * kPer + e, D, mstar, lsum, o[e]);
            }
        }
    }
    if (threadIdx.x == 0) GQA_TRACE_STAMP(blin, 5);
}

struct CombineParams {
    const float* part_o;
    const float* part_m;
    const float* part_l;
    const int32_t* seqlens;
    uint16_t* o;
    float* o32;  // fp32 output instead of o (partial decode), or null
    float* lse;
    int B, H_q, S_max, n_groups;
    int64_t group_len;  // keys per group: cluster size * L
};

constexpr int kCombineWarps = 8;
[[maybe_unused]] constexpr int kTraceCombineBase = 60000;  // trace rows of combine blocks

// Level 1 of the reduction. One warp per (batch, query head): merge the row's
// non-empty group partials with the log-sum-exp rule, normalise once, write O
// and lse. Lane j holds group j's (m, l); the O partials of up to 8 groups are
// loaded together so one L2 round trip serves them. The arithmetic order
// depends only on the group count: results are deterministic.
template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const CombineParams p) {
    constexpr int kPer = D / 32;  // dims per lane
    using VecT = typename std::conditional<kPer == 4, float4, float2>::type;
    if (threadIdx.x == 0) GQA_TRACE_STAMP(kTraceCombineBase + blockIdx.x, 0);
    pdl_launch_dependents();      // the next kernel may start its own set-up
    pdl_wait_primary();           // the split grid's partials are complete and visible
    if (threadIdx.x == 0) GQA_TRACE_STAMP(kTraceCombineBase + blockIdx.x, 1);
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (row >= p.B * p.H_q) return;
    const int b = row / p.H_q;
    int seqlen = p.seqlens ? p.seqlens[b] : p.S_max;
    seqlen = seqlen < 0 ? 0 : (seqlen > p.S_max ? p.S_max : seqlen);
    const int n_act = int((seqlen + p.group_len - 1) / p.group_len);
    float* out_lse = p.lse ? p.lse + row : nullptr;
    uint16_t* out = p.o32 ? nullptr : p.o + size_t(row) * D + lane * kPer;
    float* out32 = p.o32 ? p.o32 + size_t(row) * D + lane * kPer : nullptr;
    if (n_act == 0) {
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (out32)
                out32[j] = 0.f;
            else
                out[j] = 0;
        }
        if (lane == 0 && out_lse) *out_lse = -INFINITY;
        return;
    }
    const float* pm = p.part_m + size_t(row) * p.n_groups;
    const float* pl = p.part_l + size_t(row) * p.n_groups;
    const float* po = p.part_o + size_t(row) * p.n_groups * D + lane * kPer;
    float mx = -INFINITY;
    for (int s = lane; s < n_act; s += 32) mx = fmaxf(mx, pm[s]);
    mx = warp_max(mx);
    float lpart = 0.f;
    float acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
    for (int base = 0; base < n_act; base += 32) {
        const int cnt = min(32, n_act - base);
        float w = 0.f;
        if (lane < cnt) {
            w = fast_exp2(pm[base + lane] - mx);
            lpart += w * pl[base + lane];
        }
        for (int j = 0; j < cnt; j += 8) {
            VecT v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (j + u < cnt) v[u] = *reinterpret_cast<const VecT*>(po + size_t(base + j + u) * D);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float ww = __shfl_sync(0xffffffffu, w, (j + u) & 31);
                if (j + u < cnt) {
                    const float* f = reinterpret_cast<const float*>(&v[u]);
#pragma unroll
                    for (int e = 0; e < kPer; ++e) acc[e] += ww * f[e];
                }
            }
        }
    }
    const float lsum = warp_sum(lpart);
    const float inv = 1.f / lsum;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (out32)
            out32[j] = acc[j] * inv;
        else
            out[j] = to_bf16_bits(acc[j] * inv);
    }
    if (lane == 0 && out_lse) *out_lse = (mx + __log2f(lsum)) * kLn2;
    if (threadIdx.x == 0) GQA_TRACE_STAMP(kTraceCombineBase + blockIdx.x, 2);
}

// ------------------------------------------------------------------ host side

#ifndef GQA_DEC_TILE_T
#define GQA_DEC_TILE_T 32
#endif
#ifndef GQA_DEC_STAGES
#define GQA_DEC_STAGES 3
#endif
#ifndef GQA_DEC_WARPS
#define GQA_DEC_WARPS 2
#endif
constexpr int kTileT = GQA_DEC_TILE_T, kStages = GQA_DEC_STAGES, kWarps = GQA_DEC_WARPS;
// int8 caches: 64 tokens per stage; the warps x stages per CTA are chosen in
// launch() below.
constexpr int kTileTQ8 = 64;
// int4 caches: 64 tokens per stage (8 KB of codes + 512 B of scales), 4 warps x
// 2 stages per CTA on one-wave and longer grids alike (GB300: 8K decode 9.35 us,
// ragged 128K 80.4 us; 4 x 3: 9.39 / 81.3; 3 x 3 on the long grid: 99.7; 2 x 4:
// 10.3 / 80.4; 6 x 2 and 8 x 1, at one CTA per SM: 15-16 / 125-134)
constexpr int kTileTQ4 = 64;
#ifndef GQA_DEC_Q4_WARPS
#define GQA_DEC_Q4_WARPS 4
#endif
#ifndef GQA_DEC_Q4_STAGES
#define GQA_DEC_Q4_STAGES 2
#endif
#ifndef GQA_DEC_Q4_WARPS_MW
#define GQA_DEC_Q4_WARPS_MW 4
#endif
#ifndef GQA_DEC_Q4_STAGES_MW
#define GQA_DEC_Q4_STAGES_MW 2
#endif
constexpr int kQ4WarpsOneWave = GQA_DEC_Q4_WARPS, kQ4StagesOneWave = GQA_DEC_Q4_STAGES;
constexpr int kQ4Warps = GQA_DEC_Q4_WARPS_MW, kQ4Stages = GQA_DEC_Q4_STAGES_MW;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// CTAs of a decode launch: one per (split, KV head, batch row), times the
// groups of at most kMaxG query heads a KV head's group splits into.
// num_splits = 0: the plan `pick` (gqa_attn_pick_num_splits or its INT8 / INT4
// forms). A bf16 group of more than 8 query heads runs as two CTAs per split
// and KV head that read the same keys: the plan for 2 * H_kv heads (the CTAs
// the launch has) is taken when it is one wave of splits of at most 1024 keys,
// else the plan for H_kv heads (GB300, 128/8 heads at 8K: B = 1 12.7 us with
// 8 splits against 14.6 with 16; B = 2 18.5 us with 8 against 21.8 with 4,
// where the shared reads make the SMs' intake the bound). Returns the split
// count, or a negative error code.
int auto_splits(int (*pick)(int, int, int, int), int B, int H_q, int H_kv, int S_max) {
    const int sms = num_sms();
    if (sms <= 0) return GQA_ERR_CUDA;
    int ns = -1;
    if (H_q / H_kv > kMaxG && pick == gqa_attn_pick_num_splits) {
        const int ns2 = pick(B, 2 * H_kv, S_max, sms);
        if (ns2 >= 1 && int64_t(B) * 2 * H_kv * ns2 <= sms &&
            (int64_t(S_max) + ns2 - 1) / ns2 <= 1024)
            ns = ns2;
    }
    if (ns < 1) ns = pick(B, H_kv, S_max, sms);
    return ns < 1 ? GQA_ERR_INVALID_ARG : ns;
}

int64_t grid_ctas(int ns, int B, int H_q, int H_kv) {
    const int G = H_q / H_kv;
    return int64_t(ns) * H_kv * B * ((G + kMaxG - 1) / kMaxG);
}

// Cluster size of a launch on this device (the rule is decode_cluster_size in
// plan.cuh; ragged 128K decode on GB300: 141 us with clusters of 16, 132 us
// with 8).
int cluster_size_for(int ns, int64_t ctas) { return decode_cluster_size(ns, ctas, num_sms()); }
// The multi-wave choice: its clusters are never larger, so its workspace is
// never smaller.
int max_groups_cluster_size(int ns) { return decode_cluster_size(ns, INT64_MAX, 1); }

struct WsLayout {
    size_t o_off, m_off, l_off, total;
};

WsLayout ws_layout(int B, int H_q, int d, int ns, int cs) {
    WsLayout w{};
    const int groups = ns / cs;
    if (groups <= 1) return w;
    const size_t rows = size_t(B) * H_q * groups;
    w.o_off = 0;
    w.m_off = align256(rows * d * sizeof(float));
    w.l_off = w.m_off + align256(rows * sizeof(float));
    w.total = w.l_off + align256(rows * sizeof(float));
    return w;
}

// Workspace bytes of a launch on this device (0 when one cluster covers a row).
size_t launch_ws_bytes(int B, int H_q, int H_kv, int d, int ns) {
    return ws_layout(B, H_q, d, ns, cluster_size_for(ns, grid_ctas(ns, B, H_q, H_kv))).total;
}

// Cache formats of a launch: bf16 K/V, int8 codes, int4 codes.
enum Kind { kBf16 = 0, kInt8 = 1, kInt4 = 2 };

// maps: K, V (bf16) or K codes, V codes, K scales, V scales (int8, int4).
template <int D, int CS, int KIND, int kW = kWarps, int kS = kStages>
int launch_split(const SplitParams& sp, const CUtensorMap (&maps)[4], cudaStream_t stream) {
    constexpr bool kQ8 = KIND == kInt8, kQ4 = KIND == kInt4;
    constexpr int kT = kQ8 ? kTileTQ8 : kQ4 ? kTileTQ4 : kTileT;
    using C = SplitCfg<D, kT, kS, kW, kQ8, kQ4>;
    auto kern = split_kernel<D, kT, kS, kW, CS, kQ8, kQ4>;
    // once per device (a race only sets them twice, which is harmless)
    static std::atomic<uint64_t> attr_done{0};
    const int dev = current_device();
    if (device_attrs_pending(attr_done, dev)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) !=
                cudaSuccess)
            return GQA_ERR_CUDA;
        if (CS > 8 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess)
            return GQA_ERR_CUDA;
        device_attrs_mark(attr_done, dev);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sp.ns, sp.H_kv * sp.hgroups, sp.B);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    // Programmatic dependent launch: this grid may start while the previous
    // kernel in the stream finishes; it reads no global memory before
    // griddepcontrol.wait.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CS;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CS > 1 ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], sp) != cudaSuccess)
        return GQA_ERR_CUDA;
    return GQA_OK;
}

template <int D, int KIND, int kW, int kS>
int launch_cs(const SplitParams& sp, int cs, const CUtensorMap (&maps)[4], cudaStream_t stream) {
    switch (cs) {
        case 16: return launch_split<D, 16, KIND, kW, kS>(sp, maps, stream);
        case 8: return launch_split<D, 8, KIND, kW, kS>(sp, maps, stream);
        case 4: return launch_split<D, 4, KIND, kW, kS>(sp, maps, stream);
        case 2: return launch_split<D, 2, KIND, kW, kS>(sp, maps, stream);
        default: return launch_split<D, 1, KIND, kW, kS>(sp, maps, stream);
    }
}

template <int D, int KIND>
int launch(const SplitParams& sp, int cs, const CUtensorMap (&maps)[4], cudaStream_t stream) {
    int rc;
    if constexpr (KIND == kInt8)
        // one wave: 4 x 1 in clusters of 16 (the 8K single row: 8.67 us against
        // 9.34 with 2 x 3), 3 x 2 in smaller clusters (the small-batch plans,
        // whose CTAs walk more tiles) and in longer grids (ragged 128K batch:
        // 86-88 us)
        rc = sp.warm_l2 ? (cs <= 8 ? launch_cs<D, kInt8, 3, 2>(sp, cs, maps, stream)
                                   : launch_cs<D, kInt8, 4, 1>(sp, cs, maps, stream))
                        : launch_cs<D, kInt8, 3, 2>(sp, cs, maps, stream);
    else if constexpr (KIND == kInt4)
        rc = sp.warm_l2 ? launch_cs<D, kInt4, kQ4WarpsOneWave, kQ4StagesOneWave>(sp, cs, maps,
                                                                                 stream)
                        : launch_cs<D, kInt4, kQ4Warps, kQ4Stages>(sp, cs, maps, stream);
    else if constexpr (D == 64)
        // half-size stages: twice the warps (one wave) or the stages (longer
        // grids) keep d = 128's bytes in flight, and 4 warps per CTA hide the
        // per-tile softmax work that half the bytes per key leaves exposed
        rc = sp.warm_l2 ? launch_cs<D, kBf16, 4, kStages>(sp, cs, maps, stream)
                        : launch_cs<D, kBf16, 4, 2>(sp, cs, maps, stream);
    else
        rc = sp.warm_l2 ? launch_cs<D, kBf16, kWarps, kStages>(sp, cs, maps, stream)
                        : launch_cs<D, kBf16, 4, 1>(sp, cs, maps, stream);
    if (rc != GQA_OK || sp.n_groups == 1) return rc;

    static std::atomic<uint64_t> attr_done{0};
    const int dev = current_device();
    if (device_attrs_pending(attr_done, dev)) {
        if (cudaFuncSetAttribute(combine_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 100) != cudaSuccess)
            return GQA_ERR_CUDA;
        device_attrs_mark(attr_done, dev);
    }
    CombineParams cp{sp.part_o, sp.part_m, sp.part_l, sp.seqlens, sp.o, sp.o32, sp.lse,
                     sp.B, sp.H_q, sp.S_max, sp.n_groups, int64_t(cs) * sp.L};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((sp.B * sp.H_q + kCombineWarps - 1) / kCombineWarps);
    cfg.blockDim = dim3(kCombineWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, combine_kernel<D>, cp) != cudaSuccess) return GQA_ERR_CUDA;
    return GQA_OK;
}

int check_args(const void* q, const void* k, const void* v, const void* o, int B, int H_q,
               int H_kv, int d, int S_max, float scale, int num_splits) {
    if (!q || !k || !v || !o) return GQA_ERR_INVALID_ARG;
    if (B < 0 || B > 65535 || H_q <= 0 || H_kv <= 0 || H_kv > 65535 || S_max <= 0)
        return GQA_ERR_INVALID_ARG;
    if (H_q % H_kv != 0) return GQA_ERR_INVALID_ARG;
    if (num_splits < 0 || num_splits > 8192) return GQA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return GQA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GQA_ERR_UNSUPPORTED;
    if (H_q / H_kv > 2 * kMaxG) return GQA_ERR_UNSUPPORTED;
    if (int64_t(H_kv) * ((H_q / H_kv + kMaxG - 1) / kMaxG) > 65535) return GQA_ERR_UNSUPPORTED;
    if (int64_t(B) * H_kv * S_max > (int64_t(1) << 31)) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return GQA_ERR_MISALIGNED;
    return GQA_OK;
}


int run(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse,
        const int32_t* seqlens, int B, int H_q, int H_kv, int d, int S_max, float scale,
        int ns, void* ws, size_t ws_bytes, cudaStream_t stream, bool ring = false,
        const float* k_scales = nullptr, const float* v_scales = nullptr,
        float* o32 = nullptr, bool int4 = false) {
    // with scales, k and v are K codes and dim-major V codes: int8, or int4
    // (two per byte) when int4 is set
    const bool q8 = k_scales != nullptr && !int4;
    const bool q4 = k_scales != nullptr && int4;
    unsigned* status = status_word();
    if (!status) return GQA_ERR_CUDA;
    const int cs = cluster_size_for(ns, grid_ctas(ns, B, H_q, H_kv));
    const WsLayout wl = ws_layout(B, H_q, d, ns, cs);
    if (wl.total > 0) {
        if (!ws || ws_bytes < wl.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
            return GQA_ERR_WORKSPACE;
    }
    CUtensorMap maps[4];
    const uint64_t outer = uint64_t(B) * H_kv;
    if (q8) {
        const uint64_t kd[3] = {uint64_t(d), uint64_t(S_max), outer};  // K codes [.., S, d]
        const uint32_t kb[3] = {uint32_t(d), kTileTQ8, 1};
        const uint64_t vd[3] = {uint64_t(S_max), uint64_t(d), outer};  // V codes [.., d, S]
        const uint32_t vb[3] = {kTileTQ8, uint32_t(d), 1};
        const uint64_t sd[2] = {uint64_t(S_max), outer};                // scales [.., S]
        const uint32_t sb[2] = {kTileTQ8, 1};
        if (encode_tmap(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 3, k, kd, kb,
                        CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
            encode_tmap(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 3, v, vd, vb,
                        kTileTQ8 == 32   ? CU_TENSOR_MAP_SWIZZLE_32B
                        : kTileTQ8 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                         : CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
            encode_tmap(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2, k_scales, sd, sb,
                        CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess ||
            encode_tmap(&maps[3], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2, v_scales, sd, sb,
                        CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess)
            return GQA_ERR_CUDA;
    } else if (q4) {
        const uint64_t kd[3] = {uint64_t(d) / 2, uint64_t(S_max), outer};  // K codes [.., S, d/2]
        const uint32_t kb[3] = {uint32_t(d) / 2, kTileTQ4, 1};
        const uint64_t vd[3] = {uint64_t(S_max) / 2, uint64_t(d), outer};  // V codes [.., d, S/2]
        const uint32_t vb[3] = {kTileTQ4 / 2, uint32_t(d), 1};
        const uint64_t sd[2] = {uint64_t(S_max), outer};                    // scales [.., S]
        const uint32_t sb[2] = {kTileTQ4, 1};
        if (encode_tmap(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 3, k, kd, kb,
                        CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess ||
            encode_tmap(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 3, v, vd, vb,
                        CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess ||
            encode_tmap(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2, k_scales, sd, sb,
                        CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess ||
            encode_tmap(&maps[3], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 2, v_scales, sd, sb,
                        CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess)
            return GQA_ERR_CUDA;
    } else {
        if (encode_tmap_3d_bf16(&maps[0], k, d, S_max, outer, 64, kTileT,
                                CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
            encode_tmap_3d_bf16(&maps[1], v, d, S_max, outer, 64, kTileT,
                                CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
            return GQA_ERR_CUDA;
        maps[2] = maps[0];  // unused by the bf16 kernels
        maps[3] = maps[1];
    }
    SplitParams sp{};
    sp.q = q;
    sp.seqlens = seqlens;
    sp.o = o;
    sp.o32 = o32;
    sp.lse = lse;
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    const bool parts = wl.total > 0;
    sp.part_o = parts ? reinterpret_cast<float*>(w8 + wl.o_off) : nullptr;
    sp.part_m = parts ? reinterpret_cast<float*>(w8 + wl.m_off) : nullptr;
    sp.part_l = parts ? reinterpret_cast<float*>(w8 + wl.l_off) : nullptr;
    sp.status = status;
    sp.B = B;
    sp.H_q = H_q;
    sp.H_kv = H_kv;
    sp.G = H_q / H_kv;
    sp.hgroups = (sp.G + kMaxG - 1) / kMaxG;
    sp.S_max = S_max;
    sp.ns = ns;
    sp.L = split_len(S_max, ns);
    sp.n_groups = ns / cs;
    sp.warm_l2 = grid_ctas(ns, B, H_q, H_kv) <= num_sms() ? 1 : 0;  // a single wave
    sp.ring = ring ? 1 : 0;
    sp.scale_log2 = scale * kLog2e;
    sp.inject_timeout = take_injected_timeout() ? 1 : 0;
#ifdef GQA_TRACE
    static int trace_row = 0;  // consecutive launches get consecutive timeline rows
    const int nctas = int(grid_ctas(ns, B, H_q, H_kv));
    if (trace_row + nctas > kTraceCombineBase) trace_row = 0;
    sp.trace_row0 = trace_row;
    trace_row += nctas;
#endif
    if (q8) return launch<128, kInt8>(sp, cs, maps, stream);
    if (q4) return launch<128, kInt4>(sp, cs, maps, stream);
    return d == 128 ? launch<128, kBf16>(sp, cs, maps, stream)
                    : launch<64, kBf16>(sp, cs, maps, stream);
}

}  // namespace decode
}  // namespace gqa

using namespace gqa;

extern "C" int gqa_attn_debug_inject_timeout(int launches) {
    if (launches < 0) return GQA_ERR_INVALID_ARG;
    set_injected_timeouts(launches);
    return GQA_OK;
}

extern "C" size_t gqa_attn_decode_workspace_size(int B, int H_q, int d, int num_splits) {
    if (B < 0 || H_q <= 0 || (d != 64 && d != 128) || num_splits <= 0) return 0;
    return decode::ws_layout(B, H_q, d, num_splits, decode::max_groups_cluster_size(num_splits))
        .total;
}

extern "C" int gqa_attn_decode_ws(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  uint16_t* o, float* lse, const int32_t* seqlens, int B,
                                  int H_q, int H_kv, int d, int S_max, float scale,
                                  int num_splits, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
    int rc = decode::check_args(q, k, v, o, B, H_q, H_kv, d, S_max, scale, num_splits);
    if (rc != GQA_OK) return rc;
    if (num_splits < 1) return GQA_ERR_INVALID_ARG;
    if (B == 0) return GQA_OK;
    return decode::run(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, S_max, scale, num_splits,
                       workspace, workspace_bytes, stream);
}

extern "C" int gqa_attn_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               uint16_t* o, float* lse, const int32_t* seqlens, int B, int H_q,
                               int H_kv, int d, int S_max, float scale, int num_splits,
                               cudaStream_t stream) {
    int rc = decode::check_args(q, k, v, o, B, H_q, H_kv, d, S_max, scale, num_splits);
    if (rc != GQA_OK) return rc;
    if (B == 0) return GQA_OK;
    int ns = num_splits;
    if (ns == 0) {
        ns = decode::auto_splits(gqa_attn_pick_num_splits, B, H_q, H_kv, S_max);
        if (ns < 1) return ns;
    }
    const size_t bytes = decode::launch_ws_bytes(B, H_q, H_kv, d, ns);
    void* ws = nullptr;
    if (bytes > 0) {
        ws = stream_workspace(stream, bytes);
        if (!ws) return GQA_ERR_WORKSPACE;
    }
    return decode::run(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, S_max, scale, ns, ws, bytes,
                       stream);
}

// ---------------------------------------------------------------------------
// Sequence-parallel decode: partial results over disjoint key ranges and their
// merge.
//
// Page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)", §5.3 (decode
// with sequence parallelism: each rank sweeps its own slice of the keys) and
// §4 (the partials meet in a log-sum-exp reduce-to-root, normalised once at
// the root). Here a partial is normalised over its own keys and carried as
// (O_r fp32, lse_r); merging R of them in rank order gives
//   lse = ln sum_r exp(lse_r),  O = sum_r exp(lse_r - lse) O_r,
// which is the §4 merge with m = lse_r, l = 1.

namespace gqa {
namespace decode {

constexpr int kMergeWarps = 8;

// One warp per output row: lane r < R holds part r's lse (in chunks of 32);
// the O parts are folded in rank order with vector loads.
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts,
                 uint16_t* o, float* lse, int R, int rows) {
    constexpr int kPer = D / 32;
    using VecT = typename std::conditional<kPer == 4, float4, float2>::type;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    float mx = -INFINITY;
    for (int r = lane; r < R; r += 32) mx = fmaxf(mx, lse_parts[size_t(r) * rows + row]);
    mx = warp_max(mx);
    uint16_t* out = o + size_t(row) * D + lane * kPer;
    if (mx == -INFINITY) {  // no part saw a key
#pragma unroll
        for (int j = 0; j < kPer; ++j) out[j] = 0;
        if (lane == 0 && lse) lse[row] = -INFINITY;
        return;
    }
    float acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
    float wsum = 0.f;
    for (int base = 0; base < R; base += 32) {
        const int cnt = min(32, R - base);
        const float lr = lane < cnt ? lse_parts[size_t(base + lane) * rows + row] : -INFINITY;
        const float w = lr == -INFINITY ? 0.f : exp2f((lr - mx) * kLog2e);
        wsum += w;
        for (int r = 0; r < cnt; ++r) {
            const float wr = __shfl_sync(0xffffffffu, w, r);
            if (wr == 0.f) continue;  // an empty part (its O may hold anything)
            const VecT v = *reinterpret_cast<const VecT*>(
                o_parts + (size_t(base + r) * rows + row) * D + lane * kPer);
            const float* f = reinterpret_cast<const float*>(&v);
#pragma unroll
            for (int j = 0; j < kPer; ++j) acc[j] += wr * f[j];
        }
    }
    const float wtot = warp_sum(wsum);
    const float inv = 1.f / wtot;
#pragma unroll
    for (int j = 0; j < kPer; ++j) out[j] = to_bf16_bits(acc[j] * inv);
    if (lane == 0 && lse) lse[row] = mx + logf(wtot);
}

}  // namespace decode
}  // namespace gqa

extern "C" int gqa_attn_decode_partial(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                       float* o_part, float* lse_part, const int32_t* seqlens,
                                       int B, int H_q, int H_kv, int d, int S_max, float scale,
                                       int num_splits, cudaStream_t stream) {
    if (!lse_part || (reinterpret_cast<uintptr_t>(lse_part) & 3u)) return GQA_ERR_INVALID_ARG;
    int rc = decode::check_args(q, k, v, o_part, B, H_q, H_kv, d, S_max, scale, num_splits);
    if (rc != GQA_OK) return rc;
    if (B == 0) return GQA_OK;
    int ns = num_splits;
    if (ns == 0) {
        ns = decode::auto_splits(gqa_attn_pick_num_splits, B, H_q, H_kv, S_max);
        if (ns < 1) return ns;
    }
    const size_t bytes = decode::launch_ws_bytes(B, H_q, H_kv, d, ns);
    void* ws = nullptr;
    if (bytes > 0) {
        ws = stream_workspace(stream, bytes);
        if (!ws) return GQA_ERR_WORKSPACE;
    }
    return decode::run(q, k, v, nullptr, lse_part, seqlens, B, H_q, H_kv, d, S_max, scale, ns,
                       ws, bytes, stream, /*ring=*/false, nullptr, nullptr, o_part);
}

extern "C" int gqa_attn_merge(const float* o_parts, const float* lse_parts, uint16_t* o,
                              float* lse, int R, int rows, int d, cudaStream_t stream) {
    if (!o_parts || !lse_parts || !o || R < 1 || rows < 0) return GQA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GQA_ERR_UNSUPPORTED;
    if (int64_t(R) * rows * d >= (int64_t(1) << 40)) return GQA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(o_parts) & 15u) || (reinterpret_cast<uintptr_t>(o) & 15u) ||
        (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return GQA_ERR_MISALIGNED;
    if (rows == 0) return GQA_OK;
    const dim3 grid(unsigned((rows + decode::kMergeWarps - 1) / decode::kMergeWarps));
    if (d == 128)
        decode::merge_kernel<128><<<grid, decode::kMergeWarps * 32, 0, stream>>>(
            o_parts, lse_parts, o, lse, R, rows);
    else
        decode::merge_kernel<64><<<grid, decode::kMergeWarps * 32, 0, stream>>>(
            o_parts, lse_parts, o, lse, R, rows);
    return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Hard-capped ring-buffer KV cache with attention sinks.
//
// Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §2 item 4 (the
// cache has a fixed max_tokens) and §4 item 2 (a full ring overwrites its
// oldest entry, keeping the attention sinks). Slots [0, n_sink) hold the
// row's first n_sink tokens for good; token t >= n_sink lives in slot
// n_sink + (t - n_sink) mod (capacity - n_sink). Softmax attention does not
// depend on the order of its keys, so a decode step over such a cache is the
// split-KV decode over its live slots: the first min(seqlen, capacity).

namespace gqa {
namespace decode {

__global__ void __launch_bounds__(64)
    ring_append_kernel(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_new,
                       const uint16_t* v_new, const int32_t* positions, int H_kv, int d,
                       int capacity, int n_sink, unsigned* status) {
    const int bk = blockIdx.x;  // b * H_kv + kv
    const int t = positions[bk / H_kv];
    if (t < 0) {
        if (threadIdx.x == 0 && bk % H_kv == 0) atomicOr(status, kStatusBadSeqlen);
        return;
    }
    const int slot = t < n_sink ? t : n_sink + (t - n_sink) % (capacity - n_sink);
    const size_t dst = (size_t(bk) * capacity + slot) * d, src = size_t(bk) * d;
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {  // 16-byte chunks
        reinterpret_cast<uint4*>(k_cache + dst)[i] = reinterpret_cast<const uint4*>(k_new + src)[i];
        reinterpret_cast<uint4*>(v_cache + dst)[i] = reinterpret_cast<const uint4*>(v_new + src)[i];
    }
}

}  // namespace decode
}  // namespace gqa

extern "C" int gqa_attn_ring_append(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_new,
                                    const uint16_t* v_new, const int32_t* positions, int B,
                                    int H_kv, int d, int capacity, int n_sink,
                                    cudaStream_t stream) {
    if (!k_cache || !v_cache || !k_new || !v_new || !positions) return GQA_ERR_INVALID_ARG;
    if (B < 0 || H_kv <= 0 || capacity < 1 || n_sink < 0 || n_sink >= capacity)
        return GQA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GQA_ERR_UNSUPPORTED;
    if (int64_t(B) * H_kv >= (int64_t(1) << 31)) return GQA_ERR_UNSUPPORTED;
    for (const void* ptr : {static_cast<const void*>(k_cache), static_cast<const void*>(v_cache),
                            static_cast<const void*>(k_new), static_cast<const void*>(v_new)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return GQA_ERR_MISALIGNED;
    if (B == 0) return GQA_OK;
    unsigned* status = status_word();
    if (!status) return GQA_ERR_CUDA;
    decode::ring_append_kernel<<<dim3(unsigned(B * H_kv)), 64, 0, stream>>>(
        k_cache, v_cache, k_new, v_new, positions, H_kv, d, capacity, n_sink, status);
    return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

extern "C" int gqa_attn_decode_ring(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    uint16_t* o, float* lse, const int32_t* seqlens, int B,
                                    int H_q, int H_kv, int d, int capacity, int n_sink,
                                    float scale, int num_splits, cudaStream_t stream) {
    if (n_sink < 0 || capacity < 1 || n_sink >= capacity || !seqlens) return GQA_ERR_INVALID_ARG;
    int rc = decode::check_args(q, k, v, o, B, H_q, H_kv, d, capacity, scale, num_splits);
    if (rc != GQA_OK) return rc;
    if (B == 0) return GQA_OK;
    int ns = num_splits;
    if (ns == 0) {
        ns = decode::auto_splits(gqa_attn_pick_num_splits, B, H_q, H_kv, capacity);
        if (ns < 1) return ns;
    }
    const size_t bytes = decode::launch_ws_bytes(B, H_q, H_kv, d, ns);
    void* ws = nullptr;
    if (bytes > 0) {
        ws = stream_workspace(stream, bytes);
        if (!ws) return GQA_ERR_WORKSPACE;
    }
    return decode::run(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, capacity, scale, ns, ws, bytes,
                       stream, /*ring=*/true);
}

// ---------------------------------------------------------------------------
// INT8 KV cache.
//
// Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §4 item 3
// (optional INT4 / INT8 KV quantisation for long contexts; the page fixes no
// scheme). Each (batch row, KV head, token) of K and of V gets one fp32 scale
// max|x| / 127 and codes rint(x / scale) in [-127, 127] (ties to even; both
// divisions single IEEE fp32 divisions; an all-zero token gets scale 0 and
// codes 0), stored biased as the bytes code + 128. K codes stay token-major
// [S][d]; V codes are stored dim-major
// [d][S] so that the decode kernel's P.V operand reads four consecutive
// tokens of one dim with a single 32-bit load.

namespace gqa {
namespace decode {

constexpr int kQuantTokens = 32;  // tokens per block; one warp per token at a time

__global__ void __launch_bounds__(256)
    quantize_kv_q8_kernel(const uint16_t* k, const uint16_t* v, uint8_t* kc, uint8_t* vc,
                          float* ks, float* vs, int S) {
    __shared__ uint32_t vt[128][kQuantTokens / 4];  // V codes of this block, dim-major
    const int bh = blockIdx.y, t0 = blockIdx.x * kQuantTokens;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int tt = warp; tt < kQuantTokens; tt += 8) {
        const int t = t0 + tt;
        uint32_t vcode = 0;
        if (t < S) {
            const size_t row = size_t(bh) * S + t;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint16_t* src = (which ? v : k) + row * 128;
                const uint2 w = reinterpret_cast<const uint2*>(src)[lane];  // dims 4l .. 4l+3
                float x[4] = {__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                              __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u)};
                float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
                amax = warp_max(amax);
                const float sc = __fdiv_rn(amax, 127.f);
                uint32_t packed = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float qv = sc > 0.f ? rintf(__fdiv_rn(x[e], sc)) : 0.f;
                    qv = fminf(fmaxf(qv, -127.f), 127.f);
                    packed |= uint32_t(int(qv) + 128) << (8 * e);  // stored biased
                }
                if (which == 0) {
                    reinterpret_cast<uint32_t*>(kc + row * 128)[lane] = packed;
                    if (lane == 0) ks[row] = sc;
                } else {
                    vcode = packed;
                    if (lane == 0) vs[row] = sc;
                }
            }
        }
        // byte e of vcode is dim 4*lane + e of token tt
#pragma unroll
        for (int e = 0; e < 4; ++e)
            reinterpret_cast<uint8_t*>(&vt[4 * lane + e][0])[tt] = uint8_t(vcode >> (8 * e));
    }
    __syncthreads();
    // dim-major rows: 32 consecutive tokens of one dim per 32-byte run
    for (int i = threadIdx.x; i < 128 * (kQuantTokens / 4); i += blockDim.x) {
        const int dim = i / (kQuantTokens / 4), wd = i % (kQuantTokens / 4);
        const int t = t0 + 4 * wd;
        uint8_t* dst = vc + (size_t(bh) * 128 + dim) * S + t;
        const uint32_t word = vt[dim][wd];
        if (t + 3 < S) {
            *reinterpret_cast<uint32_t*>(dst) = word;  // S % 16 == 0, t % 4 == 0: aligned
        } else {
            for (int e = 0; e < 4 && t + e < S; ++e) dst[e] = uint8_t(word >> (8 * e));
        }
    }
}

}  // namespace decode
}  // namespace gqa

extern "C" int gqa_attn_quantize_kv_q8(const uint16_t* k, const uint16_t* v, uint8_t* k_codes,
                                       uint8_t* v_codes, float* k_scales, float* v_scales, int B,
                                       int H_kv, int S, int d, cudaStream_t stream) {
    if (!k || !v || !k_codes || !v_codes || !k_scales || !v_scales) return GQA_ERR_INVALID_ARG;
    if (B < 0 || H_kv <= 0 || S <= 0) return GQA_ERR_INVALID_ARG;
    if (d != 128 || S % 16 != 0) return GQA_ERR_UNSUPPORTED;
    if (int64_t(B) * H_kv > 65535 || int64_t(B) * H_kv * S >= (int64_t(1) << 31))
        return GQA_ERR_UNSUPPORTED;
    for (const void* ptr : {static_cast<const void*>(k), static_cast<const void*>(v),
                            static_cast<const void*>(k_codes), static_cast<const void*>(v_codes),
                            static_cast<const void*>(k_scales), static_cast<const void*>(v_scales)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return GQA_ERR_MISALIGNED;
    if (B == 0) return GQA_OK;
    const dim3 grid(unsigned((S + decode::kQuantTokens - 1) / decode::kQuantTokens),
                    unsigned(B * H_kv));
    decode::quantize_kv_q8_kernel<<<grid, 256, 0, stream>>>(k, v, k_codes, v_codes, k_scales,
                                                             v_scales, S);
    return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

extern "C" int gqa_attn_decode_q8(const uint16_t* q, const uint8_t* k_codes,
                                  const uint8_t* v_codes, const float* k_scales,
                                  const float* v_scales, uint16_t* o, float* lse,
                                  const int32_t* seqlens, int B, int H_q, int H_kv, int d,
                                  int S_max, float scale, int num_splits, cudaStream_t stream) {
    if (!k_scales || !v_scales) return GQA_ERR_INVALID_ARG;
    int rc = decode::check_args(q, k_codes, v_codes, o, B, H_q, H_kv, d, S_max, scale, num_splits);
    if (rc != GQA_OK) return rc;
    if (d != 128 || S_max % 16 != 0) return GQA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(k_scales) | reinterpret_cast<uintptr_t>(v_scales)) & 15u)
        return GQA_ERR_MISALIGNED;
    if (B == 0) return GQA_OK;
    int ns = num_splits;
    if (ns == 0) {
        ns = decode::auto_splits(gqa_attn_pick_num_splits_q8, B, H_q, H_kv, S_max);
        if (ns < 1) return ns;
    }
    const size_t bytes = decode::launch_ws_bytes(B, H_q, H_kv, d, ns);
    void* ws = nullptr;
    if (bytes > 0) {
        ws = stream_workspace(stream, bytes);
        if (!ws) return GQA_ERR_WORKSPACE;
    }
    return decode::run(q, reinterpret_cast<const uint16_t*>(k_codes),
                       reinterpret_cast<const uint16_t*>(v_codes), o, lse, seqlens, B, H_q, H_kv,
                       d, S_max, scale, ns, ws, bytes, stream, /*ring=*/false, k_scales, v_scales);
}

// ---------------------------------------------------------------------------
// INT4 KV cache: the INT8 scheme with 4-bit codes (page 3, §4 item 3). Each
// (batch row, KV head, token) of K and of V gets one fp32 scale max|x| / 7 and
// codes rint(x / scale) in [-7, 7] (ties to even; both divisions single IEEE
// fp32 divisions; an all-zero token gets scale 0 and codes 0), stored biased
// as the nibbles code + 8, two per byte with the lower dim (K) or the lower
// token (V) in the low nibble. K codes stay token-major [S][d/2]; V codes are
// dim-major [d][S/2].

namespace gqa {
namespace decode {

constexpr int kQuant4Tokens = 32;  // tokens per block; one warp per token pair at a time

__global__ void __launch_bounds__(256)
    quantize_kv_q4_kernel(const uint16_t* k, const uint16_t* v, uint8_t* kc, uint8_t* vc,
                          float* ks, float* vs, int S) {
    __shared__ __align__(16) uint8_t vt[128][kQuant4Tokens / 2];  // V codes, dim-major
    const int bh = blockIdx.y, t0 = blockIdx.x * kQuant4Tokens;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int pr = warp; pr < kQuant4Tokens / 2; pr += 8) {
        uint32_t vnib[2] = {0u, 0u};  // per token of the pair: this lane's 4 V nibbles
        for (int h = 0; h < 2; ++h) {
            const int t = t0 + 2 * pr + h;
            if (t >= S) continue;  // uniform over the warp
            const size_t row = size_t(bh) * S + t;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint16_t* src = (which ? v : k) + row * 128;
                const uint2 w = reinterpret_cast<const uint2*>(src)[lane];  // dims 4l .. 4l+3
                float x[4] = {__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                              __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u)};
                float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
                amax = warp_max(amax);
                const float sc = __fdiv_rn(amax, 7.f);
                uint32_t nib = 0;  // nibble e = dim 4l + e
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float qv = sc > 0.f ? rintf(__fdiv_rn(x[e], sc)) : 0.f;
                    qv = fminf(fmaxf(qv, -7.f), 7.f);
                    nib |= uint32_t(int(qv) + 8) << (4 * e);
                }
                if (which == 0) {
                    reinterpret_cast<uint16_t*>(kc + row * 64)[lane] = uint16_t(nib);
                    if (lane == 0) ks[row] = sc;
                } else {
                    vnib[h] = nib;
                    if (lane == 0) vs[row] = sc;
                }
            }
        }
        // byte pr of dim row 4l + e: token 2pr in the low nibble, 2pr + 1 high
#pragma unroll
        for (int e = 0; e < 4; ++e)
            vt[4 * lane + e][pr] =
                uint8_t(((vnib[0] >> (4 * e)) & 0xFu) | (((vnib[1] >> (4 * e)) & 0xFu) << 4));
    }
    __syncthreads();
    // dim-major rows: the block's 32 tokens of one dim are 16 bytes
    for (int dim = threadIdx.x; dim < 128; dim += blockDim.x) {
        const int nbytes = min(kQuant4Tokens, S - t0) / 2;  // S % 32 == 0: always 16
        uint8_t* dst = vc + (size_t(bh) * 128 + dim) * (S / 2) + t0 / 2;
        if (nbytes == kQuant4Tokens / 2)
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&vt[dim][0]);
        else
            for (int j = 0; j < nbytes; ++j) dst[j] = vt[dim][j];
    }
}

}  // namespace decode
}  // namespace gqa

extern "C" int gqa_attn_quantize_kv_q4(const uint16_t* k, const uint16_t* v, uint8_t* k_codes,
                                       uint8_t* v_codes, float* k_scales, float* v_scales, int B,
                                       int H_kv, int S, int d, cudaStream_t stream) {
    if (!k || !v || !k_codes || !v_codes || !k_scales || !v_scales) return GQA_ERR_INVALID_ARG;
    if (B < 0 || H_kv <= 0 || S <= 0) return GQA_ERR_INVALID_ARG;
    if (d != 128 || S % 32 != 0) return GQA_ERR_UNSUPPORTED;
    if (int64_t(B) * H_kv > 65535 || int64_t(B) * H_kv * S >= (int64_t(1) << 31))
        return GQA_ERR_UNSUPPORTED;
    for (const void* ptr : {static_cast<const void*>(k), static_cast<const void*>(v),
                            static_cast<const void*>(k_codes), static_cast<const void*>(v_codes),
                            static_cast<const void*>(k_scales), static_cast<const void*>(v_scales)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return GQA_ERR_MISALIGNED;
    if (B == 0) return GQA_OK;
    const dim3 grid(unsigned(S / decode::kQuant4Tokens), unsigned(B * H_kv));
    decode::quantize_kv_q4_kernel<<<grid, 256, 0, stream>>>(k, v, k_codes, v_codes, k_scales,
                                                             v_scales, S);
    return cudaGetLastError() == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

extern "C" int gqa_attn_decode_q4(const uint16_t* q, const uint8_t* k_codes,
                                  const uint8_t* v_codes, const float* k_scales,
                                  const float* v_scales, uint16_t* o, float* lse,
                                  const int32_t* seqlens, int B, int H_q, int H_kv, int d,
                                  int S_max, float scale, int num_splits, cudaStream_t stream) {
    if (!k_scales || !v_scales) return GQA_ERR_INVALID_ARG;
    int rc = decode::check_args(q, k_codes, v_codes, o, B, H_q, H_kv, d, S_max, scale, num_splits);
    if (rc != GQA_OK) return rc;
    if (d != 128 || S_max % 32 != 0) return GQA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(k_scales) | reinterpret_cast<uintptr_t>(v_scales)) & 15u)
        return GQA_ERR_MISALIGNED;
    if (B == 0) return GQA_OK;
    int ns = num_splits;
    if (ns == 0) {
        ns = decode::auto_splits(gqa_attn_pick_num_splits_q4, B, H_q, H_kv, S_max);
        if (ns < 1) return ns;
    }
    const size_t bytes = decode::launch_ws_bytes(B, H_q, H_kv, d, ns);
    void* ws = nullptr;
    if (bytes > 0) {
        ws = stream_workspace(stream, bytes);
        if (!ws) return GQA_ERR_WORKSPACE;
    }
    return decode::run(q, reinterpret_cast<const uint16_t*>(k_codes),
                       reinterpret_cast<const uint16_t*>(v_codes), o, lse, seqlens, B, H_q, H_kv,
                       d, S_max, scale, ns, ws, bytes, stream, /*ring=*/false, k_scales, v_scales,
                       /*o32=*/nullptr, /*int4=*/true);
}

#ifdef GQA_TRACE
extern "C" GQA_API int gqa_attn_trace_dump(void* host, size_t bytes, int clear) {
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

// ---------------------------------------------------------------------------
// Decode that allocates no device memory.
//
// Some callers cannot call cudaMalloc: a serving process that partitions HBM
// once at start-up and forbids later allocations, a host that routes every
// device byte through its own allocator, or a latency-critical path that
// cannot afford cudaMalloc's implicit device synchronisation. For them the
// split-KV decode above runs with the scratch of its split merge (the
// per-cluster partials) in a fixed array that lives in this library's module:
// every GPU that loads the library holds it until the process exits. The
// status word is the library's own (also module memory), so gqa_attn_check()
// reports this entry point's device errors without allocating either.

namespace gqa {
namespace decode {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static_assert(kNoAllocScratchBytes == GQA_NOALLOC_SCRATCH_BYTES, "header limit");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
static std::atomic<void*> g_noalloc_addr[kNoAllocMaxDevices];  // zero-initialised, no heap

// Looks up the device address of the array once per device (with that device
// current). In host code the array's name is a host-side stand-in, not a
// device address, so it must never be passed to a kernel directly.
static int noalloc_scratch(void** scratch) {
    const int dev = current_device();
    if (dev < 0) return GQA_ERR_CUDA;
    if (dev >= kNoAllocMaxDevices) return GQA_ERR_UNSUPPORTED;
    void* a = g_noalloc_addr[dev].load(std::memory_order_acquire);
    if (!a) {
        if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || !a) return GQA_ERR_CUDA;
        g_noalloc_addr[dev].store(a, std::memory_order_release);
    }
    *scratch = a;
    return GQA_OK;
}

}  // namespace decode
}  // namespace gqa

extern "C" int gqa_attn_decode_noalloc(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                       uint16_t* o, float* lse, const int32_t* seqlens, int B,
                                       int H_q, int H_kv, int d, int S_max, float scale,
                                       int num_splits, cudaStream_t stream) {
    using namespace gqa::decode;
    int rc = check_args(q, k, v, o, B, H_q, H_kv, d, S_max, scale, num_splits);
    if (rc != GQA_OK) return rc;
    if (B == 0) return GQA_OK;
    int ns = num_splits;
    if (ns == 0) {
        ns = decode::auto_splits(gqa_attn_pick_num_splits, B, H_q, H_kv, S_max);
        if (ns < 1) return ns;
    }
    const WsLayout wl = ws_layout(B, H_q, d, ns, cluster_size_for(ns, grid_ctas(ns, B, H_q, H_kv)));
    if (wl.total > kNoAllocScratchBytes) return GQA_ERR_WORKSPACE;
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc != GQA_OK) return rc;
    // The same path as gqa_attn_decode_ws, with the fixed array as workspace.
    return run(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, S_max, scale, ns, scratch,
               kNoAllocScratchBytes, stream);
}
