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
// GB300 mapping. One CTA per work item (batch, query head, 128-row query
// block), heaviest blocks first; the heads of one KV group are adjacent so
// their K/V tiles are shared through L2. Six warps:
//   warp 0   TMA producer: the Q block once, then K_j and V_j (128 keys each)
//            into a 2-stage shared-memory ring, 128-byte swizzled.
//   warp 1   owns the tensor memory (512 columns: S double buffer + O) and
//            issues tcgen05.mma from one thread: S_j = Q K_j^T (both operands
//            K-major) into S[j % 2], then O += P_{j-1} V_{j-1} (V read
//            MN-major straight from its [keys][d] layout). S_{j} is issued
//            before O += P_{j-1} V_{j-1} so the tensor core runs while the
//            softmax works on S_{j-1}.
//   warps 2-5 softmax, one query row per thread (tensor-memory lane): load the
//            S row, mask, row max, exp2, row sum, P (bf16) into shared memory
//            in the MMA's swizzled layout; rescale the O row in tensor memory
//            only when the running max grows by more than 2^8 (the exps stay
//            below 256, well inside bf16 and fp32); epilogue O / l -> bf16.
// Every wait is bounded and reports a timeout in the status word.

#include <cuda_runtime.h>
#include <math.h>

#include "gqa_attn.h"
#include "plan.cuh"
#include "ptx.cuh"
#include "runtime.cuh"
#include "tcgen05.cuh"

namespace gqa {
namespace prefill {

constexpr int BM = kPrefillBlockM;  // 128 query rows per work item
constexpr int BN = kPrefillBlockN;  // 128 keys per KV tile
constexpr int D = 128;
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr uint32_t kBoxBytes = 128 * 128;        // [128 rows][64 bf16]
constexpr uint32_t kTileBytes = 2 * kBoxBytes;   // [128 rows][128 bf16], two boxes
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKVOff = kTileBytes;                          // stage s: K, then V
constexpr uint32_t kPOff = kKVOff + kStages * 2 * kTileBytes;    // P tile
constexpr uint32_t kBarOff = kPOff + kTileBytes;
constexpr int kSmemBytes = 1024 + kBarOff + 256;
constexpr uint32_t kTmemCols = 512;  // S0 [0,128), S1 [128,256), O [256,384)
constexpr uint32_t kTmemO = 256;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units: rescale O when max grows by > 256x

enum Bar { kQFull = 0, kKVFull = 1, kKVEmpty = 3, kSFull = 5, kSFree = 7, kPFull = 9,
           kPVDone = 10, kMmaDrain = 11, kNumBars = 12 };

struct Params {
    uint16_t* o;        // [B, H_q, T_q, D]
    float* lse;         // [B, H_q, T_q] or null
    unsigned* status;
    int B, H_q, H_kv, G, T_q, S_kv, q_offset, causal, n_mblocks;
    float scale_log2;
};

__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, int x, int y,
                                         int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Sum of the two bf16 values packed in x (widening bf16 to fp32 is exact).
__device__ __forceinline__ float bf16x2_sum(uint32_t x) {
    return __uint_as_float(x << 16) + __uint_as_float(x & 0xFFFF0000u);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kNumBars * 8);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- work item: heaviest query blocks first, heads of a KV group adjacent
    const int bh_count = p.B * p.H_q;
    const int mb = p.n_mblocks - 1 - int(blockIdx.x) / bh_count;
    const int bh = int(blockIdx.x) % bh_count;
    const int b = bh / p.H_q, h = bh % p.H_q, kvh = h / p.G;
    const int m0 = mb * BM;
    const int qs = p.q_offset + m0;                          // global query positions
    const int qe = p.q_offset + min(m0 + BM, p.T_q);
    int n_tiles = (p.S_kv + BN - 1) / BN;
    if (p.causal) n_tiles = min(n_tiles, (qe - 1) / BN + 1);  // all-future tiles skipped

    if (threadIdx.x == 0) {
        mbar_init(bar(kQFull), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(kKVFull + s), 1);
            mbar_init(bar(kKVEmpty + s), 1);
            mbar_init(bar(kSFull + s), 1);
            mbar_init(bar(kSFree + s), 4);
        }
        mbar_init(bar(kPFull), 4);
        mbar_init(bar(kPVDone), 1);
        mbar_init(bar(kMmaDrain), 1);
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

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
            const uint32_t qdst = smem_u32(smem + kQOff);
            mbar_arrive_expect_tx(bar(kQFull), kTileBytes);
            for (int hh = 0; hh < 2; ++hh)
                tma_load(qdst + hh * kBoxBytes, &tmap_q, hh * 64, m0, b * p.H_q + h, bar(kQFull));
            bool alive = true;
            int issued = 0;
            for (int j = 0; j < n_tiles && alive; ++j) {
                const int s = j % kStages;
                if (j >= kStages)
                    alive = mbar_wait_bounded(bar(kKVEmpty + s), ((j / kStages) - 1) & 1, p.status);
                if (!alive) break;
                const uint32_t kdst = smem_u32(smem + kKVOff + s * 2 * kTileBytes);
                const uint32_t vdst = kdst + kTileBytes;
                mbar_arrive_expect_tx(bar(kKVFull + s), 2 * kTileBytes);
                for (int hh = 0; hh < 2; ++hh) {
                    tma_load(kdst + hh * kBoxBytes, &tmap_k, hh * 64, j * BN, b * p.H_kv + kvh,
                             bar(kKVFull + s));
                    tma_load(vdst + hh * kBoxBytes, &tmap_v, hh * 64, j * BN, b * p.H_kv + kvh,
                             bar(kKVFull + s));
                }
                issued = j + 1;
            }
            // Never leave with copies in flight into this CTA's shared memory.
            mbar_wait_bounded(bar(kQFull), 0, p.status);
            for (int j = max(0, issued - kStages); j < issued; ++j)
                mbar_wait_bounded(bar(kKVFull + j % kStages), (j / kStages) & 1, p.status);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = tc::idesc_bf16_f32(BM, BN, false);
            const uint32_t idesc_pv = tc::idesc_bf16_f32(BM, D, true);
            const uint32_t qsm = smem_u32(smem + kQOff), psm = smem_u32(smem + kPOff);
            bool alive = mbar_wait_bounded(bar(kQFull), 0, p.status);
            for (int j = 0; j <= n_tiles && alive; ++j) {
                if (j < n_tiles) {
                    const int s = j % kStages;
                    alive = mbar_wait_bounded(bar(kKVFull + s), (j / kStages) & 1, p.status);
                    if (alive && j >= 2)
                        alive = mbar_wait_bounded(bar(kSFree + (j & 1)), ((j >> 1) - 1) & 1,
                                                  p.status);
                    if (!alive) break;
                    tc::fence_after_sync();
                    const uint32_t ksm = smem_u32(smem + kKVOff + s * 2 * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                        tc::mma_ss(tmem + (j & 1) * BN, tc::sdesc_sw128(qsm + off, 16, 1024),
                                   tc::sdesc_sw128(ksm + off, 16, 1024), idesc_s, kk > 0);
                    }
                    tc::commit(bar(kSFull + (j & 1)));
                }
                if (j >= 1) {
                    const int jp = j - 1, s = jp % kStages;
                    alive = mbar_wait_bounded(bar(kPFull), jp & 1, p.status);
                    if (!alive) break;
                    tc::fence_after_sync();
                    const uint32_t vsm = smem_u32(smem + kKVOff + s * 2 * kTileBytes + kTileBytes);
#pragma unroll
                    for (int ks = 0; ks < BN / 16; ++ks) {
                        const uint32_t aoff = (ks >> 2) * kBoxBytes + (ks & 3) * 32;
                        tc::mma_ss(tmem + kTmemO, tc::sdesc_sw128(psm + aoff, 16, 1024),
                                   tc::sdesc_sw128(vsm + ks * 2048, kBoxBytes, 1024), idesc_pv,
                                   (jp > 0 || ks > 0) ? 1u : 0u);
                    }
                    tc::commit(bar(kPVDone));
                    tc::commit(bar(kKVEmpty + s));
                }
            }
            // No MMA may still be running when the tensor memory is freed.
            tc::commit(bar(kMmaDrain));
            mbar_wait_bounded(bar(kMmaDrain), 0, p.status);
        }
    } else {
        // ------------------------------------------------- softmax warpgroup
        const int quad = warp & 3;            // tensor-memory lanes 32*quad .. +31
        const int row = quad * 32 + lane;     // query row within the block
        const int qg = qs + row;              // its global position
        const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);
        uint8_t* psm = smem + kPOff;
        // l_run: sum of the fp32 probabilities (for lse); lb_run: sum of the
        // bf16-rounded probabilities the P.V MMA actually consumed, so that
        // O / lb_run is an exact convex combination of V rows.
        float m_run = -INFINITY, l_run = 0.f, lb_run = 0.f;
        bool alive = true;
        for (int j = 0; j < n_tiles && alive; ++j) {
            alive = mbar_wait_bounded(bar(kSFull + (j & 1)), (j >> 1) & 1, p.status);
            alive = __all_sync(0xffffffffu, alive);
            if (!alive) break;
            tc::fence_after_sync();
            float sv[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tc::tmem_ld32(lane_base + (j & 1) * BN + c * 32, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(r[i]);
            }
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kSFree + (j & 1)));  // S buffer may be rewritten

            // scale into log2 units, mask the boundary tile, row max
            const int ks = j * BN, ke = min(ks + BN, p.S_kv);
            const bool masked =
                (p.causal && tile_class(qs, qe, ks, ke) == kTilePartial) || (ke - ks < BN);
            float mx = -INFINITY;
            if (masked) {
                const int lim = p.causal ? min(qg, p.S_kv - 1) : p.S_kv - 1;
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    sv[c] = (ks + c <= lim) ? sv[c] * p.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, sv[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    sv[c] *= p.scale_log2;
                    mx = fmaxf(mx, sv[c]);
                }
            }
            const float m_new = fmaxf(m_run, mx);
            const bool need = m_new > m_run + kRescaleThreshold;  // true while m_run = -inf
            const float corr = need ? fast_exp2(m_run - m_new) : 1.f;
            const float m_use = need ? m_new : m_run;
            float rs = 0.f;
#pragma unroll
            for (int c = 0; c < BN; ++c) {
                sv[c] = fast_exp2(sv[c] - m_use);
                rs += sv[c];
            }
            l_run = l_run * corr + rs;
            lb_run *= corr;
            m_run = m_use;

            // P and O are free once the previous tile's P.V has completed.
            if (j >= 1) {
                alive = mbar_wait_bounded(bar(kPVDone), (j - 1) & 1, p.status);
                alive = __all_sync(0xffffffffu, alive);
                if (!alive) break;
                tc::fence_after_sync();
                if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tc::tmem_ld32(lane_base + kTmemO + c * 32, r);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
                        tc::tmem_st32(lane_base + kTmemO + c * 32, r);
                    }
                    tc::tmem_wait_st();
                }
            }
            // P row -> shared memory, bf16, in the 128-byte swizzled K-major layout
            float rsb = 0.f;
#pragma unroll
            for (int c16 = 0; c16 < BN / 8; ++c16) {
                uint4 v;
                v.x = pack_bf16x2(sv[c16 * 8 + 0], sv[c16 * 8 + 1]);
                v.y = pack_bf16x2(sv[c16 * 8 + 2], sv[c16 * 8 + 3]);
                v.z = pack_bf16x2(sv[c16 * 8 + 4], sv[c16 * 8 + 5]);
                v.w = pack_bf16x2(sv[c16 * 8 + 6], sv[c16 * 8 + 7]);
                rsb += bf16x2_sum(v.x) + bf16x2_sum(v.y) + bf16x2_sum(v.z) + bf16x2_sum(v.w);
                *reinterpret_cast<uint4*>(psm + (c16 >> 3) * kBoxBytes + swz128(row, c16 & 7)) = v;
            }
            lb_run += rsb;
            fence_proxy_async_smem();  // generic-proxy writes -> the MMA's async proxy
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kPFull));
        }

        // ---- epilogue: O / l -> bf16, lse = (m + log2 l) * ln 2
        if (alive) alive = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kPVDone),
                                                                      (n_tiles - 1) & 1, p.status));
        if (alive) {
            tc::fence_after_sync();
            const bool valid = m0 + row < p.T_q;
            const float inv = 1.f / lb_run;
            const size_t orow = (size_t(b) * p.H_q + h) * p.T_q + m0 + row;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tc::tmem_ld32(lane_base + kTmemO + c * 32, r);
                tc::tmem_wait_ld();
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(p.o + orow * D + c * 32);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(r[v4 * 8 + 0]) * inv,
                                          __uint_as_float(r[v4 * 8 + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(r[v4 * 8 + 2]) * inv,
                                          __uint_as_float(r[v4 * 8 + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(r[v4 * 8 + 4]) * inv,
                                          __uint_as_float(r[v4 * 8 + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(r[v4 * 8 + 6]) * inv,
                                          __uint_as_float(r[v4 * 8 + 7]) * inv);
                        dst[v4] = w;
                    }
                }
            }
            if (valid && p.lse) p.lse[orow] = (m_run + __log2f(l_run)) * kLn2;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

int check_args(const void* q, const void* k, const void* v, const void* o, int B, int H_q,
               int H_kv, int d, int T_q, int S_kv, int q_offset, int causal, float scale) {
    if (!q || !k || !v || !o) return GQA_ERR_INVALID_ARG;
    if (B < 0 || B > 65535 || H_q <= 0 || H_kv <= 0 || T_q < 0 || S_kv < 1 || q_offset < 0)
        return GQA_ERR_INVALID_ARG;
    if (H_q % H_kv != 0 || !isfinite(scale)) return GQA_ERR_INVALID_ARG;
    if (causal && int64_t(q_offset) + T_q > S_kv) return GQA_ERR_INVALID_ARG;
    if (d != D) return GQA_ERR_UNSUPPORTED;
    if (int64_t(B) * H_q * T_q >= (int64_t(1) << 31) ||
        int64_t(B) * H_kv * S_kv >= (int64_t(1) << 31))
        return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return GQA_ERR_MISALIGNED;
    return GQA_OK;
}

}  // namespace prefill
}  // namespace gqa

using namespace gqa;

extern "C" int gqa_attn_prefill_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   uint16_t* o, float* lse, int B, int H_q, int H_kv, int d,
                                   int T_q, int S_kv, int q_offset, int causal, float scale,
                                   cudaStream_t stream) {
    using namespace gqa::prefill;
    int rc = check_args(q, k, v, o, B, H_q, H_kv, d, T_q, S_kv, q_offset, causal, scale);
    if (rc != GQA_OK) return rc;
    if (B == 0 || T_q == 0) return GQA_OK;
    unsigned* status = status_word();
    if (!status) return GQA_ERR_CUDA;
    CUtensorMap tq, tk, tv;
    if (encode_tmap_3d_bf16(&tq, q, D, T_q, uint64_t(B) * H_q, 64, BM,
                            CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
        encode_tmap_3d_bf16(&tk, k, D, S_kv, uint64_t(B) * H_kv, 64, BN,
                            CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
        encode_tmap_3d_bf16(&tv, v, D, S_kv, uint64_t(B) * H_kv, 64, BN,
                            CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
        return GQA_ERR_CUDA;
    Params prm{};
    prm.o = o;
    prm.lse = lse;
    prm.status = status;
    prm.B = B;
    prm.H_q = H_q;
    prm.H_kv = H_kv;
    prm.G = H_q / H_kv;
    prm.T_q = T_q;
    prm.S_kv = S_kv;
    prm.q_offset = causal ? q_offset : 0;
    prm.causal = causal ? 1 : 0;
    prm.n_mblocks = (T_q + BM - 1) / BM;
    prm.scale_log2 = scale * 1.4426950408889634f;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess)
            return GQA_ERR_CUDA;
        attr_set = true;
    }
    const int64_t items = int64_t(prm.n_mblocks) * B * H_q;
    if (items > 0x7fffffff) return GQA_ERR_UNSUPPORTED;
    prefill_kernel<<<dim3(unsigned(items)), kThreads, kSmemBytes, stream>>>(tq, tk, tv, prm);
    if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    return GQA_OK;
}

extern "C" int gqa_attn_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                uint16_t* o, float* lse, int B, int T_q, int S_kv, int q_offset,
                                int causal, float scale, cudaStream_t stream) {
    return gqa_attn_prefill_ex(q, k, v, o, lse, B, 64, 8, 128, T_q, S_kv, q_offset, causal,
                               scale, stream);
}
