// Split-KV GQA decode for sm_103a: a KV-bandwidth-bound sweep that writes
// per-split (m, l, O) partials, and a log-sum-exp combine.
//
// Page: "ADR-0060: AHBM GQA Fused Attention kernel (Llama3-70B)".
//   §5.2 decode, no SP: T_q = 1, the G query heads of one KV head are folded
//        into the matmul M dimension, so every K/V tile is read from HBM once
//        for all G heads; only the ragged tail is masked.
//   §3 per-tile op sequence: S_j = q_g K_j^T * scale, m_new = max(m, rowmax),
//        P = exp(S_j - m_new), corr = exp(m - m_new), l = l*corr + rowsum P,
//        O = O*corr + P V_j.
//   §4 reduction: the split partials merge with the log-sum-exp rule and are
//        normalised once (here: by the combine kernel, in split order).
//
// GB300 mapping. One CTA per (split, KV head, batch row). Each warp owns an
// independent ring of STAGES shared-memory stages, each holding TILE_T keys
// of K and V, filled by TMA (128-byte swizzle, so the ldmatrix reads below
// are bank-conflict free). Warps take the split's tiles round-robin. The
// tensor-core work runs "swapped": S^T = K_j q^T (M = 16 keys, N = 8 query
// heads) and O^T += V_j^T P^T (M = 16 dims, N = 8 heads), so the 8 heads of a
// group fill the N = 8 side of mma.m16n8k16 with no padding; P^T moves from
// the accumulator layout to the B-operand layout with movmatrix. The
// exponentials run in base 2 with the scale folded into log2(e)*scale.
// Warps merge their partials in shared memory in fixed order, so results
// are deterministic. A split's last, ragged tile is loaded shifted back to
// end at the split's last key, so every row TMA brings in holds either a
// real cache entry of this row or zero fill; keys outside the tile's own
// range are masked by selection (-inf), never by arithmetic on garbage.

#include <cuda_runtime.h>
#include <math.h>

#include "gqa_attn.h"
#include "plan.cuh"
#include "ptx.cuh"
#include "runtime.cuh"

namespace gqa {
namespace decode {

constexpr int kMaxG = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct SplitParams {
    const uint16_t* q;        // [B, H_q, D]
    const int32_t* seqlens;   // [B] or null
    uint16_t* o;              // [B, H_q, D]   (written when ns == 1)
    float* lse;               // [B, H_q] or null (written when ns == 1)
    float* part_o;            // [B, H_q, ns, D]  unnormalised
    float* part_m;            // [B, H_q, ns]     base-2 running max
    float* part_l;            // [B, H_q, ns]
    unsigned* status;
    int B, H_q, H_kv, G, S_max, ns, L;
    float scale_log2;         // scale * log2(e)
};

template <int D, int TILE_T, int STAGES, int WARPS>
struct SplitCfg {
    static constexpr int kBoxes = D / 64;               // 128-byte column boxes per row
    static constexpr int kBoxBytes = TILE_T * 128;      // one box: TILE_T rows x 128 B
    static constexpr int kKBytes = kBoxes * kBoxBytes;  // K (or V) part of a stage
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kRingBytes = WARPS * STAGES * kStageBytes;
    static constexpr int kOPitch = D + 4;               // floats; breaks bank conflicts
    static constexpr int kMergeBytes = WARPS * kMaxG * (kOPitch + 2) * 4;
    static constexpr int kDataBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static constexpr int kBarOffset = kDataBytes;
    static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kDataBytes + WARPS * STAGES * 8;
    static constexpr int kMT = TILE_T / 16;             // 16-key m-tiles per stage
    static constexpr int kKC = D / 16;                  // 16-wide k-chunks of a head dim
    static_assert(TILE_T % 16 == 0 && TILE_T <= 256, "tile");
    static_assert(D == 64 || D == 128, "head dim");
};

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ int load_seqlen(const int32_t* seqlens, int b, int S_max,
                                           unsigned* status, bool report) {
    int sl = seqlens ? seqlens[b] : S_max;
    if (sl < 0 || sl > S_max) {
        if (report) atomicOr(status, kStatusBadSeqlen);
        sl = sl < 0 ? 0 : S_max;
    }
    return sl;
}

template <int D, int TILE_T, int STAGES, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1)
    split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v, const SplitParams p) {
    using C = SplitCfg<D, TILE_T, STAGES, WARPS>;
    const int s = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;

    // Let the combine grid get scheduled while this one streams (it waits
    // for our results with griddepcontrol.wait before reading anything).
    pdl_launch_dependents();

    const int seqlen = load_seqlen(p.seqlens, b, p.S_max, p.status,
                                   s == 0 && kv == 0 && threadIdx.x == 0);
    const SplitRange r = split_range(p.L, s, seqlen);
    if (r.end <= r.start) {
        // Empty split. The combine skips it; with a single split this block
        // owns the output: a row with no visible keys gives O = 0, lse = -inf.
        if (p.ns == 1) {
            for (int i = threadIdx.x; i < p.G * D; i += WARPS * 32) {
                const int h = kv * p.G + i / D;
                p.o[(size_t(b) * p.H_q + h) * D + i % D] = 0;
                if (i % D == 0 && p.lse) p.lse[size_t(b) * p.H_q + h] = -INFINITY;
            }
        }
        return;
    }

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset) + warp * STAGES;
    uint8_t* ring = smem + size_t(warp) * STAGES * C::kStageBytes;

    const int len = r.end - r.start;
    const int n_tiles = (len + TILE_T - 1) / TILE_T;
    const int my_n = warp < n_tiles ? (n_tiles - warp + WARPS - 1) / WARPS : 0;
    const int zc = b * p.H_kv + kv;  // outer TMA coordinate: (batch, KV head)

    if (lane == 0) {
        for (int i = 0; i < STAGES; ++i) mbar_init(smem_u32(&bars[i]), 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
    }
    __syncwarp();

    const uint64_t policy = l2_policy_evict_first();
    // Row of the first key TMA brings in for this warp's i-th tile.
    auto tile_y = [&](int i) {
        const int tok0 = r.start + (warp + i * WARPS) * TILE_T;
        return tok0 + TILE_T <= r.end ? tok0 : r.end - TILE_T;
    };
    auto issue = [&](int i) {
        const int slot = i % STAGES;
        const uint32_t bar = smem_u32(&bars[slot]);
        const uint32_t kdst = smem_u32(ring + slot * C::kStageBytes);
        const uint32_t vdst = kdst + C::kKBytes;
        const int y = tile_y(i);
        mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
        for (int h = 0; h < C::kBoxes; ++h) {
            tma_load_3d(kdst + h * C::kBoxBytes, &tmap_k, h * 64, y, zc, bar, policy);
            tma_load_3d(vdst + h * C::kBoxBytes, &tmap_v, h * 64, y, zc, bar, policy);
        }
    };

    int issued = 0;
    if (lane == 0) {
        for (; issued < STAGES && issued < my_n; ++issued) issue(issued);
    }
    issued = __shfl_sync(0xffffffffu, issued, 0);

    // q^T as the B operand (k = head dim, n = query head g of this group).
    uint32_t qf[C::kKC][2];
    {
        const bool has = g < p.G;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            p.q + (size_t(b) * p.H_q + kv * p.G + (has ? g : 0)) * D);
#pragma unroll
        for (int kc = 0; kc < C::kKC; ++kc) {
            qf[kc][0] = has ? qrow[(kc * 16 + 2 * c) / 2] : 0u;
            qf[kc][1] = has ? qrow[(kc * 16 + 8 + 2 * c) / 2] : 0u;
        }
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
        if (alive) alive = mbar_wait_bounded(smem_u32(&bars[slot]), (i / STAGES) & 1, p.status);
        alive = __all_sync(0xffffffffu, alive);  // keep the warp's control flow uniform
        waited = i + 1;
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

        __syncwarp();
        if (lane == 0 && alive && issued < my_n) {
            issue(issued);
        }
        if (alive && issued < my_n) ++issued;
    }
    // A wait that ran out may leave copies in flight: wait for them (bounded)
    // before the shared memory is reused or released.
    for (int i = waited; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&bars[i % STAGES]), (i / STAGES) & 1, p.status);

#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }

    // ---- merge the warps' partials in shared memory, warp order fixed
    __syncthreads();  // every warp is done with its ring
    float* o_s = reinterpret_cast<float*>(smem);                  // [WARPS][8][kOPitch]
    float* m_s = o_s + WARPS * kMaxG * C::kOPitch;                // [WARPS][8]
    float* l_s = m_s + WARPS * kMaxG;                             // [WARPS][8]
    if (g == 0) {
        m_s[warp * kMaxG + 2 * c] = m0;
        m_s[warp * kMaxG + 2 * c + 1] = m1;
        l_s[warp * kMaxG + 2 * c] = l0;
        l_s[warp * kMaxG + 2 * c + 1] = l1;
    }
#pragma unroll
    for (int md = 0; md < C::kKC; ++md) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int dim = md * 16 + g + (e >> 1) * 8;
            const int head = 2 * c + (e & 1);
            o_s[(warp * kMaxG + head) * C::kOPitch + dim] = acc[md][e];
        }
    }
    __syncthreads();

    for (int i = threadIdx.x; i < p.G * D; i += WARPS * 32) {
        const int head = i / D, dim = i % D;
        float mstar = -INFINITY;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) mstar = fmaxf(mstar, m_s[w * kMaxG + head]);
        float lsum = 0.f, osum = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            const float f = fast_exp2(m_s[w * kMaxG + head] - mstar);
            lsum += f * l_s[w * kMaxG + head];
            osum += f * o_s[(w * kMaxG + head) * C::kOPitch + dim];
        }
        const size_t row = size_t(b) * p.H_q + kv * p.G + head;
        if (p.ns == 1) {
            const float out = osum / lsum;
            p.o[row * D + dim] = __bfloat16_as_ushort(__float2bfloat16_rn(out));
            if (dim == 0 && p.lse) p.lse[row] = (mstar + __log2f(lsum)) * kLn2;
        } else {
            const size_t pr = row * p.ns + s;
            p.part_o[pr * D + dim] = osum;
            if (dim == 0) {
                p.part_m[pr] = mstar;
                p.part_l[pr] = lsum;
            }
        }
    }
}

struct CombineParams {
    const float* part_o;
    const float* part_m;
    const float* part_l;
    const int32_t* seqlens;
    uint16_t* o;
    float* lse;
    int B, H_q, S_max, ns, L;
};

constexpr int kCombineWarps = 8;

// One warp per (batch, query head): fold the row's non-empty splits in order
// s = 0, 1, ... with the log-sum-exp rule, normalise once, write O and lse.
template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const CombineParams p) {
    constexpr int kPer = D / 32;  // dims per lane
    pdl_wait_primary();           // the split grid's partials are complete and visible
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (row >= p.B * p.H_q) return;
    const int b = row / p.H_q;
    int seqlen = p.seqlens ? p.seqlens[b] : p.S_max;
    seqlen = seqlen < 0 ? 0 : (seqlen > p.S_max ? p.S_max : seqlen);
    const int n_act = active_splits(p.L, seqlen);
    float* out_lse = p.lse ? p.lse + row : nullptr;
    uint16_t* out = p.o + size_t(row) * D + lane * kPer;
    if (n_act == 0) {
#pragma unroll
        for (int j = 0; j < kPer; ++j) out[j] = 0;
        if (lane == 0 && out_lse) *out_lse = -INFINITY;
        return;
    }
    const float* pm = p.part_m + size_t(row) * p.ns;
    const float* pl = p.part_l + size_t(row) * p.ns;
    const float* po = p.part_o + size_t(row) * p.ns * D + lane * kPer;
    float mx = -INFINITY;
    for (int s = lane; s < n_act; s += 32) mx = fmaxf(mx, pm[s]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float lsum = 0.f;
    float acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j] = 0.f;
    for (int s = 0; s < n_act; ++s) {
        const float w = fast_exp2(pm[s] - mx);
        lsum += w * pl[s];
        const float* src = po + size_t(s) * D;
        if constexpr (kPer == 4) {
            const float4 v = *reinterpret_cast<const float4*>(src);
            acc[0] += w * v.x;
            acc[1] += w * v.y;
            acc[2] += w * v.z;
            acc[3] += w * v.w;
        } else {
            const float2 v = *reinterpret_cast<const float2*>(src);
            acc[0] += w * v.x;
            acc[1] += w * v.y;
        }
    }
    const float inv = 1.f / lsum;
#pragma unroll
    for (int j = 0; j < kPer; ++j) out[j] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[j] * inv));
    if (lane == 0 && out_lse) *out_lse = (mx + __log2f(lsum)) * kLn2;
}

// ------------------------------------------------------------------ host side

constexpr int kTileT = 32, kStages = 3, kWarps = 4;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
    size_t o_off, m_off, l_off, total;
};

WsLayout ws_layout(int B, int H_q, int d, int ns) {
    WsLayout w{};
    if (ns <= 1) return w;
    const size_t rows = size_t(B) * H_q * ns;
    w.o_off = 0;
    w.m_off = align256(rows * d * sizeof(float));
    w.l_off = w.m_off + align256(rows * sizeof(float));
    w.total = w.l_off + align256(rows * sizeof(float));
    return w;
}

template <int D>
int launch(const SplitParams& sp, const CUtensorMap& tk, const CUtensorMap& tv,
           cudaStream_t stream) {
    using C = SplitCfg<D, kTileT, kStages, kWarps>;
    auto kern = split_kernel<D, kTileT, kStages, kWarps>;
    static bool attr_set = false;  // benign race: setting it twice is harmless
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess)
            return GQA_ERR_CUDA;
        attr_set = true;
    }
    dim3 grid(sp.ns, sp.H_kv, sp.B);
    kern<<<grid, kWarps * 32, C::kSmemBytes, stream>>>(tk, tv, sp);
    if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
    if (sp.ns == 1) return GQA_OK;

    CombineParams cp{sp.part_o, sp.part_m, sp.part_l, sp.seqlens, sp.o, sp.lse,
                     sp.B, sp.H_q, sp.S_max, sp.ns, sp.L};
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
    if (H_q / H_kv > kMaxG) return GQA_ERR_UNSUPPORTED;
    if (int64_t(B) * H_kv * S_max > (int64_t(1) << 31)) return GQA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return GQA_ERR_MISALIGNED;
    return GQA_OK;
}

int run(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse,
        const int32_t* seqlens, int B, int H_q, int H_kv, int d, int S_max, float scale,
        int ns, void* ws, size_t ws_bytes, cudaStream_t stream) {
    unsigned* status = status_word();
    if (!status) return GQA_ERR_CUDA;
    const WsLayout wl = ws_layout(B, H_q, d, ns);
    if (ns > 1) {
        if (!ws || ws_bytes < wl.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
            return GQA_ERR_WORKSPACE;
    }
    CUtensorMap tk, tv;
    const uint64_t outer = uint64_t(B) * H_kv;
    if (encode_tmap_3d_bf16(&tk, k, d, S_max, outer, 64, kTileT, CU_TENSOR_MAP_SWIZZLE_128B) !=
            cudaSuccess ||
        encode_tmap_3d_bf16(&tv, v, d, S_max, outer, 64, kTileT, CU_TENSOR_MAP_SWIZZLE_128B) !=
            cudaSuccess)
        return GQA_ERR_CUDA;
    SplitParams sp{};
    sp.q = q;
    sp.seqlens = seqlens;
    sp.o = o;
    sp.lse = lse;
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    sp.part_o = ns > 1 ? reinterpret_cast<float*>(w8 + wl.o_off) : nullptr;
    sp.part_m = ns > 1 ? reinterpret_cast<float*>(w8 + wl.m_off) : nullptr;
    sp.part_l = ns > 1 ? reinterpret_cast<float*>(w8 + wl.l_off) : nullptr;
    sp.status = status;
    sp.B = B;
    sp.H_q = H_q;
    sp.H_kv = H_kv;
    sp.G = H_q / H_kv;
    sp.S_max = S_max;
    sp.ns = ns;
    sp.L = split_len(S_max, ns);
    sp.scale_log2 = scale * kLog2e;
    return d == 128 ? launch<128>(sp, tk, tv, stream) : launch<64>(sp, tk, tv, stream);
}

}  // namespace decode
}  // namespace gqa

using namespace gqa;

extern "C" size_t gqa_attn_decode_workspace_size(int B, int H_q, int d, int num_splits) {
    if (B < 0 || H_q <= 0 || (d != 64 && d != 128) || num_splits <= 0) return 0;
    return decode::ws_layout(B, H_q, d, num_splits).total;
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
        const int sms = num_sms();
        if (sms <= 0) return GQA_ERR_CUDA;
        ns = gqa_attn_pick_num_splits(B, H_kv, S_max, sms);
        if (ns < 1) return GQA_ERR_INVALID_ARG;
    }
    const size_t bytes = decode::ws_layout(B, H_q, d, ns).total;
    void* ws = nullptr;
    if (bytes > 0) {
        ws = stream_workspace(stream, bytes);
        if (!ws) return GQA_ERR_WORKSPACE;
    }
    return decode::run(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, S_max, scale, ns, ws, bytes,
                       stream);
}
