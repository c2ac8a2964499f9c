/*
 * gqa_attn.h — C ABI of the GB300 (sm_103a) grouped-query attention library.
 *
 * The operations are the ones defined on the page "ADR-0060: AHBM GQA Fused
 * Attention kernel (Llama3-70B)" (kernbench2):
 *   - decode: FlashDecoding split-KV sweep (§5.2 decode without sequence
 *     parallelism, §3 per-tile op sequence) followed by the log-sum-exp merge
 *     of the per-split partials (§4 reduction);
 *   - prefill: FlashAttention tiled online softmax with causal tile skipping
 *     and a boundary mask on partial tiles (§5.4 prefill without sequence
 *     parallelism, §3).
 * Both compute exactly O = softmax(Q K^T * scale + mask) V (the page's
 * algorithm-lineage paragraph: no new mathematics) and lse = ln sum exp of the
 * scaled, visible scores, per query row.
 *
 * Layouts (all row-major, contiguous, device memory unless stated):
 *   q    decode  [B, H_q, d]          prefill [B, H_q, T_q, d]      bf16
 *   k, v decode  [B, H_kv, S_max, d]  prefill [B, H_kv, S_kv, d]   bf16
 *   o    like q                                                    bf16
 *   lse  decode  [B, H_q]             prefill [B, H_q, T_q]        fp32
 * bf16 values are passed as their 16-bit patterns (uint16_t).
 * Query head h reads KV head h / G with G = H_q / H_kv: the G query heads of
 * one KV head are adjacent (§0.5 I/O contract stores Q per KV head as
 * [G, T_q, d]).
 *
 * Ownership: the caller owns every buffer passed in; the library never frees
 * or retains a caller pointer after the call returns. All calls are
 * asynchronous on `stream` (NULL = the legacy default stream) and do not
 * synchronise. Inputs are read-only (§0.5 preconditions: Q and K are
 * post-RoPE and the cache already holds the current token).
 *
 * Errors: every entry point returns 0 (GQA_OK) or a negative code and checks
 * its arguments on the host before launching anything; an invalid argument
 * never reaches the GPU. Errors the device detects (a bounded wait that ran
 * out, a seqlen outside [0, S_max]) set the library's device status word (one
 * per GPU, in the library's own device memory), which gqa_attn_check() reads
 * and clears. Every entry point reports there, gqa_attn_decode_noalloc
 * included.
 */
#ifndef GQA_ATTN_H_
#define GQA_ATTN_H_

#include <stddef.h>
#include <stdint.h>

/* The library is built with hidden symbol visibility; only the calls below
 * are exported. */
#if defined(__GNUC__)
#define GQA_API __attribute__((visibility("default")))
#else
#define GQA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* cudaStream_t;

enum {
    GQA_OK = 0,
    GQA_ERR_INVALID_ARG = -1,    /* null pointer, bad size, H_q % H_kv != 0, ... */
    GQA_ERR_UNSUPPORTED = -2,    /* d not in {64, 128}; decode: G > 16 */
    GQA_ERR_MISALIGNED = -3,     /* a tensor pointer is not 16-byte aligned */
    GQA_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed */
    GQA_ERR_DEVICE_TIMEOUT = -5, /* a kernel's bounded wait ran out (device status) */
    GQA_ERR_WORKSPACE = -6,      /* caller workspace too small or misaligned */
    GQA_ERR_DEVICE_BAD_INPUT = -7 /* the device saw a seqlen outside [0, S_max] */
};

/* ---------------------------------------------------------------- decode --
 * gqa_attn_decode: one new query token per sequence (T_q = 1) against a KV
 * cache of S_max slots, of which the first seqlens[b] are valid for row b
 * (seqlens == NULL: all S_max). Page: §5.2 (decode, no SP) — every past key is
 * visible, only the ragged tail is masked; G query heads are folded into the
 * matmul M dimension so each K/V tile is read once per KV head.
 *
 * Group size G = H_q / H_kv up to 16: a group of more than 8 query heads runs
 * as two CTAs per (split, KV head), each folding up to 8 heads into the MMA,
 * over the same K/V tiles (the second read mostly from L2).
 *
 * Split plan (§4 FlashDecoding split-and-combine; the page's round-robin
 * rank placement has no counterpart on one GPU): num_splits contiguous
 * chunks of L = ceil(S_max / num_splits) keys; split s of row b covers
 * [min(s*L, seqlen_b), min((s+1)*L, seqlen_b)). num_splits <= 0 picks it
 * with gqa_attn_pick_num_splits(B, H_kv, S_max, SMs of the current device);
 * for G > 8 (two CTAs per split and KV head, heads 0-7 and 8-15) the plan for
 * 2 * H_kv heads is taken instead when B * 2 * H_kv * n <= SMs and its splits
 * hold at most 1024 keys. gqa_attn_decode_partial, _ring and _noalloc resolve
 * num_splits == 0 the same way; _q8 and _q4 use their own plan for H_kv.
 *
 *   q, k, v, o : see layouts above; 16-byte aligned.
 *   lse        : [B, H_q] fp32, or NULL to skip it. A row with seqlen 0 gets
 *                O = 0 and lse = -inf.
 *   seqlens    : device int32 [B], or NULL. Values outside [0, S_max] are
 *                clamped and reported as GQA_ERR_DEVICE_BAD_INPUT by
 *                gqa_attn_check().
 *   scale      : softmax scale (finite), usually 1/sqrt(d).
 *   num_splits : 0 = automatic, else 1..8192.
 * The workspace for the per-split partials is library-owned: one buffer per
 * (device, stream), grown with stream-ordered allocation when a call needs
 * more than it holds. A call that would have to grow it during stream capture
 * returns GQA_ERR_WORKSPACE, so make the first (largest) call on a stream
 * before capturing. A buffer replaced by a larger one is kept until the
 * process exits (never freed), so work captured earlier on the stream, such
 * as a CUDA graph, stays valid; the kept buffers together are smaller than the
 * current one. Calls on different streams never share a workspace.
 */
GQA_API int gqa_attn_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            uint16_t* o, float* lse, const int32_t* seqlens,
                            int B, int H_q, int H_kv, int d, int S_max,
                            float scale, int num_splits, cudaStream_t stream);

/* The same, with a caller-provided device workspace (256-byte aligned) of at
 * least gqa_attn_decode_workspace_size(B, H_q, d, num_splits) bytes; here
 * num_splits must be >= 1 (resolve 0 with gqa_attn_pick_num_splits first).
 * The workspace holds no state between calls; calls that overlap on the GPU
 * must not share one. */
GQA_API int gqa_attn_decode_ws(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               uint16_t* o, float* lse, const int32_t* seqlens,
                               int B, int H_q, int H_kv, int d, int S_max,
                               float scale, int num_splits,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of decode workspace for these sizes (0 when num_splits == 1, which
 * writes O directly). Returns 0 on invalid sizes as well. */
GQA_API size_t gqa_attn_decode_workspace_size(int B, int H_q, int d, int num_splits);

/* gqa_attn_decode for callers that must not allocate device memory. (The page
 * has no counterpart: this is a deployment option, not part of the method.)
 * Some callers cannot call cudaMalloc: a serving process that partitions HBM
 * once at start-up and forbids later allocations, a host that routes every
 * device byte through its own allocator, or a latency-critical path that
 * cannot afford cudaMalloc's implicit device synchronisation. This entry
 * point allocates nothing: the caller passes inputs and outputs exactly as for
 * gqa_attn_decode, and the scratch the split merge needs lives in a fixed
 * 8 MiB array inside the library (GQA_NOALLOC_SCRATCH_BYTES), which every GPU
 * that loads the library holds until the process exits.
 *   - Returns GQA_ERR_WORKSPACE, without launching, when the problem needs more
 *     scratch than that: gqa_attn_decode_workspace_size(B, H_q, d, n) must be
 *     <= GQA_NOALLOC_SCRATCH_BYTES for the split count n in use (the resolved
 *     one when num_splits == 0).
 *   - The first call on a device looks up the array's device address; make
 *     that first call before any stream capture.
 *   - Every call shares the one array, and it keeps the last call's contents
 *     (nothing in it needs to start at zero: each call writes every partial
 *     before reading it). Calls that overlap on the GPU, on any streams, race
 *     on it: serialise them.
 *   - Device-detected errors (a clamped seqlen, a bounded wait that ran out)
 *     go to the library's status word like every other call's; read them
 *     with gqa_attn_check(), which allocates nothing either.
 */
#define GQA_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
GQA_API int gqa_attn_decode_noalloc(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    uint16_t* o, float* lse, const int32_t* seqlens,
                                    int B, int H_q, int H_kv, int d, int S_max,
                                    float scale, int num_splits, cudaStream_t stream);

/* ------------------------------------------ sequence-parallel decode ------
 * Page: ADR-0060 §5.3 (decode with sequence parallelism: every rank sweeps its
 * own slice of the keys) and §4 (the partials meet in a log-sum-exp
 * reduce-to-root, normalised once at the root). A sequence can be cut into R
 * contiguous key ranges, one per device or stream: slice r of every row is
 * [start_r, end_r) from gqa_attn_split_bounds(S_max, R, S_max, ...), and a row
 * of length seqlen has max(0, min(seqlen, end_r) - start_r) keys in it. Each
 * slice is decoded on its own into a partial (O_r normalised over the slice's
 * keys, lse_r), and gqa_attn_merge folds the R partials into the result. Only
 * (d + 1) * 4 bytes per (row, query head) move between ranks. */

/* gqa_attn_decode over one slice, with the output kept in fp32 for the merge:
 * arguments, split plan, workspace and errors as gqa_attn_decode, where k and
 * v are the slice's own cache [B, H_kv, S_max, d] (S_max = the slice length)
 * and seqlens the rows' key counts inside it.
 *   o_part   : fp32 [B, H_q, d], 16-byte aligned; a row with no keys gets 0.
 *   lse_part : fp32 [B, H_q] (required); a row with no keys gets -inf. */
GQA_API int gqa_attn_decode_partial(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                    float* o_part, float* lse_part, const int32_t* seqlens,
                                    int B, int H_q, int H_kv, int d, int S_max, float scale,
                                    int num_splits, cudaStream_t stream);

/* Merges R partials in rank order with the log-sum-exp rule:
 *   lse = ln sum_r exp(lse_r),  O = sum_r exp(lse_r - lse) O_r  (then bf16).
 *   o_parts   : fp32 [R, rows, d] (16-byte aligned), rows = B * H_q;
 *   lse_parts : fp32 [R, rows]; a part with lse_r = -inf (no keys) is skipped
 *               whatever its O_r holds;
 *   o         : bf16 [rows, d]; lse: fp32 [rows] or NULL.
 * A row whose parts are all empty gets O = 0 and lse = -inf. d in {64, 128},
 * R >= 1. Async on `stream`; deterministic (fixed order). */
GQA_API int gqa_attn_merge(const float* o_parts, const float* lse_parts, uint16_t* o, float* lse,
                           int R, int rows, int d, cudaStream_t stream);

/* ------------------------------------------ ring-buffer cache with sinks --
 * Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §2 item 4 (a KV
 * cache of fixed max_tokens that never grows) and §4 item 2 (once it wraps,
 * the oldest entry is overwritten under an attention-sink + local-window
 * policy). The cache of each (batch row, KV head) has `capacity` slots:
 * slots [0, n_sink) keep the row's first n_sink tokens for good, and token
 * t >= n_sink lives in slot n_sink + (t - n_sink) % (capacity - n_sink), so a
 * row that has produced seqlen tokens holds its sinks plus its last
 * capacity - n_sink tokens (all of them while seqlen <= capacity).
 * Requires 0 <= n_sink < capacity. */

/* Writes each row's newest token into its slot: k_new/v_new [B, H_kv, d]
 * (bf16, 16-byte aligned) go to k_cache/v_cache [B, H_kv, capacity, d] at
 * the slot of token positions[b] (a device int32 [B]: the token's index, i.e.
 * the row's length before this append). A negative position writes nothing
 * and sets the status word's bad-length bit (gqa_attn_check reports
 * GQA_ERR_DEVICE_BAD_INPUT). Async on `stream`; d in {64, 128}. */
GQA_API int gqa_attn_ring_append(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_new,
                                 const uint16_t* v_new, const int32_t* positions, int B, int H_kv,
                                 int d, int capacity, int n_sink, cudaStream_t stream);

/* Decode over such a cache: arguments as gqa_attn_decode with S_max =
 * capacity, except that seqlens (required, device int32 [B]) counts every
 * token the row has produced and may exceed capacity. The row attends to its
 * live slots, min(seqlens[b], capacity) of them, which are exactly the sink
 * and window tokens; a negative length is clamped to 0 and reported. Uses the
 * library-owned workspace like gqa_attn_decode. */
GQA_API int gqa_attn_decode_ring(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 uint16_t* o, float* lse, const int32_t* seqlens,
                                 int B, int H_q, int H_kv, int d, int capacity, int n_sink,
                                 float scale, int num_splits, cudaStream_t stream);

/* ------------------------------------------------------- INT8 KV cache ----
 * Page: "Gemma 3N E4B on pccx v002 — Execution / Scheduling", §4 item 3
 * (optional INT4 / INT8 KV quantisation, recommended above 4 K tokens; the page
 * fixes no scheme). Here: one fp32 scale per (batch row, KV head, token) for K
 * and one for V, scale = max|x| / 127 over the token's d values, codes
 * rint(x / scale) in [-127, 127] (ties to even; both divisions are single IEEE
 * fp32 divisions; an all-zero token has scale 0 and codes 0). A code x is
 * stored as the byte x + 128 (uint8, so 128 is zero). Layouts:
 *   k_codes  uint8 [B, H_kv, S, d]   token-major, like the bf16 K cache
 *   v_codes  uint8 [B, H_kv, d, S]   dim-major (V transposed)
 *   k_scales, v_scales  fp32 [B, H_kv, S]
 * d must be 128 and S a multiple of 16; every pointer 16-byte aligned. */

/* Quantises a bf16 cache k, v [B, H_kv, S, d] into the layouts above.
 * Async on `stream`. */
GQA_API int gqa_attn_quantize_kv_q8(const uint16_t* k, const uint16_t* v, uint8_t* k_codes,
                                    uint8_t* v_codes, float* k_scales, float* v_scales,
                                    int B, int H_kv, int S, int d, cudaStream_t stream);

/* Split-KV decode over an INT8 cache: arguments, outputs, split plan,
 * workspace and errors as gqa_attn_decode (num_splits == 0 resolved with
 * gqa_attn_pick_num_splits_q8), with K and V given as codes and
 * scales (S_max = the caches' S). The result is attention over the
 * dequantised cache code * scale: the kernel turns each stored byte into the
 * exact f16 value code + 1152, takes the 1152 offset off once per head, and
 * applies the K scale to each token's scores and the V scale to each token's
 * softmax weight. Rows, ragged lengths and seqlens behave as in
 * gqa_attn_decode; scales and codes beyond a row's length are never used (they
 * may hold anything). */
GQA_API int gqa_attn_decode_q8(const uint16_t* q, const uint8_t* k_codes,
                               const uint8_t* v_codes, const float* k_scales,
                               const float* v_scales, uint16_t* o, float* lse,
                               const int32_t* seqlens, int B, int H_q, int H_kv, int d,
                               int S_max, float scale, int num_splits, cudaStream_t stream);

/* ------------------------------------------------------- INT4 KV cache ----
 * The same page and recommendation (§4 item 3), with 4-bit codes: one fp32
 * scale per (batch row, KV head, token) for K and one for V, scale =
 * max|x| / 7, codes rint(x / scale) in [-7, 7] (ties to even; single IEEE
 * fp32 divisions; an all-zero token has scale 0 and codes 0). A code x is
 * stored as the nibble x + 8, two per byte, the lower dim (K) or the lower
 * token (V) in the low nibble. Layouts:
 *   k_codes  uint8 [B, H_kv, S, d/2]  token-major
 *   v_codes  uint8 [B, H_kv, d, S/2]  dim-major (V transposed)
 *   k_scales, v_scales  fp32 [B, H_kv, S]
 * d must be 128 and S a multiple of 32; every pointer 16-byte aligned. */

/* Quantises a bf16 cache k, v [B, H_kv, S, d] into the layouts above.
 * Async on `stream`. */
GQA_API int gqa_attn_quantize_kv_q4(const uint16_t* k, const uint16_t* v, uint8_t* k_codes,
                                    uint8_t* v_codes, float* k_scales, float* v_scales,
                                    int B, int H_kv, int S, int d, cudaStream_t stream);

/* Split-KV decode over an INT4 cache: as gqa_attn_decode_q8 (num_splits == 0
 * resolved with gqa_attn_pick_num_splits_q4). The result is attention over
 * the dequantised cache code * scale: the kernel turns each nibble into an
 * exact f16 value (K: 1032 + code, or 1152 + 16 x code for every second
 * nibble; V: 1152 + 16 x code), scales the partner operand of the 16 x code
 * values by 1/16, takes the offsets off once per head, and applies the K
 * scale to each token's scores and the V scale to each token's softmax
 * weight. */
GQA_API int gqa_attn_decode_q4(const uint16_t* q, const uint8_t* k_codes,
                               const uint8_t* v_codes, const float* k_scales,
                               const float* v_scales, uint16_t* o, float* lse,
                               const int32_t* seqlens, int B, int H_q, int H_kv, int d,
                               int S_max, float scale, int num_splits, cudaStream_t stream);

/* --------------------------------------------------------------- prefill --
 * gqa_attn_prefill: T_q new queries at global positions q_offset + t against
 * S_kv keys (the cache already holds the new keys: q_offset + T_q <= S_kv).
 * causal != 0: key j is visible to query t iff j <= q_offset + t; fully
 * future KV tiles are skipped and partial tiles masked (§5.4). causal == 0:
 * every key is visible. Fixed to the Llama3-70B head geometry of §0
 * (H_q = 64, H_kv = 8, d = 128); gqa_attn_prefill_ex takes any supported one
 * (d = 64 or 128, any H_q divisible by H_kv).
 *   lse   : [B, H_q, T_q] fp32, or NULL.
 *   scale : softmax scale, finite and > 0 (§0.5 fixes 1/sqrt(d)); anything
 *           else returns GQA_ERR_INVALID_ARG.
 */
GQA_API int gqa_attn_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             uint16_t* o, float* lse,
                             int B, int T_q, int S_kv, int q_offset, int causal,
                             float scale, cudaStream_t stream);

GQA_API int gqa_attn_prefill_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                uint16_t* o, float* lse,
                                int B, int H_q, int H_kv, int d, int T_q, int S_kv,
                                int q_offset, int causal, float scale, cudaStream_t stream);

/* Sequence-parallel prefill (page: ADR-0060 §5.5 prefill with SP, where the
 * K/V slices travel between ranks, and §4 for the merge): the prefill of T_q
 * queries at global positions q_offset + t against ONE slice of the keys, the
 * S_kv keys at global positions key_offset + j held in the slice's own cache
 * k, v [B, H_kv, S_kv, d]. causal != 0: query t sees key j iff
 * key_offset + j <= q_offset + t (keys past the slice come from other
 * slices, so q_offset + T_q may exceed key_offset + S_kv); causal == 0: every
 * key of the slice. A row that sees no key of the slice gets O = 0 and
 * lse = -inf. O is kept in fp32 for gqa_attn_merge over the slices (rows =
 * B * H_q * T_q):
 *   o_part   : fp32 [B, H_q, T_q, d], 16-byte aligned;
 *   lse_part : fp32 [B, H_q, T_q] (required).
 * q_offset, key_offset >= 0; other arguments and errors as
 * gqa_attn_prefill_ex. */
GQA_API int gqa_attn_prefill_partial(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                     float* o_part, float* lse_part, int B, int H_q, int H_kv,
                                     int d, int T_q, int S_kv, int q_offset, int key_offset,
                                     int causal, float scale, cudaStream_t stream);

/* ------------------------------------------------------ plan / scheduler --
 * Integer helpers the kernels use, exported so tests can compare them with
 * independent derivations bit for bit. Host-only; no GPU needed.
 */

/* Split count for a decode problem. First, one wave of whole-row clusters:
 * the largest n of 16, 8, 4, 2 with B * H_kv * n <= num_sms, taken if
 * B * H_kv * n >= 0.8 * num_sms and 256 <= ceil(S_max / n) <= 2048, or
 * <= 16384 when B == 1 (the tighter bound guards ragged batches), or, with
 * fewer SMs busy, if 256 <= ceil(S_max / n) <= 512 (every row then merges on
 * chip, with no combine kernel). Otherwise
 * n = ceil(num_sms / (B * H_kv)) blocks per row (when above 16, rounded down
 * to a multiple of 16 if the blocks then still cover >= 80% of the SMs), at
 * least ceil(S_max / 1024) (rounded up to a multiple of 16 when above 16), and
 * at most max(1, S_max / 256) so no split is shorter than 256 keys. Returns
 * >= 1, or GQA_ERR_INVALID_ARG. */
GQA_API int gqa_attn_pick_num_splits(int B, int H_kv, int S_max, int num_sms);

/* Split count for a decode over an INT8 cache: gqa_attn_pick_num_splits for a
 * row of ceil(S_max / 2) keys, except that the one-wave plan's bound stays
 * 2048 keys for B == 1 too (these decodes are bound by each CTA's issue rate,
 * not by HBM). The split-length bounds are sized in bytes, and an INT8 token
 * (2 x d code bytes + 2 fp32 scales) is about half a bf16 token (4 x d
 * bytes). Returns >= 1, or GQA_ERR_INVALID_ARG. */
GQA_API int gqa_attn_pick_num_splits_q8(int B, int H_kv, int S_max, int num_sms);

/* Split count for a decode over an INT4 cache: the INT8 rule,
 * gqa_attn_pick_num_splits_q8. An INT4 token is about a quarter of a bf16 one
 * in bytes, but both quantised decodes are bound by instruction issue rather
 * than bytes, and measured faster with the INT8 split counts. Returns >= 1, or
 * GQA_ERR_INVALID_ARG. */
GQA_API int gqa_attn_pick_num_splits_q4(int B, int H_kv, int S_max, int num_sms);

/* Cluster size a decode launch uses on a GPU with num_sms SMs: the largest of
 * 16, 8, 4, 2 that divides num_splits (else 1), at most 8 when the grid of
 * num_splits * H_kv * B CTAs needs more than one wave (more CTAs than SMs).
 * (For a group of more than 8 query heads the grid has twice that many CTAs:
 * pass 2 * H_kv.)
 * The splits of one cluster are merged on chip; a row spanning several
 * clusters is finished by the combine kernel. Returns the size, or
 * GQA_ERR_INVALID_ARG. */
GQA_API int gqa_attn_decode_cluster_size(int B, int H_kv, int num_splits, int num_sms);

/* Fills starts[s], ends[s] (s < num_splits) with the decode split plan above
 * for one row of length seqlen (0 <= seqlen <= S_max). */
GQA_API int gqa_attn_split_bounds(int S_max, int num_splits, int seqlen,
                                  int32_t* starts, int32_t* ends);

/* §5.4 classification of query block [qs, qe) against KV tile [ks, ke), in
 * global positions: 0 = all past (ke <= qs, no mask), 2 = all future
 * (ks >= qe, skipped), 1 = partial (masked). */
GQA_API int gqa_attn_tile_class(int qs, int qe, int ks, int ke);

/* Tile counts of the prefill kernel's own schedule for one (batch, head):
 * query blocks of gqa_attn_prefill_block_m() rows, KV tiles of
 * gqa_attn_prefill_block_n() keys, classified as above. Writes the number of
 * all-past, partial and all-future (skipped) tile pairs. */
GQA_API int gqa_attn_prefill_tile_counts(int T_q, int S_kv, int q_offset, int causal,
                                         int64_t* n_past, int64_t* n_partial, int64_t* n_future);
GQA_API int gqa_attn_prefill_block_m(void);
GQA_API int gqa_attn_prefill_block_n(void);

/* Work order of a prefill launch (page: ADR-0060 §5.4 prefill scheduling;
 * the kernel is persistent, one CTA per SM over all work items). A work item
 * is one query block of two query heads of a KV group (even G) or two
 * consecutive query blocks of one head (odd G). When the K and V rows of all
 * B * H_kv groups are larger than an L2 budget (48 MiB), the items are
 * ordered by super-groups of (batch, KV head) whose K/V fits in the budget
 * (n_sg = ceil(groups / max(1, floor(budget / group bytes))) super-groups;
 * group g in super-group g * n_sg / groups),
 * heaviest first within a super-group, and each goes to the CTA with the
 * least work so far (item cost: its KV tiles + 1), so that concurrently
 * running CTAs share their keys in L2; otherwise the kernel's closed-form
 * order runs. Host-only: writes off[0..num_ctas] and items[0..off[num_ctas])
 * (CTA c runs items[off[c]] .. items[off[c+1]-1], in the kernel's own item
 * numbers) and returns the number of items, or 0 when the closed-form order is
 * kept (nothing written) or the table does not fit (more than 12288 items or
 * 160 CTAs). item_cap bounds `items`. Errors: GQA_ERR_INVALID_ARG (bad sizes,
 * q_offset < 0, null pointers, item_cap too small), GQA_ERR_UNSUPPORTED (d not
 * in {64, 128}, or a shape the prefill entry points reject). */
GQA_API int gqa_attn_prefill_schedule(int B, int H_q, int H_kv, int d, int T_q, int S_kv,
                                      int q_offset, int causal, int num_ctas, int32_t* off,
                                      int32_t* items, int item_cap);

/* ------------------------------------------------------------ status ----- */

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device (allocates no memory). Returns GQA_OK,
 * GQA_ERR_DEVICE_TIMEOUT, GQA_ERR_DEVICE_BAD_INPUT or GQA_ERR_CUDA. The word
 * collects the errors of every call on that device since the last check. */
GQA_API int gqa_attn_check(cudaStream_t stream);

/* Test hook for failure reporting: the next `launches` decode or prefill
 * calls (gqa_attn_decode*, gqa_attn_prefill*) each make their first block
 * withhold one copy (decode: its first K/V copy; prefill: its first Q copy).
 * The bounded waits on it then run out (after about one second each), the
 * kernel records the timeout in the device status word and finishes
 * normally, and gqa_attn_check() returns GQA_ERR_DEVICE_TIMEOUT. The output of
 * such a call is undefined; nothing faults and later calls are unaffected.
 * 0 disarms. Returns GQA_OK or GQA_ERR_INVALID_ARG (launches < 0). */
GQA_API int gqa_attn_debug_inject_timeout(int launches);

/* Causal-skip check (page: ADR-0060 §11, verification plan: the number of
 * tile GEMMs equals the lower-triangle tile count). In a library built with
 * -DGQA_DEBUG the prefill MMA issuers count every S = Q K^T tile they issue,
 * per (batch row, query head, query block, KV tile), split by the §5.4 class
 * of gqa_attn_tile_class (causal == 0: every tile counts as all past). This
 * synchronises the device, writes counts[0..2] = all-past, partial,
 * all-future tiles issued since the last clear, and zeroes the counters when
 * clear != 0. A correct schedule issues no all-future tile. Other builds
 * return GQA_ERR_UNSUPPORTED and touch nothing. */
GQA_API int gqa_attn_debug_tile_counts(int64_t* counts, int clear);

/* Test hook for the prefill work order (see gqa_attn_prefill_schedule):
 * budget_bytes < 0 restores the library's 48 MiB L2 budget; 0 keeps the
 * closed-form order for every launch; > 0 uses that budget (a small one makes
 * even tiny problems run a host-made order of one group per super-group).
 * Applies to later calls of gqa_attn_prefill* and gqa_attn_prefill_schedule.
 * Returns GQA_OK. */
GQA_API int gqa_attn_debug_prefill_order(int64_t budget_bytes);

/* Static, human-readable text for a return code. */
GQA_API const char* gqa_attn_strerror(int code);

/* Library version as major * 10000 + minor * 100 + patch. */
GQA_API int gqa_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H_ */
