// Causal GQA prefill entry points. The tcgen05 kernel is not in this build
// yet: both entry points validate their arguments and return
// GQA_ERR_UNSUPPORTED.

#include "gqa_attn.h"

extern "C" int gqa_attn_prefill_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   uint16_t* o, float* lse, int B, int H_q, int H_kv, int d,
                                   int T_q, int S_kv, int q_offset, int causal, float scale,
                                   cudaStream_t stream) {
    (void)lse; (void)causal; (void)scale; (void)stream;
    if (!q || !k || !v || !o || B < 0 || H_q <= 0 || H_kv <= 0 || T_q < 0 || S_kv < 0 ||
        q_offset < 0 || H_q % H_kv != 0)
        return GQA_ERR_INVALID_ARG;
    (void)d;
    return GQA_ERR_UNSUPPORTED;
}

extern "C" int gqa_attn_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                uint16_t* o, float* lse, int B, int T_q, int S_kv, int q_offset,
                                int causal, float scale, cudaStream_t stream) {
    return gqa_attn_prefill_ex(q, k, v, o, lse, B, 64, 8, 128, T_q, S_kv, q_offset, causal,
                               scale, stream);
}
