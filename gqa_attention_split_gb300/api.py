"""ctypes binding for libgqa_attn.so — argument marshalling only.

The functions named ``gqa_attn_*`` mirror the C ABI in ``include/gqa_attn.h``
one to one (raw device pointers as ints, sizes, a ``cudaStream_t`` as an int).
``decode`` and ``prefill`` are conveniences over them for torch tensors: they
check dtype/shape/device, allocate outputs, pass ``data_ptr()`` and the current
stream, and raise ``GqaError`` on a non-zero return code. Every step of the
computation runs in the library's CUDA kernels; nothing here computes.

The library must be built first (``python -m gqa_attention_split_gb300.build``
or ``__graft_entry__.build()``); loading fails loudly otherwise.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgqa_attn.so")

GQA_OK = 0
GQA_ERR_INVALID_ARG = -1
GQA_ERR_UNSUPPORTED = -2
GQA_ERR_MISALIGNED = -3
GQA_ERR_CUDA = -4
GQA_ERR_DEVICE_TIMEOUT = -5
GQA_ERR_WORKSPACE = -6
GQA_ERR_DEVICE_BAD_INPUT = -7

# name -> (restype, argtypes); every symbol include/gqa_attn.h declares.
_P, _I, _F, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGNATURES = {
    "gqa_attn_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "gqa_attn_decode_ws": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _S,
                                _P]),
    "gqa_attn_decode_workspace_size": (_S, [_I, _I, _I, _I]),
    "gqa_attn_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "gqa_attn_decode_partial": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I,
                                     _P]),
    "gqa_attn_merge": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "gqa_attn_ring_append": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "gqa_attn_quantize_kv_q8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "gqa_attn_decode_q8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "gqa_attn_decode_ring": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "gqa_attn_prefill": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "gqa_attn_prefill_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "gqa_attn_prefill_partial": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                      _F, _P]),
    "gqa_attn_pick_num_splits": (_I, [_I, _I, _I, _I]),
    "gqa_attn_pick_num_splits_q8": (_I, [_I, _I, _I, _I]),
    "gqa_attn_pick_num_splits_q4": (_I, [_I, _I, _I, _I]),
    "gqa_attn_quantize_kv_q4": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "gqa_attn_decode_q4": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "gqa_attn_decode_cluster_size": (_I, [_I, _I, _I, _I]),
    "gqa_attn_split_bounds": (_I, [_I, _I, _I, _P, _P]),
    "gqa_attn_tile_class": (_I, [_I, _I, _I, _I]),
    "gqa_attn_prefill_tile_counts": (_I, [_I, _I, _I, _I, _P, _P, _P]),
    "gqa_attn_prefill_block_m": (_I, []),
    "gqa_attn_prefill_block_n": (_I, []),
    "gqa_attn_prefill_schedule": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I]),
    "gqa_attn_check": (_I, [_P]),
    "gqa_attn_debug_inject_timeout": (_I, [_I]),
    "gqa_attn_debug_tile_counts": (_I, [_P, _I]),
    "gqa_attn_debug_prefill_order": (_I, [ctypes.c_int64]),
    "gqa_attn_strerror": (ctypes.c_char_p, [_I]),
    "gqa_attn_version": (_I, []),
}

_lib = None
_lock = threading.Lock()


class GqaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


def load(path: str) -> ctypes.CDLL:
    """Loads a build of the library at ``path`` with every signature set.
    ``lib()`` uses it for the product library; tests use it for the debug
    build (``build.build(debug=True)``), which loads beside it."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with "
            "`python -m gqa_attention_split_gb300.build` (CUDA 13, sm_103a)")
    L = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib() -> ctypes.CDLL:
    """Loads libgqa_attn.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            _lib = load(LIB_PATH)
    return _lib


def symbols():
    return list(_SIGNATURES)


# ---- one-to-one C ABI mirrors --------------------------------------------


def gqa_attn_decode(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, S_max, scale, num_splits,
                    stream):
    return lib().gqa_attn_decode(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, S_max, scale,
                                 num_splits, stream)


def gqa_attn_decode_ws(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, S_max, scale, num_splits,
                       workspace, workspace_bytes, stream):
    return lib().gqa_attn_decode_ws(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, S_max, scale,
                                    num_splits, workspace, workspace_bytes, stream)


def gqa_attn_decode_noalloc(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, S_max, scale,
                            num_splits, stream):
    return lib().gqa_attn_decode_noalloc(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, S_max,
                                         scale, num_splits, stream)


NOALLOC_SCRATCH_BYTES = 8 << 20  # GQA_NOALLOC_SCRATCH_BYTES


def gqa_attn_decode_workspace_size(B, H_q, d, num_splits):
    return lib().gqa_attn_decode_workspace_size(B, H_q, d, num_splits)


def gqa_attn_prefill(q, k, v, o, lse, B, T_q, S_kv, q_offset, causal, scale, stream):
    return lib().gqa_attn_prefill(q, k, v, o, lse, B, T_q, S_kv, q_offset, causal, scale,
                                  stream)


def gqa_attn_prefill_ex(q, k, v, o, lse, B, H_q, H_kv, d, T_q, S_kv, q_offset, causal, scale,
                        stream):
    return lib().gqa_attn_prefill_ex(q, k, v, o, lse, B, H_q, H_kv, d, T_q, S_kv, q_offset,
                                     causal, scale, stream)


def gqa_attn_prefill_partial(q, k, v, o_part, lse_part, B, H_q, H_kv, d, T_q, S_kv, q_offset,
                             key_offset, causal, scale, stream):
    return lib().gqa_attn_prefill_partial(q, k, v, o_part, lse_part, B, H_q, H_kv, d, T_q, S_kv,
                                          q_offset, key_offset, causal, scale, stream)


def gqa_attn_pick_num_splits(B, H_kv, S_max, num_sms):
    return lib().gqa_attn_pick_num_splits(B, H_kv, S_max, num_sms)


def gqa_attn_pick_num_splits_q8(B, H_kv, S_max, num_sms):
    return lib().gqa_attn_pick_num_splits_q8(B, H_kv, S_max, num_sms)


def gqa_attn_pick_num_splits_q4(B, H_kv, S_max, num_sms):
    return lib().gqa_attn_pick_num_splits_q4(B, H_kv, S_max, num_sms)


def gqa_attn_quantize_kv_q4(k, v, k_codes, v_codes, k_scales, v_scales, B, H_kv, S, d, stream):
    return lib().gqa_attn_quantize_kv_q4(k, v, k_codes, v_codes, k_scales, v_scales, B, H_kv, S,
                                         d, stream)


def gqa_attn_decode_q4(q, k_codes, v_codes, k_scales, v_scales, o, lse, seqlens, B, H_q, H_kv, d,
                       S_max, scale, num_splits, stream):
    return lib().gqa_attn_decode_q4(q, k_codes, v_codes, k_scales, v_scales, o, lse, seqlens, B,
                                    H_q, H_kv, d, S_max, scale, num_splits, stream)


def gqa_attn_decode_cluster_size(B, H_kv, num_splits, num_sms):
    return lib().gqa_attn_decode_cluster_size(B, H_kv, num_splits, num_sms)


def gqa_attn_split_bounds(S_max, num_splits, seqlen):
    """Returns (rc, [(start, end), ...])."""
    starts = (ctypes.c_int32 * max(num_splits, 1))()
    ends = (ctypes.c_int32 * max(num_splits, 1))()
    rc = lib().gqa_attn_split_bounds(S_max, num_splits, seqlen, starts, ends)
    return rc, [(starts[i], ends[i]) for i in range(max(num_splits, 0))] if rc == 0 else []


def gqa_attn_tile_class(qs, qe, ks, ke):
    return lib().gqa_attn_tile_class(qs, qe, ks, ke)


def gqa_attn_prefill_tile_counts(T_q, S_kv, q_offset, causal):
    """Returns (rc, n_past, n_partial, n_future)."""
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    rc = lib().gqa_attn_prefill_tile_counts(T_q, S_kv, q_offset, causal, ctypes.byref(a),
                                            ctypes.byref(b), ctypes.byref(c))
    return rc, a.value, b.value, c.value


def gqa_attn_prefill_block_m():
    return lib().gqa_attn_prefill_block_m()


def gqa_attn_prefill_block_n():
    return lib().gqa_attn_prefill_block_n()


def gqa_attn_prefill_schedule(B, H_q, H_kv, d, T_q, S_kv, q_offset, causal, num_ctas,
                              item_cap=12288):
    """Returns (rc, per-CTA item lists); rc = 0 (closed-form order) gives []."""
    off = (ctypes.c_int32 * (num_ctas + 1))()
    items = (ctypes.c_int32 * max(1, item_cap))()
    rc = lib().gqa_attn_prefill_schedule(B, H_q, H_kv, d, T_q, S_kv, q_offset, causal, num_ctas,
                                         off, items, item_cap)
    if rc <= 0:
        return rc, []
    return rc, [list(items[off[c]:off[c + 1]]) for c in range(num_ctas)]


def gqa_attn_check(stream=None):
    return lib().gqa_attn_check(stream)


def gqa_attn_debug_inject_timeout(launches):
    return lib().gqa_attn_debug_inject_timeout(launches)


def gqa_attn_debug_prefill_order(budget_bytes):
    return lib().gqa_attn_debug_prefill_order(budget_bytes)


def gqa_attn_debug_tile_counts(clear=False, L=None):
    """Returns (rc, [all_past, partial, all_future]) from ``L`` (default: the
    product library, whose non-debug build returns GQA_ERR_UNSUPPORTED)."""
    c = (ctypes.c_int64 * 3)()
    rc = (L or lib()).gqa_attn_debug_tile_counts(c, 1 if clear else 0)
    return rc, [c[0], c[1], c[2]]


def strerror(code: int) -> str:
    return lib().gqa_attn_strerror(code).decode()


def gqa_attn_version():
    return lib().gqa_attn_version()


# ---- torch conveniences -----------------------------------------------------


def _stream_ptr(stream=None):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_cuda_bf16(name, t, ndim):
    import torch

    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor, got {tuple(t.shape)}")


def decode(q, k, v, seqlens=None, *, num_splits: int = 0, scale: float | None = None,
           out=None, lse=None, stream=None, workspace=None):
    """Split-KV decode. q [B,H_q,d], k/v [B,H_kv,S_max,d] bf16 CUDA; seqlens int32 [B] or None.

    Returns (o [B,H_q,d] bf16, lse [B,H_q] fp32). With ``workspace`` (a uint8
    CUDA tensor) the call goes through gqa_attn_decode_ws.
    """
    import torch

    _check_cuda_bf16("q", q, 3)
    _check_cuda_bf16("k", k, 4)
    _check_cuda_bf16("v", v, 4)
    B, H_q, d = q.shape
    H_kv, S_max = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k, v must be [B, H_kv, S_max, d] matching q")
    if seqlens is not None and (seqlens.dtype != torch.int32 or not seqlens.is_cuda
                                or seqlens.numel() != B):
        raise TypeError("seqlens must be an int32 CUDA tensor of B elements")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = _stream_ptr(stream)
    if workspace is None:
        rc = gqa_attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(seqlens),
                             B, H_q, H_kv, d, S_max, sc, num_splits, st)
    else:
        rc = gqa_attn_decode_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                _ptr(seqlens), B, H_q, H_kv, d, S_max, sc, num_splits,
                                _ptr(workspace), workspace.numel(), st)
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_decode")
    return out, lse


def gqa_attn_decode_partial(q, k, v, o_part, lse_part, seqlens, B, H_q, H_kv, d, S_max, scale,
                            num_splits, stream):
    return lib().gqa_attn_decode_partial(q, k, v, o_part, lse_part, seqlens, B, H_q, H_kv, d,
                                         S_max, scale, num_splits, stream)


def gqa_attn_merge(o_parts, lse_parts, o, lse, R, rows, d, stream):
    return lib().gqa_attn_merge(o_parts, lse_parts, o, lse, R, rows, d, stream)


def decode_partial(q, k, v, seqlens=None, *, num_splits: int = 0, scale: float | None = None,
                   out=None, lse=None, stream=None):
    """Decode over one key slice with fp32 output for ``merge``: q [B,H_q,d],
    k/v [B,H_kv,S_slice,d] bf16 CUDA. Returns (o fp32 [B,H_q,d], lse [B,H_q])."""
    import torch

    _check_cuda_bf16("q", q, 3)
    _check_cuda_bf16("k", k, 4)
    _check_cuda_bf16("v", v, 4)
    B, H_q, d = q.shape
    H_kv, S_max = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k, v must be [B, H_kv, S, d] matching q")
    if seqlens is not None and (seqlens.dtype != torch.int32 or not seqlens.is_cuda
                                or seqlens.numel() != B):
        raise TypeError("seqlens must be an int32 CUDA tensor of B elements")
    if out is None:
        out = torch.empty((B, H_q, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = gqa_attn_decode_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(seqlens),
                                 B, H_q, H_kv, d, S_max, sc, num_splits, _stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_decode_partial")
    return out, lse


def merge(o_parts, lse_parts, *, out=None, lse=None, stream=None):
    """Log-sum-exp merge of R partials: o_parts fp32 [R, ..., d], lse_parts
    fp32 [R, ...] (CUDA, contiguous). Returns (o bf16 [..., d], lse [...])."""
    import torch

    if (o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32 or not o_parts.is_cuda
            or not o_parts.is_contiguous() or not lse_parts.is_contiguous()
            or tuple(o_parts.shape[:-1]) != tuple(lse_parts.shape)):
        raise ValueError("o_parts [R, ..., d] and lse_parts [R, ...] must be contiguous fp32 CUDA")
    R, d = o_parts.shape[0], o_parts.shape[-1]
    rows = lse_parts[0].numel()
    if out is None:
        out = torch.empty(tuple(o_parts.shape[1:]), dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty(tuple(lse_parts.shape[1:]), dtype=torch.float32, device=o_parts.device)
    rc = gqa_attn_merge(_ptr(o_parts), _ptr(lse_parts), _ptr(out), _ptr(lse), R, rows, d,
                        _stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_merge")
    return out, lse


def gqa_attn_ring_append(k_cache, v_cache, k_new, v_new, positions, B, H_kv, d, capacity, n_sink,
                         stream):
    return lib().gqa_attn_ring_append(k_cache, v_cache, k_new, v_new, positions, B, H_kv, d,
                                      capacity, n_sink, stream)


def gqa_attn_decode_ring(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, capacity, n_sink, scale,
                         num_splits, stream):
    return lib().gqa_attn_decode_ring(q, k, v, o, lse, seqlens, B, H_q, H_kv, d, capacity,
                                      n_sink, scale, num_splits, stream)


def gqa_attn_quantize_kv_q8(k, v, k_codes, v_codes, k_scales, v_scales, B, H_kv, S, d, stream):
    return lib().gqa_attn_quantize_kv_q8(k, v, k_codes, v_codes, k_scales, v_scales, B, H_kv, S,
                                         d, stream)


def gqa_attn_decode_q8(q, k_codes, v_codes, k_scales, v_scales, o, lse, seqlens, B, H_q, H_kv, d,
                       S_max, scale, num_splits, stream):
    return lib().gqa_attn_decode_q8(q, k_codes, v_codes, k_scales, v_scales, o, lse, seqlens, B,
                                    H_q, H_kv, d, S_max, scale, num_splits, stream)


def quantize_kv_q8(k, v, *, stream=None):
    """INT8 cache from a bf16 cache k, v [B,H_kv,S,d] (CUDA): returns
    (k_codes [B,H_kv,S,d], v_codes [B,H_kv,d,S] as uint8 bytes code + 128,
    k_scales, v_scales [B,H_kv,S] fp32)."""
    import torch

    _check_cuda_bf16("k", k, 4)
    _check_cuda_bf16("v", v, 4)
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    B, H_kv, S, d = k.shape
    kc = torch.empty((B, H_kv, S, d), dtype=torch.uint8, device=k.device)
    vc = torch.empty((B, H_kv, d, S), dtype=torch.uint8, device=k.device)
    ks = torch.empty((B, H_kv, S), dtype=torch.float32, device=k.device)
    vs = torch.empty_like(ks)
    rc = gqa_attn_quantize_kv_q8(_ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), B, H_kv,
                                 S, d, _stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_quantize_kv_q8")
    return kc, vc, ks, vs


def decode_q8(q, k_codes, v_codes, k_scales, v_scales, seqlens=None, *, num_splits: int = 0,
              scale: float | None = None, out=None, lse=None, stream=None):
    """Split-KV decode over an INT8 cache (layouts as ``quantize_kv_q8``).
    Returns (o [B,H_q,d] bf16, lse [B,H_q] fp32)."""
    import torch

    _check_cuda_bf16("q", q, 3)
    B, H_q, d = q.shape
    H_kv, S_max = k_codes.shape[1], k_codes.shape[2]
    if (k_codes.dtype != torch.uint8 or v_codes.dtype != torch.uint8
            or k_codes.shape != (B, H_kv, S_max, d) or v_codes.shape != (B, H_kv, d, S_max)):
        raise ValueError("k_codes [B,H_kv,S,d] and v_codes [B,H_kv,d,S] must be uint8")
    for nm, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        if t.dtype != torch.float32 or t.shape != (B, H_kv, S_max) or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous fp32 [B, H_kv, S] tensor")
    if seqlens is not None and (seqlens.dtype != torch.int32 or not seqlens.is_cuda
                                or seqlens.numel() != B):
        raise TypeError("seqlens must be an int32 CUDA tensor of B elements")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = gqa_attn_decode_q8(_ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales),
                            _ptr(v_scales), _ptr(out), _ptr(lse), _ptr(seqlens), B, H_q, H_kv, d,
                            S_max, sc, num_splits, _stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_decode_q8")
    return out, lse


def quantize_kv_q4(k, v, *, stream=None):
    """INT4 cache from a bf16 cache k, v [B,H_kv,S,d] (CUDA): returns
    (k_codes [B,H_kv,S,d/2], v_codes [B,H_kv,d,S/2] as uint8, two nibbles
    code + 8 per byte, k_scales, v_scales [B,H_kv,S] fp32)."""
    import torch

    _check_cuda_bf16("k", k, 4)
    _check_cuda_bf16("v", v, 4)
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    B, H_kv, S, d = k.shape
    kc = torch.empty((B, H_kv, S, d // 2), dtype=torch.uint8, device=k.device)
    vc = torch.empty((B, H_kv, d, S // 2), dtype=torch.uint8, device=k.device)
    ks = torch.empty((B, H_kv, S), dtype=torch.float32, device=k.device)
    vs = torch.empty_like(ks)
    rc = gqa_attn_quantize_kv_q4(_ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), B, H_kv,
                                 S, d, _stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_quantize_kv_q4")
    return kc, vc, ks, vs


def decode_q4(q, k_codes, v_codes, k_scales, v_scales, seqlens=None, *, num_splits: int = 0,
              scale: float | None = None, out=None, lse=None, stream=None):
    """Split-KV decode over an INT4 cache (layouts as ``quantize_kv_q4``).
    Returns (o [B,H_q,d] bf16, lse [B,H_q] fp32)."""
    import torch

    _check_cuda_bf16("q", q, 3)
    B, H_q, d = q.shape
    H_kv, S_max = k_codes.shape[1], k_codes.shape[2]
    if (k_codes.dtype != torch.uint8 or v_codes.dtype != torch.uint8
            or k_codes.shape != (B, H_kv, S_max, d // 2)
            or v_codes.shape != (B, H_kv, d, S_max // 2)):
        raise ValueError("k_codes [B,H_kv,S,d/2] and v_codes [B,H_kv,d,S/2] must be uint8")
    for nm, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        if t.dtype != torch.float32 or t.shape != (B, H_kv, S_max) or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous fp32 [B, H_kv, S] tensor")
    if seqlens is not None and (seqlens.dtype != torch.int32 or not seqlens.is_cuda
                                or seqlens.numel() != B):
        raise TypeError("seqlens must be an int32 CUDA tensor of B elements")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = gqa_attn_decode_q4(_ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales),
                            _ptr(v_scales), _ptr(out), _ptr(lse), _ptr(seqlens), B, H_q, H_kv, d,
                            S_max, sc, num_splits, _stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_decode_q4")
    return out, lse


def ring_append(k_cache, v_cache, k_new, v_new, positions, *, n_sink: int, stream=None):
    """Writes each row's newest token into its ring slot. k_cache/v_cache
    [B,H_kv,capacity,d] bf16 CUDA; k_new/v_new [B,H_kv,d]; positions int32 [B]
    (the new token's index in its row)."""
    import torch

    _check_cuda_bf16("k_cache", k_cache, 4)
    _check_cuda_bf16("v_cache", v_cache, 4)
    _check_cuda_bf16("k_new", k_new, 3)
    _check_cuda_bf16("v_new", v_new, 3)
    B, H_kv, capacity, d = k_cache.shape
    if v_cache.shape != k_cache.shape or k_new.shape != (B, H_kv, d) or v_new.shape != k_new.shape:
        raise ValueError("k_new, v_new must be [B, H_kv, d] matching the caches")
    if positions.dtype != torch.int32 or not positions.is_cuda or positions.numel() != B:
        raise TypeError("positions must be an int32 CUDA tensor of B elements")
    rc = gqa_attn_ring_append(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                              _ptr(positions), B, H_kv, d, capacity, n_sink, _stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_ring_append")


def decode_ring(q, k, v, seqlens, *, n_sink: int, num_splits: int = 0,
                scale: float | None = None, out=None, lse=None, stream=None):
    """Decode over a ring-buffer cache with attention sinks: k/v
    [B,H_kv,capacity,d]; seqlens int32 [B] counts every token each row has
    produced (it may exceed capacity). Returns (o, lse) as ``decode``."""
    import torch

    _check_cuda_bf16("q", q, 3)
    _check_cuda_bf16("k", k, 4)
    _check_cuda_bf16("v", v, 4)
    B, H_q, d = q.shape
    H_kv, capacity = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k, v must be [B, H_kv, capacity, d] matching q")
    if seqlens.dtype != torch.int32 or not seqlens.is_cuda or seqlens.numel() != B:
        raise TypeError("seqlens must be an int32 CUDA tensor of B elements")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = gqa_attn_decode_ring(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(seqlens),
                              B, H_q, H_kv, d, capacity, n_sink, sc, num_splits,
                              _stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_decode_ring")
    return out, lse


def prefill(q, k, v, *, q_offset: int = 0, causal: bool = True, scale: float | None = None,
            out=None, lse=None, stream=None):
    """Causal (or full) prefill. q [B,H_q,T_q,d], k/v [B,H_kv,S_kv,d] bf16 CUDA.

    Returns (o [B,H_q,T_q,d] bf16, lse [B,H_q,T_q] fp32).
    """
    import torch

    _check_cuda_bf16("q", q, 4)
    _check_cuda_bf16("k", k, 4)
    _check_cuda_bf16("v", v, 4)
    B, H_q, T_q, d = q.shape
    H_kv, S_kv = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k, v must be [B, H_kv, S_kv, d] matching q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H_q, T_q), dtype=torch.float32, device=q.device)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = gqa_attn_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H_q, H_kv, d,
                             T_q, S_kv, q_offset, 1 if causal else 0, sc, _stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_prefill")
    return out, lse


def prefill_partial(q, k, v, *, q_offset: int = 0, key_offset: int = 0, causal: bool = True,
                    scale: float | None = None, out=None, lse=None, stream=None):
    """Prefill against one slice of the keys (global positions key_offset + j),
    O in fp32 for ``merge``. q [B,H_q,T_q,d], k/v [B,H_kv,S_slice,d] bf16 CUDA.
    Returns (o fp32 [B,H_q,T_q,d], lse [B,H_q,T_q])."""
    import torch

    _check_cuda_bf16("q", q, 4)
    _check_cuda_bf16("k", k, 4)
    _check_cuda_bf16("v", v, 4)
    B, H_q, T_q, d = q.shape
    H_kv, S_kv = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k, v must be [B, H_kv, S_slice, d] matching q")
    if out is None:
        out = torch.empty((B, H_q, T_q, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H_q, T_q), dtype=torch.float32, device=q.device)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    rc = gqa_attn_prefill_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H_q, H_kv,
                                  d, T_q, S_kv, q_offset, key_offset, 1 if causal else 0, sc,
                                  _stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_prefill_partial")
    return out, lse


def check(stream=None):
    """Synchronises the stream and raises if the device status word is set."""
    rc = gqa_attn_check(_stream_ptr(stream))
    if rc != GQA_OK:
        raise GqaError(rc, "gqa_attn_check")
