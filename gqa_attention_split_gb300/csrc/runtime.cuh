// Host-side runtime shared by the entry points: per-device status word,
// per-(device, stream) workspace cache, SM count, TMA descriptor encoding.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gqa {

// Device pointer to the status word of the current device (allocated and
// zeroed on first use). Returns nullptr if that fails.
unsigned* status_word();

// Current device's SM count (cached), or a negative value on failure.
int num_sms();
// Test hook for failure reporting: the next n launches (decode or prefill)
// each make their first block withhold one copy (set / take one).
void set_injected_timeouts(int launches);
bool take_injected_timeout();

// Library-owned workspace of at least `bytes` for (current device, stream).
// Grows with stream-ordered allocation; returns nullptr on failure or when
// it would have to grow while `stream` is being captured.
void* stream_workspace(cudaStream_t stream, size_t bytes);

// Encodes a 3-D bf16 tensor map over a [outer, rows, inner] row-major tensor
// with a {box_inner, box_rows, 1} box and the given swizzle. Returns
// cudaSuccess or the error that describes the failure.
// Tiled tensor map over a dense array: dims[0] is innermost, strides follow
// from the dims (elem_bytes each).
cudaError_t encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes,
                        uint32_t rank, const void* base, const uint64_t* dims, const uint32_t* box,
                        CUtensorMapSwizzle swizzle);
cudaError_t encode_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t inner,
                                uint64_t rows, uint64_t outer, uint32_t box_inner,
                                uint32_t box_rows, CUtensorMapSwizzle swizzle);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace gqa
