// Host-side runtime shared by the entry points: per-device status word,
// per-(device, stream) workspace cache, SM count, TMA descriptor encoding.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace gqa {

// Device address of the status word of the current device: a variable in
// this library's own device memory (zero at load; nothing is allocated),
// looked up once per device. Returns nullptr if that fails.
unsigned* status_word();

// Current device ordinal, or -1.
int current_device();

// Per-device "launch attributes already set" flags, one bit per device in
// `done`: function attributes such as the dynamic shared-memory limit apply
// to the device current when they are set, so each device needs its own.
// pending() is true until mark() ran for that device (always true for
// ordinals >= 64, which then set the attributes on every launch).
bool device_attrs_pending(const std::atomic<uint64_t>& done, int dev);
void device_attrs_mark(std::atomic<uint64_t>& done, int dev);

// Current device's SM count (cached), or a negative value on failure.
int num_sms();
// Test hook for failure reporting: the next n launches (decode or prefill)
// each make their first block withhold one copy (set / take one).
void set_injected_timeouts(int launches);
bool take_injected_timeout();

// Library-owned workspace of at least `bytes` for (current device, stream).
// Grows with stream-ordered allocation; a buffer it replaces is kept (never
// freed) because work captured earlier may still use it. Returns nullptr on
// failure or when it would have to grow while `stream` is being captured.
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
