// common.cuh -- host-side helpers shared by the entry points: error words, tensor maps.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/blink.h"

namespace blink {

// Layout of the first 256 bytes of every workspace: the device error word, then reserved space.
struct WorkspaceHeader {
    int32_t error;      // 0 = fine, else a blink_status latched by a kernel
    int32_t reserved[63];
};
static_assert(sizeof(WorkspaceHeader) == 256, "workspace header is 256 bytes");

constexpr size_t kHeaderBytes = sizeof(WorkspaceHeader);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Encodes a rank-3 tiled tensor map over a bf16 tensor with dims {d0 (contiguous), d1, d2},
// byte strides {stride1, stride2}, box {b0, b1, b2}, 128-byte swizzle, zero fill out of bounds.
// Returns false if the driver entry point is missing or the driver rejects the map.
bool encode_tmap_3d_bf16(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace blink
