// rc_layout.h -- where each element of the ring lives in device memory.
// Used by the kernels and by the host-side export (plain C++ for both).
//
// Per layer, per head, the ring of C slots is cut into T = ceil(C/128) tiles
// of 128 slots; slot s is row s % 128 of tile s / 128.  The padded slot count
// is Cpad = 128 T.
//   K codes : kc[L][H][T][128][D]  -- row = slot, D bytes, swizzled chunks
//   V codes : vt[L][H][T][D][128]  -- row = dim, 128 bytes (slots), swizzled
//   scales  : sk, sv [L][H][Cpad]  -- fp32, the slot's write-group scale
//   groups  : grp[L][Cpad]         -- compact write-group index, -1 = empty
// A tile is a contiguous block whose bytes are already in the swizzled
// shared-memory order that tcgen05 expects for a K-major operand, so one
// bulk copy brings it into shared memory ready for the MMA.
#pragma once
#include <cstdint>

#if defined(__CUDACC__)
#define RC_HD __host__ __device__ __forceinline__
#else
#define RC_HD inline
#endif

namespace rc {

constexpr int kTileSlots = 128;

// Byte offset of (row, col) in a [rows][D] 8-bit tile (D = 128: 128-byte
// swizzle, chunk ^= row % 8; D = 64: 64-byte swizzle, chunk ^= (row / 2) % 4).
RC_HD uint32_t ktile_off(uint32_t row, uint32_t col, int D) {
    uint32_t x = (D == 128) ? (row & 7u) : ((row >> 1) & 3u);
    return row * static_cast<uint32_t>(D) + ((((col >> 4) ^ x) << 4) | (col & 15u));
}

// Byte offset of (dim row, slot) in a [D][128] 8-bit tile with 128-byte swizzle.
RC_HD uint32_t vtile_off(uint32_t drow, uint32_t slot) {
    return drow * 128u + ((((slot >> 4) ^ (drow & 7u)) << 4) | (slot & 15u));
}

RC_HD int tiles_of(int C) { return (C + kTileSlots - 1) / kTileSlots; }

// The bf16 ring (RC_F_BF16_CACHE) keeps 2-byte elements in the same 128-slot
// tiles, each a K-major tcgen05 operand image with the 128-byte swizzle:
//   K tile  : [D/64 blocks][128 slots][128 B]: element (slot, dim) in block
//             dim / 64, 16-byte chunk ((dim % 64) / 8) ^ (slot % 8);
//   Vt tile : [2 halves][D dims][128 B]: element (dim, slot) in half slot / 64,
//             16-byte chunk ((slot % 64) / 8) ^ (dim % 8).
RC_HD uint32_t bktile_off(uint32_t slot, uint32_t dim) {
    const uint32_t byte = (dim & 63u) * 2u;
    return (dim >> 6) * (kTileSlots * 128u) + slot * 128u + ((((byte >> 4) ^ (slot & 7u)) << 4) | (byte & 15u));
}
RC_HD uint32_t bvtile_off(uint32_t drow, uint32_t slot, int D) {
    const uint32_t byte = (slot & 63u) * 2u;
    return (slot >> 6) * (static_cast<uint32_t>(D) * 128u) + drow * 128u +
           ((((byte >> 4) ^ (drow & 7u)) << 4) | (byte & 15u));
}

}  // namespace rc
