// Host-side helpers shared by the pagedkv launchers.
#pragma once

#include <cuda.h>

#include <cstdint>

namespace pkv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// TMA map of one cache.
//  kRowsPlain: 3-D view (D, KV head, slot), box D x 1 x box_rows.
//  kRowsSwizzled: 4-D view (64 elements, slot, KV head, D/64 lines), box
//    64 x box_rows x 1 x D/64 with the 128-byte swizzle: whole rows of box_rows
//    slots per copy, stored line-major.
//  kLineSwizzled: the same view with the box 64 x box_rows x 1 x 1: one
//    128-byte line of box_rows slots per copy, so that a tile's rows of one
//    line can sit contiguously (the layout tcgen05 operands are read in).
// Returns false if the encoder is missing or refuses the view.
enum CacheView { kRowsPlain = 0, kRowsSwizzled = 1, kLineSwizzled = 2 };
bool encode_cache_map(CUtensorMap* tm, const void* base, int D, int num_kv_heads, int64_t slots,
                      int box_rows, CacheView view);

}  // namespace pkv
