// Host-side helpers shared by the pagedkv launchers.
#pragma once

#include <cuda.h>

#include <cstdint>

namespace pkv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// TMA map of one cache. swizzled = false: 3-D view (D, KV head, slot), box
// D x 1 x box_rows. swizzled = true: 4-D view (64 elements, D/64, KV head,
// slot), box 64 x D/64 x 1 x box_rows stored with the 128-byte swizzle (whole
// rows of box_rows slots per copy). Returns false if the encoder is missing or
// refuses the view.
bool encode_cache_map(CUtensorMap* tm, const void* base, int D, int num_kv_heads, int64_t slots,
                      int box_rows, bool swizzled);

}  // namespace pkv
