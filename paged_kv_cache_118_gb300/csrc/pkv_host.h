// Host-side helpers shared by the pagedkv launchers.
#pragma once

#include <cstdint>

namespace pkv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace pkv
