// q4nx_checks.h -- argument checks shared by the C ABI's entry points
// (internal to libq4nx.so).  The "Q4NX chunks" section of the 1bit engine
// "NPU engine" page refuses an unknown chunk size or a tensor shorter than its
// layout needs; these checks add the tile-grid shape and 16-byte alignment.
#pragma once

#include <cstdint>

#include "../../include/q4nx.h"

namespace q4nx {

// Q4NX_OK, or Q4NX_E_SHAPE when rows / cols are not positive multiples of 32 /
// 256 or the tile count does not fit 31 bits.
int check_grid(int64_t rows, int64_t cols);

// Q4NX_OK, or the status of the first failing check of a weight: NULL
// pointer, unknown kind (or nonzero reserved field), shape, length, alignment.
int check_weight(const q4nx_weight* w);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace q4nx
