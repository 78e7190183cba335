// Bits of the per-device error word that kernels OR into global memory.
#pragma once

namespace jfa {
enum : int {
  kErrTimeout = 1,      // a bounded wait ran out
  kErrBadOffsets = 2,   // offsets[0] != 0, decreasing offsets, or a length above max_len
  kErrCapacity = 4,     // work list larger than the host-sized capacity
  kErrSmemAlign = 8,    // dynamic shared memory not 1024-byte aligned
  kErrBadBlocks = 16,   // a block-sparse list: count above the key tiles, or not ascending
};
}  // namespace jfa
