// check.cuh -- device-side index checks of the checked build.
//
// The library is also built as a checked variant (CR_DEVICE_CHECKS, into
// a separate directory) for tests: every kernel then verifies, before it
// touches memory, the index arithmetic its accesses rest on -- the chunk a
// vector falls in is a rank, its offset lies inside that rank's shard, a
// tile belongs to its tensor, and so on.  A violated check sets one bit of
// a device error word (one bit per kind of check) and skips the rest of the
// thread's work instead of trapping, so the context survives and the host
// can read the word (cr_check_word) after the launch.  In the normal build
// the checks compile to nothing.
#pragma once

namespace cr {

// Which check failed: one bit each.
enum CheckBit {
  kChkFoldChunk = 0,    // fold: chunk index, element range
  kChkFoldShard = 1,    // reduce-scatter: offset inside the shard
  kChkGather = 2,       // all-gather: source offset inside the shard
  kChkHsdp = 3,         // HSDP: shard / outer chunk / offset
  kChkFused = 4,        // fused buckets: tensor, tile, element
  kChkCopy = 5,         // bucket copies: range, source granule
  kChkFsdp = 6,         // FSDP step: chunk, state offset
  kChkFsdp2 = 7,        // FSDP2: parameter, tile, state offset
  kChkAccum = 8,        // accumulate: element range
  kChkSelfTest = 31     // set on purpose by cr_check_selftest
};

#if defined(CR_DEVICE_CHECKS)
extern __device__ unsigned int g_check_word;
#define CR_DCHECK(cond, bit)                                  \
  do {                                                        \
    if (!(cond)) {                                            \
      atomicOr(&::cr::g_check_word, 1u << (unsigned)(bit));   \
      return;                                                 \
    }                                                         \
  } while (0)
#else
#define CR_DCHECK(cond, bit) \
  do {                       \
  } while (0)
#endif

}  // namespace cr
