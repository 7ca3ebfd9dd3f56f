// pa_host.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pa {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

inline int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// True when the environment asks for validating mode (PA_VALIDATE=1).
bool validating();

// Maps the last launch error to a status, clearing it.
pa_status launch_status();

}  // namespace pa
