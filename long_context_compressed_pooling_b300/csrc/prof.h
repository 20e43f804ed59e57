// Per-kernel launch timing with CUDA events (off by default). When enabled through
// csa_profiler_enable(), every kernel launch of the library is bracketed by two events recorded
// on the launch stream; csa_profiler_collect() sums the elapsed times per kernel name.
#pragma once

#include <cuda_runtime.h>

namespace csa {

bool prof_enabled();
int prof_begin(cudaStream_t stream, const char* name);  // returns a slot or -1
void prof_end(cudaStream_t stream, int slot);

struct ProfScope {
  cudaStream_t st;
  int slot;
  ProfScope(cudaStream_t s, const char* name) : st(s), slot(prof_enabled() ? prof_begin(s, name) : -1) {}
  ~ProfScope() {
    if (slot >= 0) prof_end(st, slot);
  }
};

}  // namespace csa
