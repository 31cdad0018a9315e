// Optional per-kernel timing: when enabled (pisa_profile_start), every kernel launch of
// the library is bracketed by two CUDA events recorded on the launch stream.
#pragma once

#include <cuda_runtime.h>

namespace pisa {

class ProfScope {
 public:
  ProfScope(cudaStream_t st, const char* name);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  cudaStream_t st_;
  int slot_;
};

}  // namespace pisa
