// profile.h -- RAII bracket that records a CUDA event pair around a launch when
// kernel timing is enabled (gdn_profile_enable).
#pragma once
#include <cuda_runtime.h>

namespace gdn {
class ProfScope {
  public:
    ProfScope(const char *name, cudaStream_t st);
    ~ProfScope();
    ProfScope(const ProfScope &) = delete;
    ProfScope &operator=(const ProfScope &) = delete;

  private:
    const char *name_;
    cudaStream_t st_;
    cudaEvent_t a_;
};
}  // namespace gdn
