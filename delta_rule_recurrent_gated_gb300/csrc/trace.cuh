// trace.cuh -- RAII bracket of one kernel launch for the optional event trace.
#pragma once
#include <cuda_runtime.h>

namespace dr {
class TraceScope {
  public:
    TraceScope(const char* name, cudaStream_t st);
    ~TraceScope();
    TraceScope(const TraceScope&) = delete;
    TraceScope& operator=(const TraceScope&) = delete;

  private:
    cudaStream_t st_;
    int slot_;
};
}  // namespace dr
