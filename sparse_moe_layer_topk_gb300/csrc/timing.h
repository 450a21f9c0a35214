// RAII bracket of one kernel launch for the optional per-kernel timing.
#pragma once

#include <cuda_runtime.h>

namespace moe {

class LaunchTimer {
 public:
  LaunchTimer(const char* name, cudaStream_t st);
  ~LaunchTimer();
  LaunchTimer(const LaunchTimer&) = delete;
  LaunchTimer& operator=(const LaunchTimer&) = delete;

 private:
  const char* name_;
  cudaStream_t st_;
  void* a_ = nullptr;
  void* b_ = nullptr;
};

}  // namespace moe
