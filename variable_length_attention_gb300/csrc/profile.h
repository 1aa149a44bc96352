// profile.h -- RAII event bracket around one kernel launch (see profile.cu).
#pragma once
#include <cuda_runtime.h>

namespace jfa {

// Kernel kinds, as numbered by jfa_profile_read().
enum KernelKind : int {
  kKindFwd = 0,
  kKindBwdPrep = 1,
  kKindBwdMain = 2,
  kKindDqConvert = 3,
  kKindBlockFwd = 4,
  kKindBlockBwd = 5,
  kKindFill = 6,
  kKindTopk = 7,
  kKindRope = 8,
  kNumKernelKinds = 9
};

class ProfileScope {
 public:
  ProfileScope(int kind, cudaStream_t stream);
  ~ProfileScope();
  ProfileScope(const ProfileScope&) = delete;
  ProfileScope& operator=(const ProfileScope&) = delete;

 private:
  int kind_;
  cudaStream_t stream_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
  bool active_ = false;
};

}  // namespace jfa
