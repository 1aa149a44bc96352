// rope.h -- launcher of the rotary position embedding pass (see rope.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace jfa {

struct RopeArgs {
  const void* in0;  // [rows, H, D] bf16
  void* out0;       // may equal in0 (in place)
  const void* in1;  // a second tensor with the same rows, or null
  void* out1;
  const float *rope_cos, *rope_sin;  // [positions, D/2] fp32
  const int32_t* offsets_dev;        // [batch+1]
  int batch;
  long rows;
  int H, D;
  int transpose;  // 1: the transposed rotation (gradients back to the unrotated rows)
  cudaStream_t stream;
};

int launch_rope(const RopeArgs& a, int num_sms);

}  // namespace jfa
