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

// The table the block kernels rotate with: entry [p, i] = (cos, sin) of pair i
// at position p as one half2, for positions [0, positions).
int launch_rope_pack(const float* rope_cos, const float* rope_sin, uint32_t* tab, long positions, int half_d,
                     cudaStream_t stream);

}  // namespace jfa
