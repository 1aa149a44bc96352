// rope.h -- launcher of the rotary table packing (see rope.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace jfa {

// The table the block kernels rotate with: entry [p, i] = (cos, sin) of pair i
// at position p as one half2, for positions [0, positions).
int launch_rope_pack(const float* rope_cos, const float* rope_sin, uint32_t* tab, long positions, int half_d,
                     cudaStream_t stream);

}  // namespace jfa
