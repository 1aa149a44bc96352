// rope.h -- launcher of the rotary table packing (see rope.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace jfa {

// The table the block kernels rotate with, half_d words per position for
// positions [0, positions): word 2m of row p holds cos of pairs 2m and 2m + 1
// at position p as one half2, word 2m + 1 their sines.
int launch_rope_pack(const float* rope_cos, const float* rope_sin, uint32_t* tab, long positions, int half_d,
                     cudaStream_t stream);

}  // namespace jfa
