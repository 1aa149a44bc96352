// rope.cu -- the packed rotation table of the rotary block-diagonal entry
// points.
//
// "TLX Block Attention" (introduction) reports its block kernel 3.5x faster
// than the unfused baseline once the rotary embedding is fused into the
// attention's post-processing, without stating the rotary convention.  The
// reading here is the rotate-half form: the position of a row is its index
// inside its sequence, and for i < D/2 the pair (x_i, x_{i+D/2}) of a q or k row
// at position p turns by the angle whose cosine and sine are the caller's table
// entries [p, i]:
//   forward:    (x_i, x_{i+D/2}) -> (x_i c - x_{i+D/2} s, x_{i+D/2} c + x_i s)
//   transposed: (g_i, g_{i+D/2}) -> (g_i c + g_{i+D/2} s, g_{i+D/2} c - g_i s)
// The transposed rotation carries a gradient with respect to the rotated rows
// back to the unrotated ones.
//
// The block kernels (block.cu) rotate Q and K tiles in shared memory as they
// land, and the backward's epilogue turns dQ and dK back by the transposed
// rotation, from a packed table that pack_kernel builds from the caller's fp32
// cos/sin rows: half the bytes, in the order the kernels' arithmetic takes them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "host.h"
#include "profile.h"
#include "ptx.cuh"
#include "rope.h"

namespace jfa {
namespace rope {

// The packed table: for each two pairs (2m, 2m + 1) of a row, one half2 of
// their cosines followed by one half2 of their sines, so that a kernel turns a
// word straight into the operand pair of its paired fp32 arithmetic and reads
// 4 bytes per pair instead of 8 (fp16 keeps 11 significant bits of values in
// [-1, 1], finer than the bf16 rounding of the rotated rows that follows).
// Word i of a row of half_d words: pairs 2 (i / 2) and 2 (i / 2) + 1, the sines
// when i is odd.
__global__ void pack_kernel(const float* __restrict__ cosv, const float* __restrict__ sinv, uint32_t* __restrict__ tab,
                            long n) {
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const float* src = (i & 1) ? sinv : cosv;
    const long at = i & ~1L;  // row * half_d + 2 m: the first of the two pairs
    const __half2 h = __floats2half2_rn(src[at], src[at + 1]);
    tab[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
}

}  // namespace rope

int launch_rope_pack(const float* rope_cos, const float* rope_sin, uint32_t* tab, long positions, int half_d,
                     cudaStream_t stream) {
  const long n = positions * half_d;
  if (n == 0) return JFA_OK;
  const int grid = static_cast<int>(std::min<long>((n + 255) / 256, 4096));
  ProfileScope prof(kKindRope, stream);
  rope::pack_kernel<<<grid, 256, 0, stream>>>(rope_cos, rope_sin, tab, n);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

}  // namespace jfa
