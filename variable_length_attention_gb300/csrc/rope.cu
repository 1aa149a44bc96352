// rope.cu -- the rotary block-diagonal entry points' table packing and the
// backward's transposed-rotation pass.
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
// The block kernels rotate Q and K tiles in shared memory as they land (block.cu)
// from a packed table: pack_kernel turns the caller's fp32 cos/sin rows into one
// half2 (cos, sin) per pair, half the bytes the rotation has to read per tile.
// At head_dim 64 the backward's dQ and dK, computed with respect to the rotated
// rows, go back through the transposed rotation in one streaming pass over their
// rows (rope_kernel, in place), at the HBM copy rate; at head_dim 128 the
// backward kernel's epilogue does it.
//
// rope_kernel layout: rows of [rows, H, D] bf16, one warp per row at a time, each
// lane one 16-byte chunk of the first half of a head row together with its
// partner chunk of the second half (8 column pairs), for one or two tensors (dq
// and dk share the table reads).  Each warp walks a contiguous range of rows and
// finds the position of its first row by a binary search over the offsets.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "host.h"
#include "profile.h"
#include "ptx.cuh"
#include "rope.h"

namespace jfa {
namespace rope {

// x' = x c - sgn y s, y' = y c + sgn x s for the 8 pairs of one chunk (sgn = 1:
// the rotation, -1: its transpose), in fp32, rounded to bf16 once.
__device__ __forceinline__ void rotate_chunk(const uint4& xr, const uint4& yr, const float* c, const float* s,
                                             float sgn, uint4* xo, uint4* yo) {
  const uint32_t xi[4] = {xr.x, xr.y, xr.z, xr.w};
  const uint32_t yi[4] = {yr.x, yr.y, yr.z, yr.w};
  uint32_t xw[4], yw[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 u = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xi[e]));
    const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&yi[e]));
    const float s0 = sgn * s[2 * e], s1 = sgn * s[2 * e + 1];
    xw[e] = pack_bf16(u.x * c[2 * e] - v.x * s0, u.y * c[2 * e + 1] - v.y * s1);
    yw[e] = pack_bf16(v.x * c[2 * e] + u.x * s0, v.y * c[2 * e + 1] + u.y * s1);
  }
  *xo = make_uint4(xw[0], xw[1], xw[2], xw[3]);
  *yo = make_uint4(yw[0], yw[1], yw[2], yw[3]);
}

template <int D>
__global__ void __launch_bounds__(256, 4) rope_kernel(const __nv_bfloat16* in0, __nv_bfloat16* out0,
                                                   const __nv_bfloat16* in1, __nv_bfloat16* out1,
                                                   const float* __restrict__ cosv, const float* __restrict__ sinv,
                                                   const int32_t* __restrict__ offsets, int batch, long rows, int H,
                                                   float sgn) {
  constexpr int CH = D / 16;  // 16-byte chunks in half a head row
  const int lane = threadIdx.x & 31;
  const long warp = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long n_warps = (static_cast<long>(gridDim.x) * blockDim.x) >> 5;
  const long per = (rows + n_warps - 1) / n_warps;
  long r = warp * per;
  const long r_end = min(rows, r + per);
  if (r >= r_end) return;
  // the sequence of row r: the largest b < batch with offsets[b] <= r
  int b = 0;
  for (int n = batch; n > 1;) {
    const int half = n >> 1;
    b = (__ldg(offsets + b + half) <= r) ? b + half : b;
    n -= half;
  }
  long seq_start = __ldg(offsets + b), seq_end = __ldg(offsets + b + 1);
  const int items = H * CH;  // (head, chunk) pairs of a row
  for (; r < r_end; ++r) {
    while (r >= seq_end) {  // the next non-empty sequence
      ++b;
      seq_start = seq_end;
      seq_end = __ldg(offsets + b + 1);
    }
    const long pos = r - seq_start;
    for (int it = lane; it < items; it += 32) {
      const int h = it / CH, j = it % CH;
      const float* cr = cosv + pos * (D / 2) + 8 * j;
      const float* sr = sinv + pos * (D / 2) + 8 * j;
      const float4 c0 = __ldg(reinterpret_cast<const float4*>(cr)), c1 = __ldg(reinterpret_cast<const float4*>(cr + 4));
      const float4 s0 = __ldg(reinterpret_cast<const float4*>(sr)), s1 = __ldg(reinterpret_cast<const float4*>(sr + 4));
      const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      const size_t at = (static_cast<size_t>(r) * H + h) * D + 8 * j;
      const uint4 x0 = *reinterpret_cast<const uint4*>(in0 + at);
      const uint4 y0 = *reinterpret_cast<const uint4*>(in0 + at + D / 2);
      uint4 x1 = make_uint4(0, 0, 0, 0), y1 = x1;
      if (in1 != nullptr) {
        x1 = *reinterpret_cast<const uint4*>(in1 + at);
        y1 = *reinterpret_cast<const uint4*>(in1 + at + D / 2);
      }
      uint4 xo, yo;
      rotate_chunk(x0, y0, c, s, sgn, &xo, &yo);
      *reinterpret_cast<uint4*>(out0 + at) = xo;
      *reinterpret_cast<uint4*>(out0 + at + D / 2) = yo;
      if (in1 != nullptr) {
        rotate_chunk(x1, y1, c, s, sgn, &xo, &yo);
        *reinterpret_cast<uint4*>(out1 + at) = xo;
        *reinterpret_cast<uint4*>(out1 + at + D / 2) = yo;
      }
    }
  }
}

// (cos, sin) -> one half2 per pair: the block kernels' rotation reads 4 bytes
// per pair instead of 8 (fp16 keeps 11 significant bits of values in [-1, 1],
// finer than the bf16 rounding of the rotated rows that follows)
__global__ void pack_kernel(const float* __restrict__ cosv, const float* __restrict__ sinv, uint32_t* __restrict__ tab,
                            long n) {
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const __half2 h = __floats2half2_rn(cosv[i], sinv[i]);
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

int launch_rope(const RopeArgs& a, int num_sms) {
  if (a.rows == 0) return JFA_OK;
  // one wave of 4 blocks of 8 warps per SM: each warp's row range is long
  // enough to amortise its position search, and with 4 KB of loads in flight per
  // warp and row, 32 warps per SM keep HBM busy
  const long warps = std::min<long>(static_cast<long>(num_sms) * 32, a.rows);
  const int grid = static_cast<int>((warps + 7) / 8);
  ProfileScope prof(kKindRope, a.stream);
  const auto* i0 = static_cast<const __nv_bfloat16*>(a.in0);
  const auto* i1 = static_cast<const __nv_bfloat16*>(a.in1);
  auto* o0 = static_cast<__nv_bfloat16*>(a.out0);
  auto* o1 = static_cast<__nv_bfloat16*>(a.out1);
  const float sgn = a.transpose ? -1.0f : 1.0f;
  if (a.D == 128)
    rope::rope_kernel<128><<<grid, 256, 0, a.stream>>>(i0, o0, i1, o1, a.rope_cos, a.rope_sin, a.offsets_dev, a.batch,
                                                       a.rows, a.H, sgn);
  else
    rope::rope_kernel<64><<<grid, 256, 0, a.stream>>>(i0, o0, i1, o1, a.rope_cos, a.rope_sin, a.offsets_dev, a.batch,
                                                      a.rows, a.H, sgn);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

}  // namespace jfa
