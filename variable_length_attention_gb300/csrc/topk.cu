// topk.cu -- first stage of the block-sparse forward: block means and the
// top-k key blocks of every query block.
//
// The aixai.ru summary ("MXFP8 and sparsity") describes a two-stage variant for
// long histories: a cheap kernel averages blocks of Q and K and picks the top-k
// most relevant key blocks, and the attention kernel then attends over those
// blocks only.  Here a query block is 256 rows (the forward kernel's unit: its
// two 128-row tiles share every K/V block they load) and a key block is 128 keys
// (the forward's K/V block); a block's mean is over the rows it really has; the
// score of (query block, key block) is mean query . mean key, with key/value
// head h / (H / Hkv); the k highest scores win, ties to the lower block index.
//
// Kernels, in launch order:
//   block_mean_kernel  one CTA per block: the fp32 mean of its rows (query
//                      blocks, then key blocks), each of its 8 warps loading 32
//                      rows at once, partial sums added in shared memory
//   select_kernel      one CTA per query block: the scores against every key
//                      block of its sequence (the warps share them), then k
//                      rounds of a warp arg-max;
//                      the chosen block indices are written in ascending order,
//                      -1 after the last one
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "host.h"
#include "plan.h"
#include "profile.h"
#include "ptx.cuh"
#include "topk.h"

namespace jfa {
namespace topk {

// One block of rows to average: rows [row0, row0 + n) of head `head` in a
// [rows, heads, D] tensor; the mean goes to out[D].
struct MeanTask {
  int row0, n, head, tensor;  // tensor 0: q, 1: k
};

// One CTA per block: warp w sums rows [32 w, 32 w + 32) of it with all 32 rows'
// loads in flight at once (a block has at most 256 rows, so one round), and the
// eight partial sums are added in shared memory.  Every row is read once, so
// the loads allocate no L1 line.  (Selection call: a warp per block walking its
// rows 32 at a time took 67 us, 55 us without L1 allocation; this, 49 us.)
constexpr int kMeanWarps = 8;
template <int D>
__global__ void __launch_bounds__(32 * kMeanWarps) block_mean_kernel(const __nv_bfloat16* __restrict__ q,
                                                                      const __nv_bfloat16* __restrict__ k, int H,
                                                                      int Hkv, const int4* __restrict__ tasks,
                                                                      float* __restrict__ out) {
  constexpr int PER = D / 32;  // columns per lane: 4 (D = 128) or 2 (D = 64)
  constexpr int U = 32;        // rows per warp
  __shared__ float part[kMeanWarps][D];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int4 t = tasks[blockIdx.x];
  const __nv_bfloat16* base = t.w == 0 ? q : k;
  const int heads = t.w == 0 ? H : Hkv;
  const size_t stride = static_cast<size_t>(heads) * D;
  const int r0 = U * warp;
  const __nv_bfloat16* row0 = base + (static_cast<size_t>(t.x + r0) * heads + t.z) * D + lane * PER;
  uint2 raw[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    raw[u] = make_uint2(0u, 0u);  // bf16 zeros past the block's end
    if (r0 + u < t.y) {
      const __nv_bfloat16* row = row0 + static_cast<size_t>(u) * stride;
      if constexpr (PER == 4)
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(raw[u].x), "=r"(raw[u].y) : "l"(row));
      else
        asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(raw[u].x) : "l"(row));
    }
  }
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[u].x));
    acc[0] += a.x;
    acc[1] += a.y;
    if constexpr (PER == 4) {
      const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[u].y));
      acc[2] += c.x;
      acc[3] += c.y;
    }
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) part[warp][lane * PER + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kMeanWarps; ++w) sum += part[w][threadIdx.x];
    const float inv = t.y > 0 ? 1.0f / static_cast<float>(t.y) : 0.f;
    out[static_cast<size_t>(blockIdx.x) * D + threadIdx.x] = sum * inv;
  }
}

// One query block per CTA of kSelWarps warps: its mean (row x of the means),
// the mean of its sequence's key block 0 for its key/value head (row y) and the
// number of key blocks (z).  The warps share the dot products (block n goes to
// warp n % kSelWarps, eight blocks' means loaded at a time), then warp 0 picks.
constexpr int kSelWarps = 4;
template <int D>
__global__ void __launch_bounds__(32 * kSelWarps) select_kernel(const float* __restrict__ means,
                                                                 const int4* __restrict__ sel_tasks, int topk,
                                                                 int32_t* __restrict__ selection) {
  extern __shared__ float sc[];  // [key blocks of the widest sequence]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int u = blockIdx.x;
  const int4 t = sel_tasks[u];
  constexpr int PER = D / 32;
  float qm[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) qm[e] = means[static_cast<size_t>(t.x) * D + lane * PER + e];
  constexpr int U = 8;
  for (int n0 = warp; n0 < t.z; n0 += U * kSelWarps) {
    float km[U][PER];
#pragma unroll
    for (int v = 0; v < U; ++v) {
      const int n = n0 + v * kSelWarps;
#pragma unroll
      for (int e = 0; e < PER; ++e) km[v][e] = n < t.z ? means[static_cast<size_t>(t.y + n) * D + lane * PER + e] : 0.f;
    }
#pragma unroll
    for (int v = 0; v < U; ++v) {
      const int n = n0 + v * kSelWarps;
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) d = fmaf(qm[e], km[v][e], d);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      if (lane == 0 && n < t.z) sc[n] = d;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  // k rounds of arg-max (ties to the lower index); chosen blocks are marked
  // with -inf, and a score is never -inf otherwise (finite inputs)
  const int cnt = min(topk, t.z);
  for (int round = 0; round < cnt; ++round) {
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int n = lane; n < t.z; n += 32) {
      const float v = sc[n];
      if (v > best || (v == best && n < bi)) {
        best = v;
        bi = n;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > best || (ov == best && oi < bi)) {
        best = ov;
        bi = oi;
      }
    }
    __syncwarp();
    if (lane == 0) sc[bi] = -INFINITY;
    __syncwarp();
  }
  // the chosen blocks in ascending order, then -1
  int32_t* out = selection + static_cast<size_t>(u) * topk;
  int written = 0;
  for (int n0 = 0; n0 < t.z; n0 += 32) {
    const int n = n0 + lane;
    const bool chosen = n < t.z && sc[n] == -INFINITY;
    const uint32_t mask = __ballot_sync(0xffffffffu, chosen);
    if (chosen) out[written + __popc(mask & ((1u << lane) - 1u))] = n;
    written += __popc(mask);
  }
  for (int i = written + lane; i < topk; i += 32) out[i] = -1;
}

}  // namespace topk

int launch_topk_select(const TopkArgs& a) {
  if (a.n_tasks == 0) return JFA_OK;
  {
    static_assert(kFwdRows <= 32 * topk::kMeanWarps && kKvBlock <= 32 * topk::kMeanWarps, "one round of rows per warp");
    ProfileScope prof(kKindTopk, a.stream);
    if (a.D == 128)
      topk::block_mean_kernel<128><<<a.n_tasks, 32 * topk::kMeanWarps, 0, a.stream>>>(
          static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k), a.H, a.Hkv, a.mean_tasks,
          a.means);
    else
      topk::block_mean_kernel<64><<<a.n_tasks, 32 * topk::kMeanWarps, 0, a.stream>>>(
          static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k), a.H, a.Hkv, a.mean_tasks,
          a.means);
    if (cudaGetLastError() != cudaSuccess) return JFA_ERR_CUDA;
  }
  if (a.n_units == 0) return JFA_OK;
  const size_t smem = static_cast<size_t>(a.nk_max) * sizeof(float);  // one score per key block
  if (smem > 48 * 1024) return JFA_ERR_UNSUPPORTED;  // the entry point rejects such sequences first
  ProfileScope prof(kKindTopk, a.stream);
  if (a.D == 128)
    topk::select_kernel<128><<<a.n_units, 32 * topk::kSelWarps, smem, a.stream>>>(a.means, a.sel_tasks, a.topk,
                                                                                 a.selection);
  else
    topk::select_kernel<64><<<a.n_units, 32 * topk::kSelWarps, smem, a.stream>>>(a.means, a.sel_tasks, a.topk,
                                                                                a.selection);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

}  // namespace jfa
