// host.h -- host-side helpers shared by the launchers: tensor-map encoding,
// device properties, error mapping.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/jfa.h"

namespace jfa {

// One-time setup of a kernel on each device (its dynamic shared-memory limit,
// the register check).  Attributes set with cudaFuncSetAttribute belong to the
// current device, so a process that drives several GPUs sets them on each.  The
// flags are atomic: first calls racing on several threads all run the setup,
// which is idempotent.
class PerDeviceOnce {
 public:
  // Runs `setup` (which returns a jfa status) unless it has already succeeded
  // on the current device.
  template <class F>
  int run(F&& setup) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return JFA_ERR_CUDA;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
    if (bit != 0 && (done_.load(std::memory_order_acquire) & bit) != 0) return JFA_OK;
    const int st = setup();
    if (st == JFA_OK && bit != 0) done_.fetch_or(bit, std::memory_order_release);
    return st;
  }

 private:
  std::atomic<uint64_t> done_{0};
};

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  int max_smem_optin = 0;
};

// Properties of the current device (cached per device).  Returns JFA_OK or an error.
int current_device(DeviceInfo* out);

// 2-D bf16 tensor map over a row-major [rows, inner] matrix, 128-byte swizzle,
// box {box_inner, box_rows}.  Rows past the end read as zero.
int make_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                uint32_t box_rows);
// Same for an fp32 matrix (box_inner * 4 bytes must be 128 for the swizzle).
int make_map_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                    uint32_t box_rows);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Launches `kernel` on `stream` as a programmatic dependent of the previous
// kernel there: it may be scheduled while that one finishes and must call
// griddepcontrol.wait before it reads the previous kernel's results.
template <class... KArgs, class... Args>
int launch_dependent(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t stream,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...) == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

// Which keys a query row sees inside its sequence: all of them, those up to
// the row (causal), or those within [row - win_left, row + win_right] (a
// sliding window; a negative bound leaves its side open).
enum MaskKind : int { kMaskNone = 0, kMaskCausal = 1, kMaskWindow = 2, kMaskTopK = 3 };
// kMaskTopK: each 256-row query unit attends over the key blocks a first
// stage chose for it (block-sparse forward; see topk.cu).

// Kernel launchers (one per .cu file).  They assume validated arguments.
struct FwdArgs {
  const void *q, *k, *v;
  void* o;
  float* lse;
  const int32_t* offsets_dev;
  int q_rows, kv_rows, o_rows;  // rows of q, of k/v, of o
  int H, Hkv, D, nq;            // nq > 0: broadcast-Q
  float scale;
  int causal;
  int mask;                     // MaskKind
  int win_left, win_right;      // kMaskWindow: visible keys [row - win_left, row + win_right]
  const int32_t* topk_sel;      // kMaskTopK: chosen key blocks [query blocks, topk], ascending, -1 padded
  const int32_t* topk_qb;       // kMaskTopK: query blocks before each sequence [batch+1]
  int topk;
  const int32_t* units;         // device, 4 ints per unit
  const int32_t* cta_start;     // device, n_cta + 1 (static plan only)
  int n_cta;                    // static plan: CTAs launched
  int n_units;
  int use_clc;                  // 1: launch n_units CTAs, units in cost order, Cluster Launch Control
  int* err;                     // device error word
  cudaStream_t stream;
};
int launch_fwd(const FwdArgs& a);

// Scheduling mode of the persistent jagged kernels: 0 static plan, 1 Cluster
// Launch Control.  Initially JFA_SCHED ("static" or "clc") if set, else
// kDefaultSched; jfa_set_schedule() changes it.
constexpr int kDefaultSched = 1;  // measured faster on every jagged workload
int sched_mode();
// The same choice for the jagged backward: JFA_SCHED_BWD, else kDefaultBwdSched;
// jfa_set_bwd_schedule() changes it.
constexpr int kDefaultBwdSched = 1;  // measured faster on the jagged, broadcast-Q and dense backward
int bwd_sched_mode();
// The same choice for the block-diagonal kernels: JFA_SCHED_BLOCK, else
// kDefaultBlockSched; jfa_set_block_schedule() changes it.  Under Cluster
// Launch Control a CTA's unit of work is a chunk of kBlockChunk consecutive
// (block pair, head) tiles.
constexpr int kDefaultBlockSched = 1;  // measured faster (D=128 forward and backward, D=64 backward)
constexpr int kBlockChunk = 16;
int block_sched_mode();

}  // namespace jfa
