// host.h -- host-side helpers shared by the launchers: tensor-map encoding,
// device properties, error mapping.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/jfa.h"

namespace jfa {

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

}  // namespace jfa
