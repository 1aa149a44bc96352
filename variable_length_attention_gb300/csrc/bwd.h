// bwd.h -- launchers of the backward kernels (see bwd.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace jfa {

struct BwdArgs {
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  const int32_t* offsets_dev;
  int q_rows, kv_rows, o_rows;
  int H, Hkv, D, nq;  // query heads, K/V heads (H % Hkv == 0)
  float scale;
  int causal;
  int mask;                 // MaskKind (host.h)
  int win_left, win_right;  // kMaskWindow: keys [row - win_left, row + win_right] are visible
  const int32_t* units;
  const int32_t* cta_start;
  int n_cta;
  int n_units;
  int use_clc;    // 1: grid of n_units CTAs under Cluster Launch Control (units in cost order)
  float* lse2;    // workspace [H, o_rows]
  float* di;      // workspace [H, o_rows]
  float* dq_acc;  // workspace [q_rows, H, D]
  int* err;
  cudaStream_t stream;
};

int launch_bwd_prep(const BwdArgs& a, int num_sms);  // also zeroes dq_acc
int launch_bwd_main(const BwdArgs& a);
int launch_dq_convert(const BwdArgs& a, int num_sms);

}  // namespace jfa
