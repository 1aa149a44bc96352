// topk.h -- launcher of the block-sparse forward's first stage (see topk.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace jfa {

struct TopkArgs {
  const void *q, *k;
  int H, Hkv, D;
  const int4* mean_tasks;  // device: (row0, rows, head, 0 = q / 1 = k) per block to average
  int n_tasks;
  float* means;            // device workspace [n_tasks, D]
  const int4* sel_tasks;   // device: (query-mean row, first key-mean row, key blocks, 0) per query block
  int n_units;
  int topk, nk_max;        // blocks to choose; most key blocks of any sequence
  int32_t* selection;      // device [n_units, topk]
  cudaStream_t stream;
};

int launch_topk_select(const TopkArgs& a);

}  // namespace jfa
