// block.h -- launchers of the block-diagonal kernels (see block.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace jfa {

struct BlockArgs {
  const void *q, *k, *v, *dout;
  void *o, *dq, *dk, *dv;
  const int32_t* offsets_dev;
  const int32_t* bpb;         // device, [batch+1]
  const int32_t* prog_start;  // device, [n_prog+1]
  int* err;
  int rows, batch, H, D, n_blocks, n_prog;
  int use_clc;                // 1: Cluster Launch Control over chunks of `chunk` tiles
  int chunk, n_tiles, n_chunks;
  const uint32_t* rope_tab;   // rotary: packed table [positions, D/2] words (see rope.h), or null
  float scale;
  cudaStream_t stream;
};

int launch_block_fwd(const BlockArgs& a);
int launch_block_bwd(const BlockArgs& a);

}  // namespace jfa
