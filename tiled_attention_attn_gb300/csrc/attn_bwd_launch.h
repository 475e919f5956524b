// Launchers of the backward kernels, one translation unit per head_dim.
#pragma once
#include <cuda_runtime.h>

#include "attn_bwd_kernel.cuh"

namespace attn {

// Inputs of the first pass (D_i = dout_i . O_i and lse in exp2 units) and
// the grids; varlen also fills the tile tables at `pref` first.
struct BwdPrep {
  const void* o;
  const void* dout;
  const float* lse;
  int* pref;          // varlen: p.tile_pref, written by the tile-count kernel
  int grid;           // first pass
  int grid_kv;        // varlen: 1-D grids (an upper bound; extra CTAs exit at once)
  int grid_q;
};

using BwdLauncher = cudaError_t (*)(const BwdParams& p, const BwdPrep& pr, cudaStream_t stream);

BwdLauncher bwd_launcher_d64(bool bf16, bool causal, bool varlen);
BwdLauncher bwd_launcher_d128(bool bf16, bool causal, bool varlen);

}  // namespace attn
