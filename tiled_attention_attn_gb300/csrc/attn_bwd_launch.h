// Launchers of the backward kernels, one translation unit per head_dim.
#pragma once
#include <cuda_runtime.h>

#include "attn_bwd_kernel.cuh"

namespace attn {

// Inputs of the first pass (D_i = dout_i . O_i and lse in exp2 units).
struct BwdPrep {
  const void* o;
  const void* dout;
  const float* lse;
  int grid;
};

using BwdLauncher = cudaError_t (*)(const BwdParams& p, const BwdPrep& pr, cudaStream_t stream);

BwdLauncher bwd_launcher_d64(bool bf16, bool causal);
BwdLauncher bwd_launcher_d128(bool bf16, bool causal);

}  // namespace attn
