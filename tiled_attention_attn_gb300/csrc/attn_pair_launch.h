// Launcher of the CTA-pair forward kernels (one per head_dim translation unit).
#pragma once
#include <cuda_runtime.h>

#include "attn_params.h"

namespace attn {

// Launches 2 * n_pairs CTAs in clusters of two; `cooperative` (schedules
// with split key ranges) makes it a cooperative launch.
using PairLauncher = cudaError_t (*)(const PairParams& p, int n_pairs, bool cooperative, cudaStream_t stream);

PairLauncher pair_launcher_d128(bool bf16, bool causal);

}  // namespace attn
