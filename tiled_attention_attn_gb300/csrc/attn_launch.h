// Launchers of the sm_103a kernels, one translation unit per head_dim.
#pragma once
#include <cuda_runtime.h>

#include "attn_params.h"

namespace attn {

using FwdLauncher = cudaError_t (*)(const FwdParams& p, int grid, cudaStream_t stream);
using CombineLauncher = cudaError_t (*)(const CombineParams& p, int n_groups, cudaStream_t stream);
// grid: one block per (sequence, head group) x 16-column slice
using DecodeCombineLauncher = cudaError_t (*)(const DecodeCombineParams& p, int n_groups, cudaStream_t stream);

FwdLauncher fwd_launcher_d64(bool bf16, bool causal, bool varlen);
FwdLauncher fwd_launcher_d128(bool bf16, bool causal, bool varlen);
CombineLauncher combine_launcher_d64(bool bf16);
CombineLauncher combine_launcher_d128(bool bf16);
DecodeCombineLauncher decode_combine_launcher_d64(bool bf16);
DecodeCombineLauncher decode_combine_launcher_d128(bool bf16);

// Test kernel: waits on a barrier that never completes, under `timeout_ns`.
cudaError_t launch_selftest_wait(int* err_word, unsigned long long timeout_ns, cudaStream_t stream);

}  // namespace attn
