// Launchers of the sm_103a kernels, one translation unit per head_dim.
#pragma once
#include <cuda_runtime.h>

#include "attn_params.h"

namespace attn {

using FwdLauncher = cudaError_t (*)(const FwdParams& p, int grid, cudaStream_t stream);
using CombineLauncher = cudaError_t (*)(const CombineParams& p, int n_groups, cudaStream_t stream);
// grid: one block per (sequence, head group) x 16-column slice, one warp per query head
using DecodeCombineLauncher = cudaError_t (*)(const DecodeCombineParams& p, int n_groups, cudaStream_t stream);

FwdLauncher fwd_launcher_d64(bool bf16, bool causal, bool varlen);
FwdLauncher fwd_launcher_d128(bool bf16, bool causal, bool varlen);
// The dense forward with the rotary embedding of Q applied in the kernel
// (FwdParams::rope_cs and its companions set).
FwdLauncher fwd_rope_launcher_d64(bool bf16, bool causal);
FwdLauncher fwd_rope_launcher_d128(bool bf16, bool causal);
// Packed varlen forwards whose keys have their own offsets: when the
// sequences (at most kVarlenSortMax) have key counts more than 4x apart, the
// kernel numbers them by key count and places the units in snake order.
FwdLauncher fwd_sorted_launcher_d64(bool bf16, bool causal);
FwdLauncher fwd_sorted_launcher_d128(bool bf16, bool causal);
CombineLauncher combine_launcher_d64(bool bf16);
CombineLauncher combine_launcher_d128(bool bf16);
DecodeCombineLauncher decode_combine_launcher_d64(bool bf16);
DecodeCombineLauncher decode_combine_launcher_d128(bool bf16);

// The transposed decode kernel (head_dim 64 or 128, d): S^T = K Q^T and u^T += V^T P^T
// with the keys, then d, on the TMEM lanes; same units, pieces and partial
// layout as the packed forward's decode mode.  With d = 64 a softmax step
// covers two key tiles: split must then be even (pieces of whole steps) for
// full steps, though any split gives the right result.  tm_q: q (B, Hq, 128) as
// (d, Hq, B, 1) with box 64 x G x 1 x 1; tm_k, tm_v: (d, Hkv, total_k, 1).
cudaError_t launch_decode_tc(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v, void* o,
                             float* lse, const int* cu_k, int* pref_out, void* part_o, float* part_ml, int* err,
                             unsigned long long timeout_ns, int B, int Hq, int Hkv, int total_k, int split,
                             float scale_log2, bool bf16, int d, int grid, cudaStream_t stream);
// Sequences per call that launch_decode_tc takes for head_dim d (its shared
// memory holds a prefix table of B + 1 ints).
int decode_tc_max_b(int d);

// Test kernel: waits on a barrier that never completes, under `timeout_ns`.
cudaError_t launch_selftest_wait(int* err_word, unsigned long long timeout_ns, cudaStream_t stream);

}  // namespace attn
