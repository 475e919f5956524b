// CTA-pair forward kernels for head_dim 128 (bf16 and fp16, causal or not)
// and their launcher: clusters of two CTAs, one CTA per SM.
#include <cuda_runtime.h>

#include "attn_pair_kernel.cuh"
#include "attn_pair_launch.h"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_pair(const PairParams& p, int n_pairs, bool cooperative, cudaStream_t stream) {
  constexpr int smem = pair::Cfg<D>::kSmem;
  static bool attr_done[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  auto kern = pair::attn_pair_kernel<D, BF16, CAUSAL>;
  if (dev < 0 || dev >= kMaxDevices || !attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * n_pairs);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // split pieces of one query block wait for each other before merging:
  // a cooperative launch guarantees that every CTA of the grid is resident
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cooperative ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

PairLauncher pair_launcher_d128(bool bf16, bool causal) {
  if (bf16) return causal ? launch_pair<128, true, true> : launch_pair<128, true, false>;
  return causal ? launch_pair<128, false, true> : launch_pair<128, false, false>;
}

}  // namespace attn
