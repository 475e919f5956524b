// Padded batches around the packed (varlen) forward: the index of the kept
// tokens of a key-padding mask, and row gather / scatter between the padded
// (B, L, ...) and the packed (total, ...) layouts.  The flash-attention
// training-integration page (inference.lei6393.com, 07-usage-tutorial /
// 02-training-integration, §2.5) drops the padded positions before the
// variable-length call and puts the outputs back at their positions after it;
// these kernels are those two steps.  All are bound by HBM (or by launch
// latency when small): 16-byte coalesced copies, one row per group of
// consecutive threads.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn.h"
#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kThreads = 256;

// kept-token count of each row b -> cu_seqlens[b + 1]
__global__ void __launch_bounds__(kThreads) count_rows_kernel(const uint8_t* __restrict__ mask, int L,
                                                              int* __restrict__ cu) {
  const int b = blockIdx.x;
  const uint8_t* row = mask + static_cast<size_t>(b) * L;
  int c = 0;
  for (int i = threadIdx.x; i < L; i += kThreads) c += (row[i] != 0);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  __shared__ int part[kThreads / 32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int w = 0; w < kThreads / 32; ++w) s += part[w];
    cu[b + 1] = s;
  }
}

// cu_seqlens[0] = 0, cu_seqlens[b + 1] = counts[0] + ... + counts[b] (in place)
__global__ void __launch_bounds__(1024) scan_counts_kernel(int B, int* __restrict__ cu) {
  __shared__ int warp_tot[32];
  __shared__ int carry;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    carry = 0;
    cu[0] = 0;
  }
  __syncthreads();
  for (int b0 = 0; b0 < B; b0 += 1024) {
    const int b = b0 + threadIdx.x;
    const int x = (b < B) ? cu[b + 1] : 0;
    int inc = x;   // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    if (lane == 31) warp_tot[w] = inc;
    __syncthreads();
    if (w == 0) {
      int t = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      warp_tot[lane] = t;   // inclusive over warps
    }
    __syncthreads();
    const int before = carry + (w > 0 ? warp_tot[w - 1] : 0);
    if (b < B) cu[b + 1] = before + inc;
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_tot[31];
    __syncthreads();
  }
}

// indices[cu[b] + k] = b * L + i for the k-th kept position i of row b
__global__ void __launch_bounds__(kThreads) index_rows_kernel(const uint8_t* __restrict__ mask, int L,
                                                              const int* __restrict__ cu, int* __restrict__ idx) {
  const int b = blockIdx.x;
  const uint8_t* row = mask + static_cast<size_t>(b) * L;
  __shared__ int warp_cnt[kThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int base = cu[b];
  for (int i0 = 0; i0 < L; i0 += kThreads) {
    const int i = i0 + threadIdx.x;
    const bool keep = (i < L) && (row[i] != 0);
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    const int rank_in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_cnt[w] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int v = 0; v < kThreads / 32; ++v) {
      const int n = warp_cnt[v];
      before += (v < w) ? n : 0;
      total += n;
    }
    if (keep) idx[base + before + rank_in_warp] = b * L + i;
    base += total;
    __syncthreads();
  }
}

// dst row r = src row idx[r] (gather) or dst row idx[r] = src row r
// (scatter), for r < n = min(n_max, *n_dev); rows are `cpr` 16-byte words.
// An index outside [0, n_other) (the padded side's row count) moves nothing.
// The gather also zeroes dst rows n .. n+127 below n_max (a tile's worth past
// the last packed row, which the attention kernels read and weight by zero).
template <bool SCATTER>
__global__ void __launch_bounds__(kThreads) move_rows_kernel(const uint4* __restrict__ src, const int* __restrict__ idx,
                                                             int n_max, const int* __restrict__ n_dev, int n_other,
                                                             int cpr, uint4* __restrict__ dst) {
  const int n = max(0, min(n_max, __ldg(n_dev)));
  const int n_zero = SCATTER ? n : min(n_max, n + 128);
  const long long words = static_cast<long long>(n_zero) * cpr;
  for (long long x = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; x < words;
       x += static_cast<long long>(gridDim.x) * kThreads) {
    const long long r = x / cpr;
    const int c = static_cast<int>(x - r * cpr);
    if (!SCATTER && r >= n) {
      dst[r * cpr + c] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const long long other = __ldg(idx + r);
    if (other < 0 || other >= n_other) continue;
    if (SCATTER)
      dst[other * cpr + c] = __ldg(src + r * cpr + c);
    else
      dst[r * cpr + c] = __ldg(src + other * cpr + c);
  }
}

// lse of the packed forward, (Hq, n_max), to the padded (B, Hq, L)
__global__ void __launch_bounds__(kThreads) scatter_lse_kernel(const float* __restrict__ src, const int* __restrict__ idx,
                                                               int n_max, const int* __restrict__ n_dev, int Hq, int B,
                                                               int L, float* __restrict__ dst) {
  const int n = min(n_max, __ldg(n_dev));
  const long long items = static_cast<long long>(n) * Hq;
  for (long long x = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; x < items;
       x += static_cast<long long>(gridDim.x) * kThreads) {
    const int h = static_cast<int>(x / n);
    const int r = static_cast<int>(x - static_cast<long long>(h) * n);
    const int p = __ldg(idx + r);
    if (p < 0 || p >= B * L) continue;
    const int b = p / L, i = p - b * L;
    dst[(static_cast<size_t>(b) * Hq + h) * L + i] = __ldg(src + static_cast<size_t>(h) * n_max + r);
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int grid_for(long long items, int sm_count) {
  const long long blocks = (items + kThreads - 1) / kThreads;
  const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * 8;
  return static_cast<int>(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

int sm_count_now() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace
}  // namespace attn

extern "C" {

int attn_unpad_index(const unsigned char* mask, int B, int L, int* cu_seqlens, int* indices, cudaStream_t stream) {
  using namespace attn;
  if (!mask || !cu_seqlens || !indices || B <= 0 || L <= 0) return ATTN_EINVAL;
  if (static_cast<long long>(B) * L > (1LL << 31) - 1) return ATTN_EINVAL;
  count_rows_kernel<<<B, kThreads, 0, stream>>>(mask, L, cu_seqlens);
  scan_counts_kernel<<<1, 1024, 0, stream>>>(B, cu_seqlens);
  index_rows_kernel<<<B, kThreads, 0, stream>>>(mask, L, cu_seqlens, indices);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  count_launch();
  count_launch();
  count_launch();
  return ATTN_OK;
}

int attn_gather_rows(const void* src, int src_rows, const int* indices, int n_max, const int* n_dev, int row_bytes,
                     void* dst, cudaStream_t stream) {
  using namespace attn;
  if (!src || !indices || !n_dev || !dst || n_max < 0 || src_rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0)
    return ATTN_EINVAL;
  if (!aligned16(src) || !aligned16(dst)) return ATTN_EINVAL;
  if (n_max == 0) return ATTN_OK;
  const int cpr = row_bytes / 16;
  move_rows_kernel<false><<<grid_for(static_cast<long long>(n_max) * cpr, sm_count_now()), kThreads, 0, stream>>>(
      static_cast<const uint4*>(src), indices, n_max, n_dev, src_rows, cpr, static_cast<uint4*>(dst));
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  count_launch();
  return ATTN_OK;
}

int attn_scatter_rows(const void* src, const int* indices, int n_max, const int* n_dev, int row_bytes, void* dst,
                      int dst_rows, cudaStream_t stream) {
  using namespace attn;
  if (!src || !indices || !n_dev || !dst || n_max < 0 || dst_rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0)
    return ATTN_EINVAL;
  if (!aligned16(src) || !aligned16(dst)) return ATTN_EINVAL;
  if (n_max == 0) return ATTN_OK;
  const int cpr = row_bytes / 16;
  move_rows_kernel<true><<<grid_for(static_cast<long long>(n_max) * cpr, sm_count_now()), kThreads, 0, stream>>>(
      static_cast<const uint4*>(src), indices, n_max, n_dev, dst_rows, cpr, static_cast<uint4*>(dst));
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  count_launch();
  return ATTN_OK;
}

int attn_scatter_lse(const float* src, const int* indices, int n_max, const int* n_dev, int Hq, int B, int L,
                     float* dst, cudaStream_t stream) {
  using namespace attn;
  if (!src || !indices || !n_dev || !dst || n_max < 0 || Hq <= 0 || B <= 0 || L <= 0) return ATTN_EINVAL;
  if (static_cast<long long>(B) * L > (1LL << 31) - 1 || static_cast<long long>(B) * Hq * L > (1LL << 40))
    return ATTN_EINVAL;
  if (n_max == 0) return ATTN_OK;
  scatter_lse_kernel<<<grid_for(static_cast<long long>(n_max) * Hq, sm_count_now()), kThreads, 0, stream>>>(
      src, indices, n_max, n_dev, Hq, B, L, dst);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  count_launch();
  return ATTN_OK;
}

}  // extern "C"
