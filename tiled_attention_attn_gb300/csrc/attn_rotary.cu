// Rotary position embedding of Q or K (training-integration page
// inference.lei6393.com, 07-usage-tutorial/02-training-integration, §4:
// rotary dimension, base frequency, GPT-NeoX or GPT-J pairing, and a position
// offset that starts new tokens at the cache length).  For pair i of the
// first rot_dim features (i < rot_dim / 2) the angle is
//   a = position * base^(-2 i / rot_dim)
// and the pair (x1, x2) becomes (x1 cos a - x2 sin a, x1 sin a + x2 cos a);
// the pair is (i, i + rot_dim/2) for GPT-NeoX and (2i, 2i+1) for GPT-J;
// features from rot_dim on are copied.  fp32 arithmetic on 16-bit data;
// bound by HBM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "attn.h"
#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kThreads = 256;
constexpr int kHeadsPerThread = 8;   // heads sharing one thread's sin / cos (vector path)

template <bool BF16>
__device__ __forceinline__ float ld16(const uint16_t* p) {
  const uint16_t v = *p;
  if constexpr (BF16) return __bfloat162float(__ushort_as_bfloat16(v));
  return __half2float(__ushort_as_half(v));
}
template <bool BF16>
__device__ __forceinline__ void st16(uint16_t* p, float x) {
  if constexpr (BF16) *p = __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else *p = __half_as_ushort(__float2half_rn(x));
}

// token r of a (rows, H, d) tensor: its sequence b and position in it
__device__ __forceinline__ int position_of(int r, int L, const int* cu, int B, const int* offset) {
  int b, i;
  if (cu == nullptr) {
    b = r / L;
    i = r - b * L;
  } else {
    int lo = 0, hi = B;   // largest b with cu[b] <= r
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(cu + mid) <= r) lo = mid; else hi = mid;
    }
    b = lo;
    i = r - __ldg(cu + b);
  }
  return i + (offset ? __ldg(offset + b) : 0);
}

// Work items per (token, head): groups of 4 rotated pairs, then groups of 8
// copied tail features (none when rotating in place).  A thread owns whole
// pairs (it loads both members before it stores either), so y == x is safe.
template <bool BF16, bool GPTJ>
__global__ void __launch_bounds__(kThreads) rotary_kernel(const uint16_t* x, uint16_t* y,
                                                          long long rows, long long token_stride, int L, int H,
                                                          int d, int rot, float log2_base,
                                                          const int* __restrict__ cu, int B,
                                                          const int* __restrict__ offset, bool in_place) {
  const int half = rot / 2;
  const int pair_groups = (half + 3) / 4;
  const int tail_groups = in_place ? 0 : (d - rot + 7) / 8;
  const int per = pair_groups + tail_groups;
  const long long items = rows * H * per;
  for (long long it = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; it < items;
       it += static_cast<long long>(gridDim.x) * kThreads) {
    const long long th = it / per;
    const int g = static_cast<int>(it - th * per);
    const long long r = th / H;
    const long long at = r * token_stride + (th - r * H) * d;
    const uint16_t* xs = x + at;
    uint16_t* ys = y + at;
    if (g >= pair_groups) {   // unrotated features
      const int c0 = rot + (g - pair_groups) * 8;
      for (int c = c0; c < min(c0 + 8, d); ++c) ys[c] = xs[c];
      continue;
    }
    const float pos = static_cast<float>(position_of(static_cast<int>(r), L, cu, B, offset));
    float x1[4], x2[4];
    int c1[4], c2[4];
    const int i0 = g * 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = i0 + e;
      c1[e] = GPTJ ? 2 * i : i;
      c2[e] = GPTJ ? 2 * i + 1 : i + half;
      if (i < half) {
        x1[e] = ld16<BF16>(xs + c1[e]);
        x2[e] = ld16<BF16>(xs + c2[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = i0 + e;
      if (i >= half) break;
      const float theta = exp2f(-2.0f * static_cast<float>(i) / static_cast<float>(rot) * log2_base);
      float sn, cs;
      sincosf(pos * theta, &sn, &cs);
      st16<BF16>(ys + c1[e], x1[e] * cs - x2[e] * sn);
      st16<BF16>(ys + c2[e], x1[e] * sn + x2[e] * cs);
    }
  }
}

// Vector path (rot_dim a multiple of 16, d a multiple of 8, 16-byte aligned
// rows): a thread takes one token, one group of 8 pairs and up to 8 heads,
// forms the 8 (sin, cos) once and applies them to those heads, with 16-byte loads and
// stores; the pair frequencies come from a table in shared memory.  Tail
// features are copied 8 at a time.
template <bool BF16, bool GPTJ>
__global__ void __launch_bounds__(kThreads) rotary_vec_kernel(const uint16_t* x, uint16_t* y, long long rows,
                                                              long long token_stride, int L, int H, int d, int rot,
                                                              float log2_base, const int* __restrict__ cu, int B,
                                                              const int* __restrict__ offset, bool in_place) {
  __shared__ float theta[256];
  const int half = rot / 2;
  for (int i = threadIdx.x; i < half; i += kThreads)
    theta[i] = exp2f(-2.0f * static_cast<float>(i) / static_cast<float>(rot) * log2_base);
  __syncthreads();
  const int pair_groups = half / 8;
  const int tail_groups = in_place ? 0 : (d - rot) / 8;
  const int per = pair_groups + tail_groups;
  const int chunks = (H + kHeadsPerThread - 1) / kHeadsPerThread;
  const long long items = rows * chunks * per;
  for (long long it = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; it < items;
       it += static_cast<long long>(gridDim.x) * kThreads) {
    const long long rc = it / per;   // (token, head chunk)
    const int g = static_cast<int>(it - rc * per);
    const long long r = rc / chunks;
    const int h_lo = static_cast<int>(rc - r * chunks) * kHeadsPerThread;
    const int h_hi = min(h_lo + kHeadsPerThread, H);
    const uint16_t* xt = x + r * token_stride;
    uint16_t* yt = y + r * token_stride;
    if (g >= pair_groups) {
      const int c0 = rot + (g - pair_groups) * 8;
      for (int h = h_lo; h < h_hi; ++h)
        *reinterpret_cast<uint4*>(yt + h * d + c0) = *reinterpret_cast<const uint4*>(xt + h * d + c0);
      continue;
    }
    const float pos = static_cast<float>(position_of(static_cast<int>(r), L, cu, B, offset));
    float sn[8], cs[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sincosf(pos * theta[8 * g + e], &sn[e], &cs[e]);
    // the 8 pairs of this group: GPT-NeoX (8g + e, half + 8g + e); GPT-J (16g + 2e, 16g + 2e + 1)
    const int oa = GPTJ ? 16 * g : 8 * g;
    const int ob = GPTJ ? 16 * g + 8 : half + 8 * g;
    for (int h = h_lo; h < h_hi; ++h) {
      uint16_t va[8], vb[8], ra[8], rb[8];
      *reinterpret_cast<uint4*>(va) = *reinterpret_cast<const uint4*>(xt + h * d + oa);
      *reinterpret_cast<uint4*>(vb) = *reinterpret_cast<const uint4*>(xt + h * d + ob);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        // GPT-J: pair e is elements 2e, 2e+1 of the 16 loaded (va holds 0..7, vb 8..15)
        const uint16_t u1 = GPTJ ? ((2 * e < 8) ? va[2 * e] : vb[2 * e - 8]) : va[e];
        const uint16_t u2 = GPTJ ? ((2 * e + 1 < 8) ? va[2 * e + 1] : vb[2 * e - 7]) : vb[e];
        const float x1 = ld16<BF16>(&u1), x2 = ld16<BF16>(&u2);
        uint16_t o1, o2;
        st16<BF16>(&o1, x1 * cs[e] - x2 * sn[e]);
        st16<BF16>(&o2, x1 * sn[e] + x2 * cs[e]);
        if (GPTJ) {
          if (2 * e < 8) ra[2 * e] = o1; else rb[2 * e - 8] = o1;
          if (2 * e + 1 < 8) ra[2 * e + 1] = o2; else rb[2 * e - 7] = o2;
        } else {
          ra[e] = o1;
          rb[e] = o2;
        }
      }
      *reinterpret_cast<uint4*>(yt + h * d + oa) = *reinterpret_cast<const uint4*>(ra);
      *reinterpret_cast<uint4*>(yt + h * d + ob) = *reinterpret_cast<const uint4*>(rb);
    }
  }
}

}  // namespace
}  // namespace attn

namespace attn {
namespace {

// Rotates the first h_rot heads of every token of a tensor whose tokens hold
// h_total heads of d features; out of place, the other heads are copied.
int rotary(const void* x, void* y, int B, int L, int h_total, int h_rot, int d, int rot_dim, float base,
           int interleaved, const int* cu, int total, const int* offsets, int fp16, cudaStream_t stream) {
  if (!x || !y || B <= 0 || h_total <= 0 || h_rot <= 0 || h_rot > h_total || d <= 0 || (fp16 != 0 && fp16 != 1))
    return ATTN_EINVAL;
  if (rot_dim <= 0 || rot_dim > d || (rot_dim & 1) || !(base > 1.0f) || !std::isfinite(base)) return ATTN_EINVAL;
  if (interleaved != 0 && interleaved != 1) return ATTN_EINVAL;
  const bool varlen = cu != nullptr;
  if (varlen ? total < 0 : L < 0) return ATTN_EINVAL;
  const long long rows = varlen ? static_cast<long long>(total) : static_cast<long long>(B) * L;
  const long long token_stride = static_cast<long long>(h_total) * d;
  if (rows * token_stride > (1LL << 40) || rows > (1LL << 31) - 1) return ATTN_EINVAL;
  // x and y either the same tensor or disjoint: a partial overlap would race
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x), ya = reinterpret_cast<uintptr_t>(y);
  const uintptr_t bytes = static_cast<uintptr_t>(rows * token_stride * 2);
  if (xa != ya && xa < ya + bytes && ya < xa + bytes) return ATTN_EINVAL;
  if (rows == 0) return ATTN_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ELAUNCH;
  const bool in_place = xa == ya;
  const int H = h_rot;
  const bool vec = (rot_dim % 16 == 0) && (d % 8 == 0) && rot_dim <= 512 && (xa % 16 == 0) && (ya % 16 == 0);
  const long long items = vec ? rows * ((H + kHeadsPerThread - 1) / kHeadsPerThread) *
                                    (rot_dim / 16 + (in_place ? 0 : (d - rot_dim) / 8))
                              : rows * H * ((rot_dim / 2 + 3) / 4 + (in_place ? 0 : (d - rot_dim + 7) / 8));
  const long long blocks = (items + kThreads - 1) / kThreads;
  const int grid = static_cast<int>(blocks < 8LL * sms ? blocks : 8LL * sms);
  const float lb = std::log2(base);
  auto* xs = static_cast<const uint16_t*>(x);
  auto* ys = static_cast<uint16_t*>(y);
  const int Lr = varlen ? 1 : L;
  if (vec) {
    if (fp16 == 0) {
      if (interleaved) rotary_vec_kernel<true, true><<<grid, kThreads, 0, stream>>>(xs, ys, rows, token_stride, Lr, H, d, rot_dim, lb, cu, B, offsets, in_place);
      else rotary_vec_kernel<true, false><<<grid, kThreads, 0, stream>>>(xs, ys, rows, token_stride, Lr, H, d, rot_dim, lb, cu, B, offsets, in_place);
    } else {
      if (interleaved) rotary_vec_kernel<false, true><<<grid, kThreads, 0, stream>>>(xs, ys, rows, token_stride, Lr, H, d, rot_dim, lb, cu, B, offsets, in_place);
      else rotary_vec_kernel<false, false><<<grid, kThreads, 0, stream>>>(xs, ys, rows, token_stride, Lr, H, d, rot_dim, lb, cu, B, offsets, in_place);
    }
  } else if (fp16 == 0) {
    if (interleaved) rotary_kernel<true, true><<<grid, kThreads, 0, stream>>>(xs, ys, rows, token_stride, Lr, H, d, rot_dim, lb, cu, B, offsets, in_place);
    else rotary_kernel<true, false><<<grid, kThreads, 0, stream>>>(xs, ys, rows, token_stride, Lr, H, d, rot_dim, lb, cu, B, offsets, in_place);
  } else {
    if (interleaved) rotary_kernel<false, true><<<grid, kThreads, 0, stream>>>(xs, ys, rows, token_stride, Lr, H, d, rot_dim, lb, cu, B, offsets, in_place);
    else rotary_kernel<false, false><<<grid, kThreads, 0, stream>>>(xs, ys, rows, token_stride, Lr, H, d, rot_dim, lb, cu, B, offsets, in_place);
  }
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  count_launch();
  if (!in_place && h_rot < h_total) {
    // the heads that are not rotated (v of a packed qkv, v of a packed kv)
    const size_t pitch = static_cast<size_t>(token_stride) * 2;
    const size_t skip = static_cast<size_t>(h_rot) * d * 2;
    if (cudaMemcpy2DAsync(static_cast<uint8_t*>(y) + skip, pitch, static_cast<const uint8_t*>(x) + skip, pitch,
                          pitch - skip, static_cast<size_t>(rows), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
      return ATTN_ELAUNCH;
  }
  return ATTN_OK;
}

// (cos, sin) of pos * theta_i for pos < n_pos and i < rot / 2, computed as
// the rotary kernels above compute them, for the forward kernel's in-kernel
// rotation of Q.
__global__ void rope_table_kernel(float2* cs, int n_pos, int rot, float log2_base) {
  const int half = rot / 2;
  const long long n = static_cast<long long>(n_pos) * half;
  for (long long it = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; it < n;
       it += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(it / half);
    const int i = static_cast<int>(it - static_cast<long long>(pos) * half);
    const float theta = exp2f(-2.0f * static_cast<float>(i) / static_cast<float>(rot) * log2_base);
    float sn, c;
    sincosf(static_cast<float>(pos) * theta, &sn, &c);
    cs[it] = make_float2(c, sn);
  }
}

}  // namespace

int rope_table(float2* cs, int n_pos, int rot, float base, cudaStream_t stream) {
  if (!cs || n_pos <= 0 || rot <= 0 || (rot & 1) || !(base > 1.0f)) return ATTN_EINVAL;
  const long long n = static_cast<long long>(n_pos) * (rot / 2);
  const int grid = static_cast<int>(std::min<long long>((n + 255) / 256, 1024));
  rope_table_kernel<<<grid, 256, 0, stream>>>(cs, n_pos, rot, std::log2(base));
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  count_launch();
  return ATTN_OK;
}

}  // namespace attn

extern "C" {

int attn_rotary(const void* x, void* y, int B, int L, int H, int d, int rot_dim, float base, int interleaved,
                const int* cu_seqlens_or_null, int total, const int* offsets_or_null, int fp16, cudaStream_t stream) {
  return attn::rotary(x, y, B, L, H, H, d, rot_dim, base, interleaved, cu_seqlens_or_null, total, offsets_or_null,
                      fp16, stream);
}

int attn_rotary_packed(const void* x, void* y, int B, int L, int h_total, int h_rot, int d, int rot_dim, float base,
                       int interleaved, const int* cu_seqlens_or_null, int total, const int* offsets_or_null, int fp16,
                       cudaStream_t stream) {
  return attn::rotary(x, y, B, L, h_total, h_rot, d, rot_dim, base, interleaved, cu_seqlens_or_null, total,
                      offsets_or_null, fp16, stream);
}

}  // extern "C"
