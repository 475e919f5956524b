// Decoding step: one new query per sequence against its packed key/value
// cache.  With one query row per head, S = q K^T and O = P V are matrix-vector
// products: each key and value row is used by the group's few query heads
// only, so the step is bound by reading the cache from HBM, not by
// arithmetic, and it runs on the CUDA cores without tensor-core tiles.
//
// Method (the exact softmax of page S23-J17, clxhxhhr.top/posts/5544, §3.1,
// split along the keys as the blocked recurrence allows): the keys of a
// sequence are cut into chunks of 128; a block scores one chunk for the
// group's query heads, keeps the chunk max m_c, the exp-sum l_c and the
// unnormalised u_c = sum_j 2^(s_j - m_c) v_j, and a second pass merges the
// chunks of a (sequence, head) with the same rescaling r = 2^(m_c - M) that
// the online softmax applies when its running max moves.
//
// Three launches: a one-warp pass that validates cu_seqlens_k and counts the
// chunks of every sequence, the chunk kernel (one block per chunk and key /
// value head; blocks past the last chunk return at once) and the merge (one
// block per sequence and query head).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"
#include "attn_params.h"

namespace attn {
namespace {

constexpr int kDecChunk = 128;     // keys per chunk
constexpr int kDecThreads = 128;   // the score pass gives each thread one key
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecMaxDevices = 64;

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t x) {
  if constexpr (BF16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&x));
  }
}

template <bool BF16>
__device__ __forceinline__ float load1(const void* p, size_t i) {
  if constexpr (BF16) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  } else {
    return __half2float(reinterpret_cast<const __half*>(p)[i]);
  }
}

template <bool BF16>
__device__ __forceinline__ void store1(void* p, size_t i, float x) {
  if constexpr (BF16) {
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  } else {
    reinterpret_cast<__half*>(p)[i] = __float2half_rn(x);
  }
}

// One warp: checks cu_seqlens_k (0 first, non-decreasing, last entry at most
// total_k) and writes pref[b] = chunks of sequences 0..b-1 (pref[B] = all).
// A malformed array records ATTN_DEVERR_BAD_SEQLENS and leaves pref all zero,
// so that nothing is scored and every output row is O = 0, lse = -inf.
__global__ void __launch_bounds__(32) attn_decode_prep_kernel(const int* __restrict__ cu_k, int B, int total_k,
                                                              int* __restrict__ pref, int* __restrict__ err) {
  const int lane = threadIdx.x;
  bool bad = (lane == 0) && (__ldg(cu_k) != 0);
  int carry = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    int cnt = 0;
    if (b < B) {
      const int a = __ldg(cu_k + b), e = __ldg(cu_k + b + 1);
      if (e < a || e > total_k) bad = true;
      const int len = e - a;
      cnt = (len > 0 && !bad) ? (len + kDecChunk - 1) / kDecChunk : 0;
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (b < B) pref[b + 1] = carry + x;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  if (lane == 0) pref[0] = 0;
  if (__any_sync(0xffffffffu, bad)) {
    __syncwarp();
    for (int b = lane; b <= B; b += 32) pref[b] = 0;
    if (lane == 0) atomicCAS(err, 0, ATTN_DEVERR_BAD_SEQLENS);
  }
}

// Shared memory of a chunk block: the chunk's key and value rows (copied in
// asynchronously with coalesced 16-byte copies; the 16-byte word c of row j
// sits at position c ^ (j mod words-per-row), so that the threads of a
// quarter warp reading one word of eight consecutive rows, or eight words of
// one row, hit distinct banks), the group's query rows, p per key, the
// warps' max and sum.  The per-warp partial outputs reuse the key rows.
template <int D, int G>
struct DecSmem {
  static constexpr int kRows = kDecChunk * D * 2;                    // one operand's rows, 16-bit
  static constexpr int kOffV = kRows;
  static constexpr int kOffQ = 2 * kRows;
  static constexpr int kOffP = kOffQ + G * D * 4;
  static constexpr int kOffW = kOffP + kDecChunk * G * 4;
  static constexpr int kBytes = kOffW + 2 * kDecWarps * G * 4;
  static_assert(kDecWarps * G * D * 4 <= kRows, "partial outputs fit in the key rows");
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool fill) {
  // fill = false: 16 zero bytes, nothing read
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(fill ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Block = (chunk cg, key/value head g), blockIdx.x = cg * Hkv + g.  Writes
// the chunk's (m, l) per query head of the group (m in scaled exp2 units)
// and u = sum_j 2^(s_j - m) v_j in fp32.
template <int D, int G, bool BF16>
__global__ void __launch_bounds__(kDecThreads, 3)
    attn_decode_chunk_kernel(const void* __restrict__ q, const void* __restrict__ k, const void* __restrict__ v,
                             const int* __restrict__ cu_k, const int* __restrict__ pref, float* __restrict__ part_o,
                             float2* __restrict__ part_ml, int B, int Hq, int Hkv, float scale_log2) {
  using S = DecSmem<D, G>;
  constexpr int kW = D / 8;   // 16-byte words per row
  extern __shared__ __align__(16) uint8_t dsm[];
  const uint4* sk = reinterpret_cast<const uint4*>(dsm);                        // [kDecChunk][kW], swizzled
  const uint4* sv = reinterpret_cast<const uint4*>(dsm + S::kOffV);             // [kDecChunk][kW], swizzled
  float (*red)[G][D] = reinterpret_cast<float (*)[G][D]>(dsm);                  // [kDecWarps][G][D], over sk
  float (*sq)[D] = reinterpret_cast<float (*)[D]>(dsm + S::kOffQ);
  float (*sp)[G] = reinterpret_cast<float (*)[G]>(dsm + S::kOffP);
  float (*wmax)[G] = reinterpret_cast<float (*)[G]>(dsm + S::kOffW);
  float (*wsum)[G] = reinterpret_cast<float (*)[G]>(dsm + S::kOffW + kDecWarps * G * 4);

  const int item = blockIdx.x;
  const int cg = item / Hkv;
  const int g = item - cg * Hkv;
  if (cg >= __ldg(pref + B)) return;
  int lo = 0, hi = B;   // largest b with pref[b] <= cg
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(pref + mid) <= cg) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int k0 = __ldg(cu_k + b) + (cg - __ldg(pref + b)) * kDecChunk;
  const int n = min(kDecChunk, __ldg(cu_k + b + 1) - k0);   // >= 1 for a counted chunk

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  // ---- key and value rows into shared memory: a warp copies whole rows
  // (two 256-byte or four 128-byte rows per step); rows past the chunk's
  // end are zero-filled
  {
    const size_t row0 = (static_cast<size_t>(k0) * Hkv + g) * kW;
    const size_t stride = static_cast<size_t>(Hkv) * kW;   // one key, in 16-byte words
    const uint4* kg = reinterpret_cast<const uint4*>(k) + row0;
    const uint4* vg = reinterpret_cast<const uint4*>(v) + row0;
    const uint32_t s0 = static_cast<uint32_t>(__cvta_generic_to_shared(dsm));
#pragma unroll
    for (int i = 0; i < kDecChunk * kW / kDecThreads; ++i) {
      const int w = i * kDecThreads + tid;
      const int j = w / kW, c = w % kW;
      const bool in = j < n;
      const size_t src = in ? static_cast<size_t>(j) * stride + c : 0;
      const uint32_t dst = static_cast<uint32_t>((j * kW + (c ^ (j % kW))) * 16);
      cp_async16(s0 + dst, kg + src, in);
      cp_async16(s0 + S::kOffV + dst, vg + src, in);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  const size_t q_base = (static_cast<size_t>(b) * Hq + static_cast<size_t>(g) * G) * D;
  for (int i = tid; i < G * D; i += kDecThreads) sq[i / D][i % D] = load1<BF16>(q, q_base + i);
  cp_async_wait_all();
  __syncthreads();

  // ---- scores: thread tid takes key tid of the chunk
  float s[G];
#pragma unroll
  for (int r = 0; r < G; ++r) s[r] = 0.0f;
#pragma unroll
  for (int i = 0; i < kW; ++i) {
    const uint4 kw = sk[tid * kW + (i ^ (tid % kW))];
    const float2 k01 = unpack2<BF16>(kw.x), k23 = unpack2<BF16>(kw.y);
    const float2 k45 = unpack2<BF16>(kw.z), k67 = unpack2<BF16>(kw.w);
#pragma unroll
    for (int r = 0; r < G; ++r) {
      const float4 qa = *reinterpret_cast<const float4*>(&sq[r][i * 8]);
      const float4 qb = *reinterpret_cast<const float4*>(&sq[r][i * 8 + 4]);
      float a = s[r];
      a = fmaf(qa.x, k01.x, a);
      a = fmaf(qa.y, k01.y, a);
      a = fmaf(qa.z, k23.x, a);
      a = fmaf(qa.w, k23.y, a);
      a = fmaf(qb.x, k45.x, a);
      a = fmaf(qb.y, k45.y, a);
      a = fmaf(qb.z, k67.x, a);
      a = fmaf(qb.w, k67.y, a);
      s[r] = a;
    }
  }
  const bool valid = tid < n;
#pragma unroll
  for (int r = 0; r < G; ++r) s[r] = valid ? s[r] * scale_log2 : -INFINITY;

  // ---- chunk max and exp-sum per query head
#pragma unroll
  for (int r = 0; r < G; ++r) {
    float x = s[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    if (lane == 0) wmax[warp][r] = x;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < G; ++r) {
    float m = wmax[0][r];
#pragma unroll
    for (int w = 1; w < kDecWarps; ++w) m = fmaxf(m, wmax[w][r]);
    const float p = valid ? exp2f(s[r] - m) : 0.0f;   // m is finite: the chunk has a key
    sp[tid][r] = p;
    float x = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) wsum[warp][r] = x;
  }
  __syncthreads();

  // ---- u = sum_j p_j v_j: thread (kl, dg) takes the 8 columns dg*8.. of
  // keys kl, kl + kKL, ... (zero rows past the end, p = 0)
  constexpr int kKL = kDecThreads / kW;
  const int dg = tid % kW, kl = tid / kW;
  float acc[G][8];
#pragma unroll
  for (int r = 0; r < G; ++r)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[r][e] = 0.0f;
#pragma unroll 4
  for (int j = kl; j < kDecChunk; j += kKL) {
    const uint4 vw = sv[j * kW + (dg ^ (j % kW))];
    const float2 v01 = unpack2<BF16>(vw.x), v23 = unpack2<BF16>(vw.y);
    const float2 v45 = unpack2<BF16>(vw.z), v67 = unpack2<BF16>(vw.w);
#pragma unroll
    for (int r = 0; r < G; ++r) {
      const float p = sp[j][r];
      acc[r][0] = fmaf(p, v01.x, acc[r][0]);
      acc[r][1] = fmaf(p, v01.y, acc[r][1]);
      acc[r][2] = fmaf(p, v23.x, acc[r][2]);
      acc[r][3] = fmaf(p, v23.y, acc[r][3]);
      acc[r][4] = fmaf(p, v45.x, acc[r][4]);
      acc[r][5] = fmaf(p, v45.y, acc[r][5]);
      acc[r][6] = fmaf(p, v67.x, acc[r][6]);
      acc[r][7] = fmaf(p, v67.y, acc[r][7]);
    }
  }
  // sum over the key lanes of a warp, then over the warps (the partials go
  // over the key rows, which nobody reads after the score pass)
#pragma unroll
  for (int o = kW; o < 32; o <<= 1)
#pragma unroll
    for (int r = 0; r < G; ++r)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[r][e] += __shfl_xor_sync(0xffffffffu, acc[r][e], o);
  if (lane < kW) {
#pragma unroll
    for (int r = 0; r < G; ++r) {
      float4* dst = reinterpret_cast<float4*>(&red[warp][r][dg * 8]);
      dst[0] = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
      dst[1] = make_float4(acc[r][4], acc[r][5], acc[r][6], acc[r][7]);
    }
  }
  __syncthreads();
  float* po = part_o + static_cast<size_t>(item) * G * D;
  for (int i = tid; i < G * D; i += kDecThreads) {
    float x = 0.0f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) x += (&red[w][0][0])[i];
    po[i] = x;
  }
  if (tid < G) {
    float m = wmax[0][tid], l = wsum[0][tid];
#pragma unroll
    for (int w = 1; w < kDecWarps; ++w) {
      m = fmaxf(m, wmax[w][tid]);
      l += wsum[w][tid];
    }
    part_ml[static_cast<size_t>(item) * G + tid] = make_float2(m, l);
  }
}

// Block = (sequence b, query head h), kMergeWarps warps: warp w merges the
// chunks w, w + kMergeWarps, ... of the sequence with a running max (lane
// holding D / 32 columns), then the warps' results are merged the same way:
// O = sum_c 2^(m_c - M) u_c / sum_c 2^(m_c - M) l_c with M = max_c m_c, and
// lse = M ln 2 + ln L.  A sequence with no key gives O = 0 and lse = -inf.
constexpr int kMergeWarps = 16;

template <int D, bool BF16>
__global__ void __launch_bounds__(kMergeWarps * 32)
    attn_decode_merge_kernel(const int* __restrict__ pref, const float* __restrict__ part_o,
                             const float2* __restrict__ part_ml, void* __restrict__ o, float* __restrict__ lse, int B,
                             int Hq, int Hkv, int G) {
  constexpr int kE = D / 32;   // columns per lane
  __shared__ float sm_m[kMergeWarps], sm_l[kMergeWarps];
  __shared__ __align__(16) float sm_o[kMergeWarps][D];
  const int bh = blockIdx.x;
  const int b = bh / Hq, h = bh - b * Hq;
  const int g = h / G, r = h - g * G;
  const int c0 = __ldg(pref + b), c1 = __ldg(pref + b + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float M = -INFINITY, L = 0.0f, acc[kE];
#pragma unroll
  for (int e = 0; e < kE; ++e) acc[e] = 0.0f;
#pragma unroll 2
  for (int c = c0 + warp; c < c1; c += kMergeWarps) {
    const size_t slot = (static_cast<size_t>(c) * Hkv + g) * G + r;
    const float2 ml = part_ml[slot];   // m is finite: every chunk has a key
    float x[kE];
    if constexpr (kE == 4) {
      const float4 t = *reinterpret_cast<const float4*>(part_o + slot * D + lane * 4);
      x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else {
      const float2 t = *reinterpret_cast<const float2*>(part_o + slot * D + lane * 2);
      x[0] = t.x; x[1] = t.y;
    }
    const float Mn = fmaxf(M, ml.x);
    const float a = (M == -INFINITY) ? 0.0f : exp2f(M - Mn);
    const float w = exp2f(ml.x - Mn);
    L = fmaf(L, a, ml.y * w);
#pragma unroll
    for (int e = 0; e < kE; ++e) acc[e] = fmaf(acc[e], a, x[e] * w);
    M = Mn;
  }
  if (lane == 0) {
    sm_m[warp] = M;
    sm_l[warp] = L;
  }
#pragma unroll
  for (int e = 0; e < kE; ++e) sm_o[warp][lane * kE + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    const int i = threadIdx.x;
    float Mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) Mx = fmaxf(Mx, sm_m[w]);
    float Lt = 0.0f, at = 0.0f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      if (sm_m[w] == -INFINITY) continue;   // a warp that merged no chunk
      const float sc = exp2f(sm_m[w] - Mx);
      Lt = fmaf(sm_l[w], sc, Lt);
      at = fmaf(sm_o[w][i], sc, at);
    }
    store1<BF16>(o, static_cast<size_t>(bh) * D + i, Lt > 0.0f ? at / Lt : 0.0f);
    if (i == 0) lse[static_cast<size_t>(h) * B + b] = (Lt > 0.0f) ? Mx * 0.69314718055994531f + logf(Lt) : -INFINITY;
  }
}

// chunk partials of the last call's shape, grown on demand and kept per device
struct DecWorkspace {
  void* buf = nullptr;
  size_t bytes = 0;
};
std::map<int, DecWorkspace> g_dec_ws;
std::mutex g_dec_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int D, int G, bool BF16>
cudaError_t launch_chunks(int grid, const void* q, const void* k, const void* v, const int* cu_k, const int* pref,
                          float* part_o, float2* part_ml, int B, int Hq, int Hkv, float scale_log2,
                          cudaStream_t stream) {
  constexpr int smem = DecSmem<D, G>::kBytes;
  static_assert(smem <= 74 * 1024, "three chunk blocks per SM");
  // per instantiation and device; calls hold the workspace lock
  static bool attr_done[kDecMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kDecMaxDevices || !attr_done[dev]) {
    e = cudaFuncSetAttribute(attn_decode_chunk_kernel<D, G, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kDecMaxDevices) attr_done[dev] = true;
  }
  attn_decode_chunk_kernel<D, G, BF16><<<grid, kDecThreads, smem, stream>>>(q, k, v, cu_k, pref, part_o, part_ml, B,
                                                                            Hq, Hkv, scale_log2);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_d(int G, int grid, const void* q, const void* k, const void* v, const int* cu_k,
                     const int* pref, float* part_o, float2* part_ml, void* o, float* lse, int B, int Hq, int Hkv,
                     float scale_log2, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (grid > 0) {
    switch (G) {
      case 1: e = launch_chunks<D, 1, BF16>(grid, q, k, v, cu_k, pref, part_o, part_ml, B, Hq, Hkv, scale_log2, stream); break;
      case 2: e = launch_chunks<D, 2, BF16>(grid, q, k, v, cu_k, pref, part_o, part_ml, B, Hq, Hkv, scale_log2, stream); break;
      case 4: e = launch_chunks<D, 4, BF16>(grid, q, k, v, cu_k, pref, part_o, part_ml, B, Hq, Hkv, scale_log2, stream); break;
      default: e = launch_chunks<D, 8, BF16>(grid, q, k, v, cu_k, pref, part_o, part_ml, B, Hq, Hkv, scale_log2, stream); break;
    }
    if (e != cudaSuccess) return e;
  }
  attn_decode_merge_kernel<D, BF16><<<B * Hq, kMergeWarps * 32, 0, stream>>>(pref, part_o, part_ml, o, lse, B, Hq,
                                                                          Hkv, G);
  return cudaGetLastError();
}

int decode(bool bf16, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
           int total_k, int d, float scale, const int* cu_k, cudaStream_t stream) {
  if (!q || !o || !lse || !cu_k) return ATTN_EINVAL;
  if (total_k != 0 && (!k || !v)) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return ATTN_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || total_k < 0 || Hq % Hkv != 0) return ATTN_EINVAL;
  if (!std::isfinite(scale) || scale < 0.0f) return ATTN_EINVAL;
  if (d != 64 && d != 128) return ATTN_EUNSUPPORTED;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return ATTN_EUNSUPPORTED;
  const long long n_chunks_max = static_cast<long long>(B) + (static_cast<long long>(total_k) + kDecChunk - 1) / kDecChunk;
  const long long items_max = n_chunks_max * Hkv;
  if (static_cast<long long>(B) * Hq > (1LL << 31) - 1 || items_max > (1LL << 31) - 1 ||
      static_cast<long long>(total_k) + kDecChunk > (1LL << 31) - 1)
    return ATTN_EINVAL;

  if (decode_tensor_cores_enabled() && total_k > 0 && B <= kVarlenMaxB)
    return decode_on_tensor_cores(bf16, q, k, v, o, lse, B, Hq, Hkv, total_k, d, scale, cu_k, stream);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ELAUNCH;
  DeviceInfo info;
  int rc = device_info(dev, info);
  if (rc) return rc;
  if (!info.supported) return ATTN_EUNSUPPORTED;

  // workspace: pref (B + 1 ints, padded to 16 bytes), (m, l) per chunk slot (padded to 256 bytes, so
  // that u rows start 16-byte aligned for the merge's vector loads), u per chunk slot
  const size_t pref_bytes = ((static_cast<size_t>(B) + 1) * sizeof(int) + 15) & ~size_t(15);
  const size_t ml_bytes = (static_cast<size_t>(items_max) * G * sizeof(float2) + 255) & ~size_t(255);
  const size_t o_bytes = static_cast<size_t>(items_max) * G * d * sizeof(float);
  const size_t need = pref_bytes + ml_bytes + o_bytes;
  std::lock_guard<std::mutex> lock(g_dec_mu);
  DecWorkspace& ws = g_dec_ws[dev];
  if (need > ws.bytes) {
    if (ws.buf) cudaFree(ws.buf);
    ws.buf = nullptr;
    ws.bytes = 0;
    if (cudaMalloc(&ws.buf, need) != cudaSuccess) return ATTN_ENOMEM;
    ws.bytes = need;
  }
  uint8_t* base = static_cast<uint8_t*>(ws.buf);
  int* pref = reinterpret_cast<int*>(base);
  float2* part_ml = reinterpret_cast<float2*>(base + pref_bytes);
  float* part_o = reinterpret_cast<float*>(base + pref_bytes + ml_bytes);

  attn_decode_prep_kernel<<<1, 32, 0, stream>>>(cu_k, B, total_k, pref, info.err_word);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  const int grid = total_k > 0 ? static_cast<int>(items_max) : 0;
  const float scale_log2 = scale * 1.4426950408889634f;
  cudaError_t e;
  if (d == 64)
    e = bf16 ? launch_d<64, true>(G, grid, q, k, v, cu_k, pref, part_o, part_ml, o, lse, B, Hq, Hkv, scale_log2, stream)
             : launch_d<64, false>(G, grid, q, k, v, cu_k, pref, part_o, part_ml, o, lse, B, Hq, Hkv, scale_log2, stream);
  else
    e = bf16 ? launch_d<128, true>(G, grid, q, k, v, cu_k, pref, part_o, part_ml, o, lse, B, Hq, Hkv, scale_log2, stream)
             : launch_d<128, false>(G, grid, q, k, v, cu_k, pref, part_o, part_ml, o, lse, B, Hq, Hkv, scale_log2, stream);
  if (e != cudaSuccess) return ATTN_ELAUNCH;
  for (int i = 0; i < (grid > 0 ? 3 : 2); ++i) count_launch();
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" {

int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                int total_k, int d, float scale, const int* cu_seqlens_k, int fp16, cudaStream_t stream) {
  if (fp16 != 0 && fp16 != 1) return ATTN_EINVAL;
  return attn::decode(fp16 == 0, q, k, v, o, lse, B, Hq, Hkv, total_k, d, scale, cu_seqlens_k, stream);
}

}  // extern "C"
