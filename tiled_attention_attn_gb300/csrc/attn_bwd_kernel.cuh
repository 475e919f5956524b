// sm_103a attention backward: the gradients dq, dk, dv of sum(dout * O),
// with the attention weights recomputed tile by tile from q, k and the lse
// the forward kept (lei6393.com training-integration page, §5.3: nothing of
// size L x L is stored).  Per (query i, key j) of one head, with scores
// s_ij = scale q_i.k_j:
//
//   P_ij  = exp(s_ij - lse_i)
//   dP_ij = dout_i . v_j
//   dS_ij = P_ij (dP_ij - D_i),   D_i = dout_i . O_i   (= sum_j P_ij dP_ij)
//   dv_j  = sum_i P_ij dout_i,  dk_j = scale sum_i dS_ij q_i,  dq_i = scale sum_j dS_ij k_j
//
// Two kernels, each with one contraction direction so that every MMA operand
// is in a layout the tensor cores read directly and no accumulator is shared
// between CTAs (no atomics; results are deterministic):
//   attn_bwd_kv_kernel  one CTA per (batch, KV head, 128-key tile): streams the
//                       query tiles of every query head of the group, forms
//                       S^T = K Q^T and dP^T = V dO^T, then P^T and dS^T per key
//                       row, and accumulates dv += P^T dO, dk += dS^T Q in TMEM.
//   attn_bwd_q_kernel   one CTA per (batch, query head, 128-query tile): streams
//                       the key tiles, forms S = Q K^T and dP = dO V^T, then dS
//                       per query row, and accumulates dq += dS K in TMEM.
// The second recomputes S and dP (two contractions more than a single pass
// with shared dq accumulation), in exchange for no atomics.
//
// CTA layout (320 threads): warps 0-7 process rows, warp w owning TMEM lanes
// 32 (w % 4) .. +31 (one row of the 128-row tile per lane) and columns
// 64 (w / 4) .. +63 of the 128-wide S and dP tiles; warp 8 issues TMA, warp 9
// allocates TMEM and one thread issues tcgen05.mma.  (Sixteen row warps of 32
// columns each measured slower: 0.809 against 0.780 ms.)  TMEM columns: S at
// [0,128), dP at [128,256), the accumulators from 256 on; the q kernel also
// keeps its Q and dO rows there as the A operands of S and dP.  The 16-bit P
// (kv kernel) and dS of a warp's columns are packed into the first half of
// those columns, so no warp writes where another still reads; the MMAs read
// the 16-column slices of the A operand from there, and are issued before the
// next tile's S and dP, which the tensor pipe runs after them.  The row
// threads signal P and dS separately, so each kernel's next S (and dP) is
// computed while the rows are still busy with this tile.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_params.h"
#include "ptx.cuh"

namespace attn {

// Row warps: warp w owns TMEM lanes 32 (w % 4) .. +31 and column part w / 4
// of the 128-wide S and dP tiles (kBwdCols columns).
constexpr int kBwdParts = 2;
constexpr int kBwdCols = 128 / kBwdParts;
constexpr int kBwdRowWarps = 4 * kBwdParts;
constexpr int kBwdWarpTMA = kBwdRowWarps;
constexpr int kBwdWarpMMA = kBwdRowWarps + 1;
constexpr int kBwdThreads = 32 * (kBwdRowWarps + 2);

struct BwdParams {
  CUtensorMap tm_q;        // (d, Hq, Lq, B), box 64 x 1 x 128 x 1
  CUtensorMap tm_k;        // (d, Hkv, Lk, B)
  CUtensorMap tm_v;
  CUtensorMap tm_do;       // like q
  const void* q;           // (B, Lq, Hq, d): the q kernel reads its Q and dO rows directly
  const void* dout;
  const float* lse2;       // dense [B][Hq][Lq_pad], varlen [Hq][query tiles][128]: lse * log2(e);
                           // +inf for rows with no key and on the padding of every tile
  const float* dvec;       // same layout: D_i = dout_i . O_i; 0 on the padding
  const int* cu_q;         // varlen: query and key offsets (B+1 each), else null
  const int* cu_k;
  const int* tile_pref;    // varlen: query tiles before sequence b (B+1), then key tiles (B+1)
  void* dq;                // like q
  void* dk;                // like k
  void* dv;                // like k
  int* err;
  unsigned long long timeout_ns;
  unsigned long long* trace;   // phase trace (traced build, attn_trace_enable), else null
  int trace_cap;               // events per stream per traced CTA
  int B, Hq, Hkv, Lq, Lk, group, Lq_pad, n_qt, n_kt;
  float scale, scale_log2;
};

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = 128 * D * 2;         // one 128-row tile in smem
  static constexpr int kNS = (D == 128) ? 2 : 4;    // stages of the streamed operands
  // kv kernel: K, V resident; stages of (Q, dO, lse2, D)
  static constexpr int kKvOffStage = 2 * kTile;
  static constexpr int kKvStageBytes = 2 * kTile;
  static constexpr int kKvOffVec = kKvOffStage + kNS * kKvStageBytes;   // per stage 128 + 128 floats
  static constexpr int kKvOffBar = kKvOffVec + kNS * 1024;
  // q kernel: Q and dO live in TMEM (the A operands of S and dP), so shared
  // memory holds only stages of (K, V)
  static constexpr int kQNS = (D == 128) ? 3 : 6;
  static constexpr int kQOffStage = 0;
  static constexpr int kQOffBar = kQOffStage + kQNS * 2 * kTile;
  static constexpr int kQNBars = 1 + 2 * kQNS + 6;
  static constexpr uint32_t kColQ = 384;             // Q packed, D/2 columns
  static constexpr uint32_t kColDO = 384 + D / 2;    // dO packed, D/2 columns
  // barriers: full (resident pair), st_full[NS], st_empty[NS], s_full, dp_full, and two
  // row-side signals (kv: p_full, ds_full; q: s_free, ds_full), acc_done, drain
  static constexpr int kNBars = 1 + 2 * kNS + 6;
  static constexpr int kKvSmem = kKvOffBar + kNBars * 8 + 64 + 1024;
  static constexpr int kQSmem = kQOffBar + kQNBars * 8 + 64 + 1024;
  static constexpr uint32_t kTmemCols = 512;
};

// Phase trace of the first 160 CTAs (linear block id): streams 0-3 for the
// kv kernel and 4-7 for the q kernel (MMA thread, row warp 0, row warp 4,
// producer); an event is (tag << 32 | tile) and the SM clock.  Compiled in
// only when ATTN_TRACE is 1.
#ifndef ATTN_TRACE
#define ATTN_TRACE 0
#endif
struct BwdTracer {
  unsigned long long* base;
  int cap, n;
  __device__ __forceinline__ void init(const BwdParams& p, int stream, bool on) {
    const int cta = blockIdx.x + gridDim.x * blockIdx.y;
    base = (ATTN_TRACE && on && p.trace && cta < 160)
               ? p.trace + (static_cast<size_t>(cta) * 8 + stream) * p.trace_cap * 2
               : nullptr;
    cap = p.trace_cap;
    n = 0;
  }
  __device__ __forceinline__ void rec(int tag, int t) {
    if (ATTN_TRACE && base != nullptr && n < cap) {
      base[2 * n] = (static_cast<unsigned long long>(tag) << 32) | static_cast<unsigned>(t);
      base[2 * n + 1] = clock64();
      ++n;
    }
  }
};

template <bool BF16>
struct BwdIO;
template <>
struct BwdIO<true> {
  using T = __nv_bfloat16;
};
template <>
struct BwdIO<false> {
  using T = __half;
};

// Stores 32 fp32 values (times `mul`) of one row as 16-bit, 64 bytes.
template <bool BF16>
__device__ __forceinline__ void store_row32(void* dst, const uint32_t (&x)[32], float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(__uint_as_float(x[2 * i]) * mul, __uint_as_float(x[2 * i + 1]) * mul);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

// Largest b with pref[b] <= x (pref non-decreasing, pref[0] = 0 <= x < pref[B]).
__device__ __forceinline__ int seq_of(const int* pref, int B, int x) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(pref + mid) <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// varlen: validates the offsets and counts 128-row tiles per sequence
// (pref[b] = query tiles before sequence b, pref[B+1+b] = key tiles before
// it); one warp.  Malformed offsets set the error word and zero the totals,
// so the kernels that follow find no work.
// ---------------------------------------------------------------------------
static __global__ void __launch_bounds__(32) attn_bwd_tiles_kernel(const int* __restrict__ cu_q, const int* __restrict__ cu_k,
                                                           int B, int total_q, int total_k, int* __restrict__ pref,
                                                           int* __restrict__ err) {
  const int lane = threadIdx.x;
  bool bad = lane == 0 && (__ldg(cu_q) != 0 || __ldg(cu_k) != 0);
  int cq = 0, ck = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    int nq = 0, nk = 0;
    if (b < B) {
      const int a = __ldg(cu_q + b), e = __ldg(cu_q + b + 1), ak = __ldg(cu_k + b), ek = __ldg(cu_k + b + 1);
      if (e < a || e > total_q || ek < ak || ek > total_k) bad = true;
      nq = e > a ? (e - a + kBM - 1) / kBM : 0;
      nk = ek > ak ? (ek - ak + kBN - 1) / kBN : 0;
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yq = __shfl_up_sync(0xffffffffu, nq, o), yk = __shfl_up_sync(0xffffffffu, nk, o);
      if (lane >= o) {
        nq += yq;
        nk += yk;
      }
    }
    if (b < B) {
      pref[b + 1] = cq + nq;
      pref[B + 1 + b + 1] = ck + nk;
    }
    cq += __shfl_sync(0xffffffffu, nq, 31);
    ck += __shfl_sync(0xffffffffu, nk, 31);
  }
  if (__any_sync(0xffffffffu, bad)) {
    __syncwarp();
    if (lane == 0) {
      pref[B] = 0;
      pref[2 * B + 1] = 0;
      atomicCAS(err, 0, ATTN_DEVERR_BAD_SEQLENS);
    }
  }
  if (lane == 0) {
    pref[0] = 0;
    pref[B + 1] = 0;
  }
}

// Dot product of 8 threads' shares of a 16-bit row pair (D / 8 elements each).
template <int D, bool BF16>
__device__ __forceinline__ float row_dot8(const void* o, const void* dout, size_t at, int sub) {
  using T = typename BwdIO<BF16>::T;
  constexpr int kPer = D / 8;
  const T* po = reinterpret_cast<const T*>(o) + at + sub * kPer;
  const T* pd = reinterpret_cast<const T*>(dout) + at + sub * kPer;
  float acc = 0.0f;
#pragma unroll
  for (int w = 0; w < kPer / 8; ++w) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(po) + w);
    const uint4 c = __ldg(reinterpret_cast<const uint4*>(pd) + w);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 fa, fc;
      if constexpr (BF16) {
        fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
        fc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&cw[e]));
      } else {
        fa = __half22float2(*reinterpret_cast<const __half2*>(&aw[e]));
        fc = __half22float2(*reinterpret_cast<const __half2*>(&cw[e]));
      }
      acc = fmaf(fa.x, fc.x, acc);
      acc = fmaf(fa.y, fc.y, acc);
    }
  }
  return acc;
}

// varlen D_i and lse in exp2 units, one slot (h, query tile, row) per 8
// threads: slot s is written at index s of [Hq][query tiles][128]; rows past
// their sequence's end get the padding values.  q, o, dout packed
// (total_q, Hq, d); lse (Hq, total_q).
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_prep_varlen_kernel(const void* __restrict__ o,
                                                                   const void* __restrict__ dout,
                                                                   const float* __restrict__ lse,
                                                                   const int* __restrict__ cu_q,
                                                                   const int* __restrict__ pref, int B, int Hq,
                                                                   int total_q, float* __restrict__ lse2,
                                                                   float* __restrict__ dvec) {
  const long long qt = __ldg(pref + B);
  const long long slots = static_cast<long long>(Hq) * qt * kBM;
  const int sub = threadIdx.x & 7;
  const long long stride = (static_cast<long long>(gridDim.x) * blockDim.x) >> 3;
  for (long long base = (static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31)) >> 3; base < slots;
       base += stride) {   // warp-uniform bound: the shuffles below need all 32 lanes
    const long long s_raw = base + ((threadIdx.x & 31) >> 3);
    const bool in = s_raw < slots;
    const long long sl = in ? s_raw : slots - 1;
    const int h = static_cast<int>(sl / (qt * kBM));
    const long long rest = sl - static_cast<long long>(h) * qt * kBM;
    const int T = static_cast<int>(rest / kBM), rr = static_cast<int>(rest - static_cast<long long>(T) * kBM);
    const int b = seq_of(pref, B, T);
    const int q0 = __ldg(cu_q + b), len = __ldg(cu_q + b + 1) - q0;
    const int i = (T - __ldg(pref + b)) * kBM + rr;
    const bool valid = in && i < len;
    const size_t row = static_cast<size_t>(q0) + (valid ? i : 0);
    float acc = valid ? row_dot8<D, BF16>(o, dout, (row * Hq + h) * D, sub) : 0.0f;
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (in && sub == 0) {
      float l2 = INFINITY;
      if (valid) {
        const float l = __ldg(lse + static_cast<size_t>(h) * total_q + row);
        l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
      }
      lse2[sl] = l2;
      dvec[sl] = valid ? acc : 0.0f;
    }
  }
}

// One warp's columns of its 32 lanes in one TMEM load (32 or 64 columns).
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld_32x32b_x32(taddr, r); }
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[64]) { tmem_ld_32x32b_x64(taddr, r); }

// Stores 16 fp32 values (times `mul`) of one row as 16-bit, 32 bytes.
template <bool BF16>
__device__ __forceinline__ void store_row16(void* dst, const uint32_t (&x)[16], float mul) {
  uint32_t pk[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) pk[i] = pack2<BF16>(__uint_as_float(x[2 * i]) * mul, __uint_as_float(x[2 * i + 1]) * mul);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

// ---------------------------------------------------------------------------
// D_i = dout_i . O_i and lse in exp2 units, one (b, h, i) row per 8 threads;
// rows i in [Lq, Lq_pad) get the padding values.
// ---------------------------------------------------------------------------
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const void* __restrict__ o, const void* __restrict__ dout,
                                                            const float* __restrict__ lse, float* __restrict__ lse2,
                                                            float* __restrict__ dvec, int B, int Hq, int Lq,
                                                            int Lq_pad) {
  using T = typename BwdIO<BF16>::T;
  constexpr int kPer = D / 8;   // elements per thread
  const long long items = static_cast<long long>(B) * Lq_pad * Hq;
  const int sub = threadIdx.x & 7;
  // the loop bound is warp-uniform (the shuffles below need all 32 lanes)
  const long long stride = (static_cast<long long>(gridDim.x) * blockDim.x) >> 3;
  for (long long base = (static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31)) >> 3; base < items;
       base += stride) {
    const long long it_raw = base + ((threadIdx.x & 31) >> 3);
    const bool valid = it_raw < items;
    const long long it = valid ? it_raw : items - 1;
    // (b, h, i) with i fastest: the lse reads and the lse2 / D writes of a
    // warp are contiguous; each O / dO row is still read as whole 256-byte
    // segments
    const int i = static_cast<int>(it % Lq_pad);
    const long long bh = it / Lq_pad;
    const int h = static_cast<int>(bh % Hq);
    const int b = static_cast<int>(bh / Hq);
    float acc = 0.0f;
    if (valid && i < Lq) {
      const size_t rb = ((static_cast<size_t>(b) * Lq + i) * Hq + h) * D + sub * kPer;
      const T* po = reinterpret_cast<const T*>(o) + rb;
      const T* pd = reinterpret_cast<const T*>(dout) + rb;
#pragma unroll
      for (int w = 0; w < kPer / 8; ++w) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(po) + w);
        const uint4 c = __ldg(reinterpret_cast<const uint4*>(pd) + w);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 fa, fc;
          if constexpr (BF16) {
            fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
            fc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&cw[e]));
          } else {
            fa = __half22float2(*reinterpret_cast<const __half2*>(&aw[e]));
            fc = __half22float2(*reinterpret_cast<const __half2*>(&cw[e]));
          }
          acc = fmaf(fa.x, fc.x, acc);
          acc = fmaf(fa.y, fc.y, acc);
        }
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (valid && sub == 0) {
      const size_t li = (static_cast<size_t>(b) * Hq + h) * Lq_pad + i;
      float l2 = INFINITY;
      if (i < Lq) {
        const float l = __ldg(lse + (static_cast<size_t>(b) * Hq + h) * Lq + i);
        l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
      }
      lse2[li] = l2;
      dvec[li] = (i < Lq) ? acc : 0.0f;
    }
  }
}

// TMEM column of the packed 16-bit A operand's kk-th 16-wide K slice inside a
// 128-column S or dP region: column part c packs its kBwdCols columns into
// the first kBwdCols / 2 of them.
__device__ __forceinline__ uint32_t packed_slice_col(int kk) {
  constexpr int kSlices = kBwdCols / 16;   // K slices per column part
  return (kk / kSlices) * kBwdCols + (kk % kSlices) * 8;
}

// kv kernel, one warp's kBwdCols query columns of its 32 key rows:
// P^T = 2^(S^T c - lse2) (c = scale log2 e), kept in pr and stored packed over
// the first half of its columns.  MASK: query column c is allowed iff
// c >= cmin (causal).
template <bool MASK, bool BF16>
__device__ __forceinline__ void kv_p_part(uint32_t t_s, const float* ls, int cmin, float cl2,
                                          float (&pr)[kBwdCols]) {
#pragma unroll
  for (int ch = 0; ch < kBwdCols / 32; ++ch) {
    uint32_t sr[32];
    tmem_ld_32x32b_x32(t_s + ch * 32, sr);
    tmem_wait_ld(sr);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      // the exponent arguments with packed fp32x2 FMA: scalar FMA streams on
      // the MMA issuer's sub-partition slow its issue
      const float4 l4 = *reinterpret_cast<const float4*>(ls + ch * 32 + e);
      const float2 c2 = make_float2(cl2, cl2);
      const float2 a0 = ffma2(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2,
                              make_float2(-l4.x, -l4.y));
      const float2 a1 = ffma2(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), c2,
                              make_float2(-l4.z, -l4.w));
      const float xs[4] = {ex2_approx(a0.x), ex2_approx(a0.y), ex2_approx(a1.x), ex2_approx(a1.y)};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = ch * 32 + e + u;
        pr[c] = (!MASK || c >= cmin) ? xs[u] : 0.0f;
      }
      pk[e / 2] = pack2<BF16>(pr[ch * 32 + e], pr[ch * 32 + e + 1]);
      pk[e / 2 + 1] = pack2<BF16>(pr[ch * 32 + e + 2], pr[ch * 32 + e + 3]);
    }
    tmem_st_32x32b_x16(t_s + ch * 16, pk);
  }
}

// dS = P (dP - D) for one warp's kBwdCols columns, stored packed over the
// first half of its dP columns.  dd: D per column (kv kernel), or null with `di` the
// row's D (q kernel).
template <bool BF16>
__device__ __forceinline__ void ds_part(uint32_t t_dp, const float* dd, float di, const float (&pr)[kBwdCols]) {
#pragma unroll
  for (int ch = 0; ch < kBwdCols / 32; ++ch) {
    uint32_t dr[32];
    tmem_ld_32x32b_x32(t_dp + ch * 32, dr);
    tmem_wait_ld(dr);
    uint32_t dk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      float dv4[4] = {di, di, di, di};
      if (dd != nullptr) {
        const float4 d4 = *reinterpret_cast<const float4*>(dd + ch * 32 + e);
        dv4[0] = d4.x;
        dv4[1] = d4.y;
        dv4[2] = d4.z;
        dv4[3] = d4.w;
      }
      const float2 d0 = fmul2(make_float2(pr[ch * 32 + e], pr[ch * 32 + e + 1]),
                              fadd2(make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])),
                                    make_float2(-dv4[0], -dv4[1])));
      const float2 d1 = fmul2(make_float2(pr[ch * 32 + e + 2], pr[ch * 32 + e + 3]),
                              fadd2(make_float2(__uint_as_float(dr[e + 2]), __uint_as_float(dr[e + 3])),
                                    make_float2(-dv4[2], -dv4[3])));
      dk[e / 2] = pack2<BF16>(d0.x, d0.y);
      dk[e / 2 + 1] = pack2<BF16>(d1.x, d1.y);
    }
    tmem_st_32x32b_x16(t_dp + ch * 16, dk);
  }
}

// q kernel, one warp's kBwdCols key columns of its 32 query rows, from S already
// in registers: P = 2^(S c - lse2_i) in pr.  MASK: key column c is allowed
// iff c <= lim.
template <bool MASK>
__device__ __forceinline__ void q_p_part(const uint32_t (&sr)[kBwdCols], float l2, int lim, float cl2,
                                         float (&pr)[kBwdCols]) {
  const float2 c2 = make_float2(cl2, cl2), nl = make_float2(-l2, -l2);
#pragma unroll
  for (int c = 0; c < kBwdCols; c += 2) {
    const float2 a = ffma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2, nl);
    const float x0 = ex2_approx(a.x), x1 = ex2_approx(a.y);
    pr[c] = (!MASK || c <= lim) ? x0 : 0.0f;
    pr[c + 1] = (!MASK || c + 1 <= lim) ? x1 : 0.0f;
  }
}

// ---------------------------------------------------------------------------
// dk, dv: one CTA per (b, g, 128-key tile n); grid (B * Hkv, n_kt)
// ---------------------------------------------------------------------------
template <int D, bool BF16, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_kv_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase, sV = sbase + C::kTile;
  auto sQ = [&](int s) { return sbase + C::kKvOffStage + s * C::kKvStageBytes; };
  auto sDO = [&](int s) { return sbase + C::kKvOffStage + s * C::kKvStageBytes + C::kTile; };
  const float* vec = reinterpret_cast<const float*>(smem + C::kKvOffVec);   // [stage][lse2 128 | D 128]
  const uint32_t bar0 = sbase + C::kKvOffBar;
  const uint32_t b_kv_full = bar0;
  auto b_st_full = [&](int s) { return bar0 + 8 + 8 * s; };
  auto b_st_empty = [&](int s) { return bar0 + 8 + 8 * (C::kNS + s); };
  const uint32_t b_s_full = bar0 + 8 + 16 * C::kNS;   // S^T(t) computed
  const uint32_t b_dp_full = b_s_full + 8;            // dP^T(t) computed
  const uint32_t b_p_full = b_s_full + 16;            // P^T(t) stored by the key rows
  const uint32_t b_ds_full = b_s_full + 24;           // dS^T(t) stored by the key rows
  const uint32_t b_acc = b_s_full + 32;
  const uint32_t b_drain = b_s_full + 40;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kKvOffBar + C::kNBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kKvOffBar + C::kNBars * 8 + 4);
  WaitCtl wc{p.err, abort_flag, p.timeout_ns};

  // this CTA's sequence b, KV head g and key tile n; q_len / k_len its
  // lengths, rq / rk the global row of its first query / key (dense: b * L)
  int b, g, n, q_len, k_len, rq, rk, nqt;
  if constexpr (!VARLEN) {
    const int bg = blockIdx.x;
    n = blockIdx.y;
    b = bg / p.Hkv;
    g = bg - b * p.Hkv;
    q_len = p.Lq;
    k_len = p.Lk;
    rq = b * p.Lq;
    rk = b * p.Lk;
    nqt = p.n_qt;
  } else {
    const int* kpref = p.tile_pref + p.B + 1;
    const int u = blockIdx.x;
    if (u >= __ldg(kpref + p.B) * p.Hkv) return;   // beyond the work: before any barrier or TMEM use
    const int nt = u / p.Hkv;
    g = u - nt * p.Hkv;
    b = seq_of(kpref, p.B, nt);
    n = nt - __ldg(kpref + b);
    rq = __ldg(p.cu_q + b);
    rk = __ldg(p.cu_k + b);
    q_len = __ldg(p.cu_q + b + 1) - rq;
    k_len = __ldg(p.cu_k + b + 1) - rk;
    nqt = (q_len + kBM - 1) / kBM;
  }
  // TMA coordinates: dense maps are (d, H, L, B), packed ones (d, H, total, 1)
  const int trow_q = VARLEN ? rq : 0, trow_k = VARLEN ? rk : 0, bc = VARLEN ? 0 : b;
  auto vtile = [&](int h, int m) -> size_t {   // first lse2 / D entry of query tile m of head h
    return VARLEN ? (static_cast<size_t>(h) * __ldg(p.tile_pref + p.B) + __ldg(p.tile_pref + b) + m) * kBM
                  : (static_cast<size_t>(b) * p.Hq + h) * p.Lq_pad + static_cast<size_t>(m) * kBM;
  };
  const int off = k_len - q_len;   // causal: key j is visible to query i iff j <= i + off
  int m_first = 0;
  if constexpr (CAUSAL) {
    const int first_q = n * kBN - off;   // smallest query that sees key n * 128
    m_first = first_q <= 0 ? 0 : first_q / kBM;
  }
  const int nm = nqt - m_first > 0 ? nqt - m_first : 0;
  const int n_tiles = p.group * nm;

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(b_kv_full, 1);
    for (int s = 0; s < C::kNS; ++s) {
      mbar_init(b_st_full(s), 1);
      mbar_init(b_st_empty(s), 1);
    }
    mbar_init(b_s_full, 1);
    mbar_init(b_dp_full, 1);
    mbar_init(b_p_full, kBwdRowWarps);
    mbar_init(b_ds_full, kBwdRowWarps);
    mbar_init(b_acc, 1);
    mbar_init(b_drain, 1);
    fence_mbar_init();
  }
  if (warp == kBwdWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kBwdWarpTMA) {
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      mbar_arrive_expect_tx(b_kv_full, 2 * C::kTile);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_4d(sK + c * 16384, &p.tm_k, b_kv_full, c * 64, g, trow_k + n * kBN, bc);
        tma_load_4d(sV + c * 16384, &p.tm_v, b_kv_full, c * 64, g, trow_k + n * kBN, bc);
      }
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int st = t % C::kNS;
        if (!mbar_wait(b_st_empty(st), ((t / C::kNS) & 1) ^ 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKEmpty))) break;
        const int h = g * p.group + t / nm, m = m_first + t % nm;
        mbar_arrive_expect_tx(b_st_full(st), 2 * C::kTile + 1024);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_4d(sQ(st) + c * 16384, &p.tm_q, b_st_full(st), c * 64, h, trow_q + m * kBM, bc);
          tma_load_4d(sDO(st) + c * 16384, &p.tm_do, b_st_full(st), c * 64, h, trow_q + m * kBM, bc);
        }
        const size_t vi = vtile(h, m);
        const uint32_t sv = smem_u32(vec + st * 256);
        bulk_load(sv, p.lse2 + vi, 512, b_st_full(st));
        bulk_load(sv + 512, p.dvec + vi, 512, b_st_full(st));
        ++issued;
      }
      if (*abort_flag) {
        // let issued loads land before the CTA exits
        mbar_wait(b_kv_full, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
        for (int s = 0; s < C::kNS; ++s) {
          const int cnt = (issued + C::kNS - 1 - s) / C::kNS;
          if (cnt > 0) mbar_wait(b_st_full(s), (cnt - 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
        }
      }
    }
  } else if (warp == kBwdWarpMMA) {
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_f16_f32acc(128, 128, BF16, false);
      constexpr uint32_t kIdescO = idesc_f16_f32acc(128, D, BF16, true);
      const uint64_t dk_k = sdesc_sw128(sK, 16, 1024);     // K as A, K-major
      const uint64_t dv_k = sdesc_sw128(sV, 16, 1024);     // V as A, K-major
      auto issue_s = [&](int st) {   // S^T = K Q^T
        const uint64_t dq_k = sdesc_sw128(sQ(st), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_ss(tmem + 0, dk_k + o, dq_k + o, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(b_s_full);
      };
      auto issue_dp = [&](int st) {   // dP^T = V dO^T
        const uint64_t ddo_k = sdesc_sw128(sDO(st), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_ss(tmem + 128, dv_k + o, ddo_k + o, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(b_dp_full);
      };
      // Order per tile t: dv(t), S^T(t+1), dk(t), dP^T(t+1).  S^T(t+1)
      // overwrites P^T(t) after dv(t) has been issued, dP^T(t+1) overwrites
      // dS^T(t) after dk(t); the key rows form P^T(t+1) while dk(t) and
      // dP^T(t+1) run, and dS^T(t) while dv(t) and S^T(t+1) run.
      BwdTracer tr;
      tr.init(p, 0, true);
      bool ok = n_tiles > 0 && mbar_wait(b_kv_full, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteQFull)) &&
                mbar_wait(b_st_full(0), 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKFull));
      if (ok) {
        issue_s(0);
        issue_dp(0);
      }
      for (int t = 0; ok && t < n_tiles; ++t) {
        const int st = t % C::kNS, st1 = (t + 1) % C::kNS;
        const bool next = t + 1 < n_tiles;
        tr.rec(1, t);
        if (!mbar_wait(b_p_full, t & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSitePFull))) break;
        tr.rec(2, t);
        tc_fence_after();
        const uint64_t ddo_mn = sdesc_sw128(sDO(st), 16384, 1024);   // dO as B, MN-major
        const uint64_t dq_mn = sdesc_sw128(sQ(st), 16384, 1024);     // Q as B, MN-major
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk)   // dv += P^T dO
          umma_ts(tmem + 256, tmem + packed_slice_col(kk), ddo_mn + ((kk * 2048) >> 4), kIdescO,
                  (t > 0 || kk > 0) ? 1u : 0u);
        tr.rec(3, t);
        if (next) {
          if (!mbar_wait(b_st_full(st1), ((t + 1) / C::kNS) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKFull))) break;
          tr.rec(4, t);
          issue_s(st1);
          tr.rec(5, t);
        }
        if (!mbar_wait(b_ds_full, t & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDsFull))) break;
        tr.rec(6, t);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk)   // dk += dS^T Q
          umma_ts(tmem + 256 + D, tmem + 128 + packed_slice_col(kk), dq_mn + ((kk * 2048) >> 4), kIdescO,
                  (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit(b_st_empty(st));
        tr.rec(7, t);
        if (next) issue_dp(st1);
        tr.rec(8, t);
      }
      umma_commit(b_acc);
      umma_commit(b_drain);
      mbar_wait(b_drain, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
    }
  } else {
    // ---------------------------------------------------------------- key rows
    const int quarter = warp & 3, part = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int c0 = part * kBwdCols;   // this warp's first column of S and dP
    const uint32_t t_s = tmem + lane_off + c0, t_dp = tmem + lane_off + 128 + c0;
    const int j = n * kBN + row;
    const float cl2 = p.scale_log2;
    BwdTracer tr;
    tr.init(p, part == 0 ? 1 : 2, lane == 0 && quarter == 0 && part < 2);
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      tr.rec(20, t);
      if (!mbar_wait_warp(b_s_full, t & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteSFull))) { ok = false; break; }
      tr.rec(21, t);
      tc_fence_after();
      const int st = t % C::kNS, m = m_first + t % nm;
      // lse2 and D of this stage came by bulk copy: observe its completion
      // here (the stage cannot be refilled before this warp arrives on ds_full)
      if (!mbar_wait_warp(b_st_full(st), (t / C::kNS) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKFull))) {
        ok = false;
        break;
      }
      const float* ls = vec + st * 256 + c0;
      const float* dd = vec + st * 256 + 128 + c0;
      // Only tiles crossing the causal diagonal are masked.  Padded query
      // columns (past Lq) have lse2 = +inf, so P = 0 there; padded key rows
      // (past Lk) only reach their own rows of dv and dk, which are not stored.
      float pr[kBwdCols];
      if (CAUSAL && n * kBN + kBN - 1 - m * kBM > off)
        kv_p_part<true, BF16>(t_s, ls, j - off - m * kBM - c0, cl2, pr);
      else
        kv_p_part<false, BF16>(t_s, ls, 0, cl2, pr);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_p_full);
      tr.rec(22, t);
      if (!mbar_wait_warp(b_dp_full, t & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteODone))) { ok = false; break; }
      tr.rec(23, t);
      tc_fence_after();
      ds_part<BF16>(t_dp, dd, 0.0f, pr);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_ds_full);
      tr.rec(24, t);
    }
    // epilogue: dv = acc, dk = scale * acc; this warp's part of the columns
    if (ok && (n_tiles == 0 || mbar_wait_warp(b_acc, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteODone)))) {
      tc_fence_after();
      using T = typename BwdIO<BF16>::T;
      constexpr int kHalf = D / kBwdParts;   // accumulator columns per warp
      const size_t orow = ((static_cast<size_t>(rk) + j) * p.Hkv + g) * D + part * kHalf;
      T* dvp = reinterpret_cast<T*>(p.dv) + orow;
      T* dkp = reinterpret_cast<T*>(p.dk) + orow;
      if (n_tiles == 0) {
        if (j < k_len) {
#pragma unroll
          for (int i = 0; i < kHalf / 8; ++i) {
            reinterpret_cast<uint4*>(dvp)[i] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4*>(dkp)[i] = make_uint4(0, 0, 0, 0);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < kHalf / 16; ++c) {
          uint32_t x[16];
          tmem_ld_32x32b_x16(tmem + lane_off + 256 + part * kHalf + c * 16, x);
          tmem_wait_ld(x);
          if (j < k_len) store_row16<BF16>(dvp + c * 16, x, 1.0f);
        }
#pragma unroll
        for (int c = 0; c < kHalf / 16; ++c) {
          uint32_t x[16];
          tmem_ld_32x32b_x16(tmem + lane_off + 256 + D + part * kHalf + c * 16, x);
          tmem_wait_ld(x);
          if (j < k_len) store_row16<BF16>(dkp + c * 16, x, p.scale);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kBwdWarpMMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// dq: one CTA per (b, h, 128-query tile m); grid (B * Hq, n_qt), heaviest
// (last) query tiles first
// ---------------------------------------------------------------------------
template <int D, bool BF16, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_q_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  auto sK = [&](int s) { return sbase + C::kQOffStage + s * 2 * C::kTile; };
  auto sV = [&](int s) { return sbase + C::kQOffStage + s * 2 * C::kTile + C::kTile; };
  const uint32_t bar0 = sbase + C::kQOffBar;
  const uint32_t b_q_full = bar0;   // the rows have stored Q and dO in TMEM
  auto b_st_full = [&](int s) { return bar0 + 8 + 8 * s; };
  auto b_st_empty = [&](int s) { return bar0 + 8 + 8 * (C::kQNS + s); };
  const uint32_t b_s_full = bar0 + 8 + 16 * C::kQNS;   // S(t) computed
  const uint32_t b_dp_full = b_s_full + 8;            // dP(t) computed
  const uint32_t b_s_free = b_s_full + 16;            // the query rows have read S(t)
  const uint32_t b_ds_full = b_s_full + 24;           // dS(t) stored by the query rows
  const uint32_t b_acc = b_s_full + 32;
  const uint32_t b_drain = b_s_full + 40;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kQOffBar + C::kQNBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kQOffBar + C::kQNBars * 8 + 4);
  WaitCtl wc{p.err, abort_flag, p.timeout_ns};

  // this CTA's sequence b, query head h and query tile m (see the kv kernel)
  int b, h, m, q_len, k_len, rq, rk, nkt;
  if constexpr (!VARLEN) {
    const int bh = blockIdx.x;
    m = p.n_qt - 1 - static_cast<int>(blockIdx.y);
    b = bh / p.Hq;
    h = bh - b * p.Hq;
    q_len = p.Lq;
    k_len = p.Lk;
    rq = b * p.Lq;
    rk = b * p.Lk;
    nkt = p.n_kt;
  } else {
    const int u = blockIdx.x;
    if (u >= __ldg(p.tile_pref + p.B) * p.Hq) return;   // beyond the work: before any barrier or TMEM use
    const int mt = u / p.Hq;
    h = u - mt * p.Hq;
    b = seq_of(p.tile_pref, p.B, mt);
    m = mt - __ldg(p.tile_pref + b);
    rq = __ldg(p.cu_q + b);
    rk = __ldg(p.cu_k + b);
    q_len = __ldg(p.cu_q + b + 1) - rq;
    k_len = __ldg(p.cu_k + b + 1) - rk;
    nkt = (k_len + kBN - 1) / kBN;
  }
  const int g = h / p.group;
  const int trow_k = VARLEN ? rk : 0, bc = VARLEN ? 0 : b;
  const int off = k_len - q_len;
  int n_tiles = nkt;
  if constexpr (CAUSAL) {
    int last_q = m * kBM + kBM - 1;
    if (last_q > q_len - 1) last_q = q_len - 1;
    const int max_key = last_q + off;
    n_tiles = max_key < 0 ? 0 : min(nkt, max_key / kBN + 1);
  }

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(b_q_full, kBwdRowWarps);
    for (int s = 0; s < C::kQNS; ++s) {
      mbar_init(b_st_full(s), 1);
      mbar_init(b_st_empty(s), 1);
    }
    mbar_init(b_s_full, 1);
    mbar_init(b_dp_full, 1);
    mbar_init(b_s_free, kBwdRowWarps);
    mbar_init(b_ds_full, kBwdRowWarps);
    mbar_init(b_acc, 1);
    mbar_init(b_drain, 1);
    fence_mbar_init();
  }
  if (warp == kBwdWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kBwdWarpTMA) {
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int st = t % C::kQNS;
        if (!mbar_wait(b_st_empty(st), ((t / C::kQNS) & 1) ^ 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKEmpty))) break;
        mbar_arrive_expect_tx(b_st_full(st), 2 * C::kTile);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_4d(sK(st) + c * 16384, &p.tm_k, b_st_full(st), c * 64, g, trow_k + t * kBN, bc);
          tma_load_4d(sV(st) + c * 16384, &p.tm_v, b_st_full(st), c * 64, g, trow_k + t * kBN, bc);
        }
        ++issued;
      }
      if (*abort_flag) {
        for (int s = 0; s < C::kQNS; ++s) {
          const int cnt = (issued + C::kQNS - 1 - s) / C::kQNS;
          if (cnt > 0) mbar_wait(b_st_full(s), (cnt - 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
        }
      }
    }
  } else if (warp == kBwdWarpMMA) {
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_f16_f32acc(128, 128, BF16, false);
      constexpr uint32_t kIdescO = idesc_f16_f32acc(128, D, BF16, true);
      auto issue_s = [&](int st) {   // S = Q K^T, Q from TMEM
        const uint64_t dk_k = sdesc_sw128(sK(st), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_ts(tmem + 0, tmem + C::kColQ + kk * 8, dk_k + o, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(b_s_full);
      };
      auto issue_dp = [&](int st) {   // dP = dO V^T, dO from TMEM
        const uint64_t dv_k = sdesc_sw128(sV(st), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_ts(tmem + 128, tmem + C::kColDO + kk * 8, dv_k + o, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(b_dp_full);
      };
      // Order per tile t: S(t+1) (once the rows have read S(t)), dq(t),
      // dP(t+1).  dS(t) lives over dP(t)'s columns, so S(t+1) does
      // not wait for dq(t); dP(t+1) is issued after dq(t) has been.
      BwdTracer tr;
      tr.init(p, 4, true);
      bool ok = n_tiles > 0 && mbar_wait(b_q_full, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteQFull)) &&
                mbar_wait(b_st_full(0), 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKFull));
      if (ok) {
        tc_fence_after();   // Q and dO were written into TMEM by the rows (tcgen05.st)
        issue_s(0);
        issue_dp(0);
      }
      for (int t = 0; ok && t < n_tiles; ++t) {
        const int st = t % C::kQNS, st1 = (t + 1) % C::kQNS;
        const bool next = t + 1 < n_tiles;
        tr.rec(1, t);
        if (next) {
          if (!mbar_wait(b_s_free, t & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSitePFull))) break;
          tr.rec(2, t);
          if (!mbar_wait(b_st_full(st1), ((t + 1) / C::kQNS) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKFull))) break;
          tr.rec(3, t);
          issue_s(st1);
          tr.rec(4, t);
        }
        if (!mbar_wait(b_ds_full, t & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDsFull))) break;
        tr.rec(6, t);
        tc_fence_after();
        const uint64_t dk_mn = sdesc_sw128(sK(st), 16384, 1024);   // K as B, MN-major
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk)   // dq += dS K
          umma_ts(tmem + 256, tmem + 128 + packed_slice_col(kk), dk_mn + ((kk * 2048) >> 4), kIdescO,
                  (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit(b_st_empty(st));
        tr.rec(7, t);
        if (next) issue_dp(st1);
        tr.rec(8, t);
      }
      umma_commit(b_acc);
      umma_commit(b_drain);
      mbar_wait(b_drain, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
    }
  } else {
    // ---------------------------------------------------------------- query rows
    const int quarter = warp & 3, part = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int c0 = part * kBwdCols;   // this warp's first column of S and dP
    const uint32_t t_s = tmem + lane_off + c0, t_dp = tmem + lane_off + 128 + c0;
    const int i = m * kBM + row;
    const float cl2 = p.scale_log2;
    const size_t vi = VARLEN ? (static_cast<size_t>(h) * __ldg(p.tile_pref + p.B) + __ldg(p.tile_pref + b) + m) * kBM + row
                             : (static_cast<size_t>(b) * p.Hq + h) * p.Lq_pad + i;
    const float l2 = __ldg(p.lse2 + vi);   // +inf past the sequence's last query, so P = 0 there
    const float di = __ldg(p.dvec + vi);
    int lim_key = k_len - 1;
    if constexpr (CAUSAL) lim_key = min(lim_key, i + off);
    BwdTracer tr;
    tr.init(p, part == 0 ? 5 : 6, lane == 0 && quarter == 0 && part < 2);
    if (n_tiles > 0) {
      // this row's Q and dO (a quarter of the features per column part) into
      // TMEM, packed two 16-bit values per column in memory order; rows past
      // the sequence's end are zero
      using T = typename BwdIO<BF16>::T;
      constexpr int kE = D / kBwdParts;   // features per warp
      constexpr int kW = kE / 8;          // uint4 words per warp's share of a row
      const size_t src = ((static_cast<size_t>(rq) + i) * p.Hq + h) * D + part * kE;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint4* g4 = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(which ? p.dout : p.q) + src);
        uint32_t w[4 * kW];
#pragma unroll
        for (int u = 0; u < kW; ++u) {
          const uint4 x = (i < q_len) ? __ldg(g4 + u) : make_uint4(0, 0, 0, 0);
          w[4 * u] = x.x;
          w[4 * u + 1] = x.y;
          w[4 * u + 2] = x.z;
          w[4 * u + 3] = x.w;
        }
        const uint32_t col = tmem + lane_off + (which ? C::kColDO : C::kColQ) + part * (kE / 2);
        if constexpr (kE / 2 == 32) {
          tmem_st_32x32b_x32(col, w);
        } else if constexpr (kE / 2 == 16) {
          tmem_st_32x32b_x16(col, w);
        } else {
          tmem_st_32x32b_x8(col, w);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_q_full);
    }
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      tr.rec(20, t);
      if (!mbar_wait_warp(b_s_full, t & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteSFull))) { ok = false; break; }
      tr.rec(21, t);
      tc_fence_after();
      // S is released as soon as it is in registers; P is formed after
      uint32_t sr[kBwdCols];
      tmem_ld_cols(t_s, sr);
      tmem_wait_ld(sr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_s_free);
      // masked: tiles crossing the causal diagonal and the ragged last key tile
      float pr[kBwdCols];
      if ((CAUSAL && t * kBN + kBN - 1 > m * kBM + off) || t * kBN + kBN > k_len)
        q_p_part<true>(sr, l2, lim_key - t * kBN - c0, cl2, pr);
      else
        q_p_part<false>(sr, l2, 0, cl2, pr);
      tr.rec(22, t);
      if (!mbar_wait_warp(b_dp_full, t & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteODone))) { ok = false; break; }
      tr.rec(23, t);
      tc_fence_after();
      ds_part<BF16>(t_dp, nullptr, di, pr);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_ds_full);
      tr.rec(24, t);
    }
    if (ok && (n_tiles == 0 || mbar_wait_warp(b_acc, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteODone)))) {
      tc_fence_after();
      using T = typename BwdIO<BF16>::T;
      constexpr int kHalf = D / kBwdParts;   // accumulator columns per warp
      T* dst = reinterpret_cast<T*>(p.dq) + ((static_cast<size_t>(rq) + i) * p.Hq + h) * D + part * kHalf;
      if (n_tiles == 0) {
        if (i < q_len) {
#pragma unroll
          for (int w = 0; w < kHalf / 8; ++w) reinterpret_cast<uint4*>(dst)[w] = make_uint4(0, 0, 0, 0);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kHalf / 16; ++c) {
          uint32_t x[16];
          tmem_ld_32x32b_x16(tmem + lane_off + 256 + part * kHalf + c * 16, x);
          tmem_wait_ld(x);
          if (i < q_len) store_row16<BF16>(dst + c * 16, x, p.scale);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kBwdWarpMMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace attn
