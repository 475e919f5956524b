// sm_103a attention forward: TMA-fed, tcgen05 tensor cores accumulating in
// TMEM, online softmax in registers, persistent over a schedule of work units.
//
// Method (page S23-J17, clxhxhhr.top/posts/5544, §3.1): per query row keep the
// running max m, the exp-sum l relative to m and the value accumulator u with
// the same weights; when m grows, r = exp(m_old - m_new) rescales l and u.
// The score tile S and probability tile P live only in TMEM and registers.
//
// CTA layout (320 threads, one CTA per SM):
//   warps 0-3  softmax warpgroup for query sub-tile 0 (rows 0..127 of the block)
//   warps 4-7  softmax warpgroup for query sub-tile 1 (rows 128..255)
//   warp 8     TMA producer: Q block once per unit, K and V tiles through one ring
//   warp 9     TMEM allocator and single-thread tcgen05.mma issuer
// TMEM (512 columns x 128 lanes, fp32): S_t at columns [128t, 128t+128); P_t
// (16-bit, two per column) overwrites the first 64 columns of S_t; the
// accumulator u_t (= O before normalisation) at [256+128t, 256+128t+D).
// Lane i of TMEM is query row i of a sub-tile, owned by one softmax thread.
//
// Rescaling of u is skipped while the running max grows by at most 2^8 in
// exp2 units (the exponentials then stay <= 256); the final O = u / l uses
// the same stale max in both numerator and denominator, so the result is
// unchanged.  This is the conditional rescale of the published
// FlashAttention-4 write-up; the pages' recurrence rescales on every change.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_params.h"
#include "ptx.cuh"

namespace attn {

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kChunks = D / 64;                  // 128-byte swizzle atoms per row
  static constexpr int kTile = kBM * D * 2;               // bytes of one 128-row tile
  // Ring of key/value stages.  Stage use i of a unit holds K tile
  // kv_begin + i and V tile kv_begin + i - 1 (the first use K only, the last
  // V only): the P.V of tile j and the S of tile j + 1 read one stage, which
  // is then released with a single commit.
  static constexpr int kNS = (D == 128) ? 2 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kNSub * kTile;
  static constexpr int kOffV = kOffK + kNS * kTile;
  static constexpr int kOffBar = kOffV + kNS * kTile;
  // barriers: q_full, q_empty, kv_full[NS], kv_empty[NS], s_full[2], p_full[2],
  //           o_done[2], drain, q_rot
  static constexpr int kNBars = 2 + 2 * kNS + 10;   // + q_rot (rotary variant), in-cluster merge ready / done
  static constexpr int kOffMisc = kOffBar + kNBars * 8;   // tmem slot, abort flag, bad flag
  static constexpr int kOffVarlen = kOffMisc + 64;        // varlen unit prefix table
  static constexpr int kSmemDense = kOffVarlen + 1024;    // + alignment slack
  static constexpr int kSmemVarlen = kOffVarlen + 4 * (kVarlenMaxB + 1) + 1024;
  // the sorting variant: the sequence of each rank after the prefix table
  static constexpr int kOffOrder = kOffVarlen + 4 * (kVarlenMaxB + 1);
  static constexpr int kSmemVarlenSorted = kOffOrder + 4 * kVarlenSortMax + 1024;
  static constexpr uint32_t kTmemCols = 512;
};

template <bool BF16>
struct IO;
template <>
struct IO<true> {
  using T = __nv_bfloat16;
  static constexpr bool bf16 = true;
};
template <>
struct IO<false> {
  using T = __half;
  static constexpr bool bf16 = false;
};

// One scheduled work unit, decoded identically by every role.
struct Unit {
  int b, h, g;
  int q_row0;            // first query row of the 256-row block (within the sequence)
  int q_len, k_len;      // sequence lengths
  int row_q, row_k;      // TMA row coordinate of the sequence start
  int bcoord;            // TMA batch coordinate
  int kv_begin, kv_end;  // 128-key tiles covered
  int split, n_split, slot;
  int kv_last[2];
};

// SORT (varlen, the sorting variant) with `sorted` set by its prefix pass:
// the sequences are numbered by rank, most keys first (the prefix table is
// over ranks; the sequence of rank i follows it, at vl_pref[kVarlenMaxB + 1 +
// i]), and `u`, the CTA's loop index, is permuted into snake order.
template <bool CAUSAL, bool VARLEN, bool SORT = false>
__device__ __forceinline__ bool decode_unit(const FwdParams& p, const int* vl_pref, int u, Unit& U,
                                            bool sorted = false) {
  if constexpr (!VARLEN) {
    const int* e = (p.n_inline ? p.units_inline : p.units) + u * kUnitInts;
    const int bh = e[0];
    U.b = bh / p.Hq;
    U.h = bh - U.b * p.Hq;
    U.q_row0 = e[1] * kBlockRows;
    U.kv_begin = e[2];
    U.kv_end = e[3];
    U.split = e[4];
    U.n_split = e[5];
    U.slot = e[6];
    U.q_len = p.Lq;
    U.k_len = p.Lk;
    U.row_q = 0;
    U.row_k = 0;
    U.bcoord = U.b;
  } else {
    if constexpr (SORT) {
      if (sorted) {
        // odd rounds of gridDim.x units reversed (a last, partial round
        // keeps its order, so every unit is still visited once): the CTA
        // that takes a long unit in one round takes a short one in the next
        const int G = gridDim.x, r = u / G;
        if ((r & 1) && (r + 1) * G <= vl_pref[p.B]) u = r * G + (G - 1) - (u - r * G);
      }
    }
    // binary search: largest b with vl_pref[b] <= u
    int lo = 0, hi = p.B;   // vl_pref[0] = 0 <= u < vl_pref[B]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (vl_pref[mid] <= u) lo = mid; else hi = mid;
    }
    U.b = lo;
    // units of a sequence: (query block, head group) with the group fastest;
    // a group is one head, or the 2^pack_log2 heads sharing a key/value head
    const int lp = p.pack_log2;
    const int n_hu = p.Hq >> lp;
    const int local = u - vl_pref[lo];
    if constexpr (SORT) {
      if (sorted) {
        lo = vl_pref[kVarlenMaxB + 1 + lo];
        U.b = lo;
      }
    }
    const int s0k = __ldg(p.cu_seqlens_k + lo);
    U.k_len = __ldg(p.cu_seqlens_k + lo + 1) - s0k;
    U.row_k = s0k;
    U.bcoord = 0;
    U.kv_begin = 0;
    U.kv_end = 0;
    if (p.vl_decode) {
      // one query, row lo of q; units (key piece, head group), the group
      // fastest (CTAs side by side read the same keys of neighbouring heads)
      const int pcs = decode_pieces(U.k_len, p.vl_split);
      const int piece = local / n_hu;
      const int hg = local - piece * n_hu;
      U.h = hg << lp;
      U.q_row0 = 0;
      U.q_len = 1;
      U.row_q = lo;
      U.split = piece;
      U.n_split = pcs;
      U.slot = (pcs > 1) ? u : -1;
    } else {
      const int mb = local / n_hu;
      U.h = (local - mb * n_hu) << lp;   // first query head of the unit
      U.q_row0 = mb * (kBlockRows >> lp);
      const int s0 = __ldg(p.cu_seqlens + lo);
      U.q_len = __ldg(p.cu_seqlens + lo + 1) - s0;
      U.row_q = s0;
      U.split = 0;
      U.n_split = 1;
      U.slot = -1;
    }
  }
  U.g = U.h / p.group;
  const int span = VARLEN ? (kBM >> p.pack_log2) : kBM;   // queries per sub-tile
  U.kv_last[0] = kv_last_tile(U.q_row0, 0, U.q_len, U.k_len, CAUSAL, span);
  U.kv_last[1] = kv_last_tile(U.q_row0, 1, U.q_len, U.k_len, CAUSAL, span);
  const int end = max(U.kv_last[0], U.kv_last[1]) + 1;
  if constexpr (VARLEN) {
    U.kv_end = end;
    if (U.n_split > 1) {   // a decode piece: its own range of key tiles
      U.kv_begin = U.split * p.vl_split;
      U.kv_end = min(end, U.kv_begin + p.vl_split);
    }
  } else {
    U.kv_end = min(U.kv_end, end);
  }
  return true;
}

__device__ __forceinline__ bool unit_active(const Unit& U, int t, int j) { return j <= U.kv_last[t]; }

// Phase trace: one writer thread per stream; events beyond the capacity are
// dropped.  Compiled in only when ATTN_TRACE is 1 (the library's traced
// build); otherwise every call below compiles to nothing.
#ifndef ATTN_TRACE
#define ATTN_TRACE 0
#endif
struct Tracer {
  unsigned long long* base;   // this CTA's region of this stream, or null
  int cap, n;
  __device__ __forceinline__ void init(const FwdParams& p, int stream) {
    base = (ATTN_TRACE && p.trace)
               ? p.trace + (static_cast<size_t>(blockIdx.x) * kTrStreams + stream) * p.trace_cap * 2
               : nullptr;
    cap = p.trace_cap;
    n = 0;
  }
  __device__ __forceinline__ void off() { base = nullptr; }
  __device__ __forceinline__ void rec(int tag, int t, int a, int b) {
    if (ATTN_TRACE && base != nullptr && n < cap) {
      base[2 * n] = (static_cast<unsigned long long>(tag) << 56) |
                    (static_cast<unsigned long long>(t & 0xff) << 48) |
                    (static_cast<unsigned long long>(a & 0xffffff) << 24) |
                    static_cast<unsigned long long>(b & 0xffffff);
      base[2 * n + 1] = (tag >= kTagGEnter) ? global_timer_ns() : clock64();
      ++n;
    }
  }
};

// ---------------------------------------------------------------------------
// softmax of one S tile for the calling thread's row
// ---------------------------------------------------------------------------
struct RowState {
  float m;     // running max in scaled exp2 units (scale * log2(e) * max score); -inf if none
  float l;     // exp-sum relative to m
};

// Loads S (128 fp32) of this thread's row, masks keys beyond `lim` when
// MASK, updates (m, l), writes P to TMEM and, when the max moved by more than
// 2^8, rescales u in TMEM.  The previous tile's P.V has completed by then
// (the commit that signalled this S was issued after it), and this tile's P.V
// is issued only after this thread arrives.
template <bool MASK, bool BF16, int D>
__device__ __forceinline__ void softmax_tile(uint32_t t_s, uint32_t t_o, int lim, float c_log2, RowState& st,
                                             bool first) {
  // S in two halves: the second half loads while the first half's max is
  // taken.  Row max over eight chains of three-input max.
  float s[128];
  float mx[8];
  {
    uint32_t r0[64];
    tmem_ld_32x32b_x64(t_s + 0, r0);
    tmem_wait_ld(r0);
#pragma unroll
    for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(r0[i]);
  }
  {
    uint32_t r2[64];
    tmem_ld_32x32b_x64(t_s + 64, r2);
    if constexpr (MASK) {
#pragma unroll
      for (int i = 0; i < 64; ++i) s[i] = (i <= lim) ? s[i] : -INFINITY;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = fmaxf(s[k], s[k + 8]);
#pragma unroll
    for (int i = 16; i < 64; i += 16)
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], s[i + k], s[i + 8 + k]);
    tmem_wait_ld(r2);
#pragma unroll
    for (int i = 0; i < 64; ++i) s[64 + i] = __uint_as_float(r2[i]);
  }
  if constexpr (MASK) {
#pragma unroll
    for (int i = 64; i < 128; ++i) s[i] = (i <= lim) ? s[i] : -INFINITY;
  }
#pragma unroll
  for (int i = 64; i < 128; i += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], s[i + k], s[i + 8 + k]);
  const float mx_all = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
  const float m_tile = (mx_all == -INFINITY) ? -INFINITY : mx_all * c_log2;
  const float m_old = st.m;
  bool resc = false;
  if (m_tile > m_old && (first || m_old == -INFINITY || m_tile - m_old > 8.0f)) {
    resc = true;
    st.m = m_tile;
  }
  const float moff = (st.m == -INFINITY) ? 0.0f : st.m;
  // p = exp2(s * c - m): the argument with packed fp32x2 FMA, one ex2 per
  // element, row sums with packed adds; P packed to 16-bit pairs and stored
  // 32 columns at a time
  const float2 c2 = make_float2(c_log2, c_log2);
  const float2 nm2 = make_float2(-moff, -moff);
  float2 sum_a = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const int c0 = q * 32 + 2 * i;
      const float2 x0 = ffma2(make_float2(s[c0], s[c0 + 1]), c2, nm2);
      const float2 x1 = ffma2(make_float2(s[c0 + 2], s[c0 + 3]), c2, nm2);
      float2 e0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
      float2 e1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
      if constexpr (MASK) {
        e0.x = (c0 <= lim) ? e0.x : 0.0f;
        e0.y = (c0 + 1 <= lim) ? e0.y : 0.0f;
        e1.x = (c0 + 2 <= lim) ? e1.x : 0.0f;
        e1.y = (c0 + 3 <= lim) ? e1.y : 0.0f;
      }
      sum_a = fadd2(sum_a, e0);
      sum_b = fadd2(sum_b, e1);
      pk[i] = pack2<BF16>(e0.x, e0.y);
      pk[i + 1] = pack2<BF16>(e1.x, e1.y);
    }
    tmem_st_32x32b_x16(t_s + q * 16, pk);
  }
  // rescale l and, when anything is accumulated, u
  const float r = resc ? ((m_old == -INFINITY) ? 0.0f : ex2_approx(m_old - st.m)) : 1.0f;
  const float2 sum2 = fadd2(sum_a, sum_b);
  st.l = st.l * r + (sum2.x + sum2.y);
  if (!first && __any_sync(0xffffffffu, resc)) {
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      uint32_t o[16];
      tmem_ld_32x32b_x16(t_o + c * 16, o);
      tmem_wait_ld(o);
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * r);
      tmem_st_32x32b_x16(t_o + c * 16, o);
    }
  }
  tmem_wait_st();
}

// Rotary embedding of one 128-byte-swizzled Q row in shared memory (row
// `row` of a 128-row sub-tile starting at `tile`, D/64 chunks of 64 columns,
// 16 KB apart): pair (x1, x2) -> (x1 cos a - x2 sin a, x1 sin a + x2 cos a)
// with (cos a, sin a) = p.rope_cs[pos * rot / 2 + i], computed and rounded
// as the standalone rotary pass does; 8 pairs per step with 16-byte accesses.
template <int D, bool BF16>
__device__ __forceinline__ void rope_row(uint8_t* tile, int row, const FwdParams& p, int pos) {
  const int half = p.rope_rot >> 1;
  const float2* cs = reinterpret_cast<const float2*>(p.rope_cs) + static_cast<size_t>(pos) * half;
  auto at = [&](int col) -> uint4* {   // the 16-byte granule holding columns col .. col + 7
    return reinterpret_cast<uint4*>(tile + (col >> 6) * 16384 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4));
  };
  auto unpack = [](uint32_t w, float& lo, float& hi) {
    if constexpr (BF16) {
      lo = __uint_as_float(w << 16);
      hi = __uint_as_float(w & 0xffff0000u);
    } else {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
      lo = f.x;
      hi = f.y;
    }
  };
  for (int g = 0; g < half; g += 8) {
    float c[8], s[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float2 v = __ldg(cs + g + e);
      c[e] = v.x;
      s[e] = v.y;
    }
    if (p.rope_gptj) {
      // pairs (2i, 2i+1): columns 2g .. 2g + 15 in two granules
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint4* gp = at(2 * g + 8 * k);
        uint4 w = *gp;
        uint32_t* ww = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x1, x2;
          unpack(ww[e], x1, x2);
          const int i = 4 * k + e;
          ww[e] = pack2<BF16>(x1 * c[i] - x2 * s[i], x1 * s[i] + x2 * c[i]);
        }
        *gp = w;
      }
    } else {
      // pairs (i, i + rot/2): columns g .. g + 7 and g + half .. g + half + 7
      uint4* ga = at(g);
      uint4* gb = at(g + half);
      uint4 wa = *ga, wb = *gb;
      uint32_t* a = reinterpret_cast<uint32_t*>(&wa);
      uint32_t* b = reinterpret_cast<uint32_t*>(&wb);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a0, a1, b0, b1;
        unpack(a[e], a0, a1);
        unpack(b[e], b0, b1);
        const int i = 2 * e;
        a[e] = pack2<BF16>(a0 * c[i] - b0 * s[i], a1 * c[i + 1] - b1 * s[i + 1]);
        b[e] = pack2<BF16>(a0 * s[i] + b0 * c[i], a1 * s[i + 1] + b1 * c[i + 1]);
      }
      *ga = wa;
      *gb = wb;
    }
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// The sorting variant's prefix pass (packed varlen forwards with their own
// key offsets: cross-attention, a key/value cache), by one warp: validates
// cu_seqlens (queries) and cu_seqlens_k (keys), writes the prefix table of
// units per sequence (vl_pref[0..B]) and sets *bad_flag on malformed offsets,
// as the kernel's own pass does; and sets *sort_flag when it numbers the
// sequences by rank instead.
// ---------------------------------------------------------------------------
static __device__ __noinline__ void varlen_prefix_pass_sorted(const FwdParams& p, int* vl_pref, volatile int* bad_flag,
                                                       volatile int* sort_flag) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  bool bad = false;
  if (lane == 0 && ((!p.vl_decode && __ldg(p.cu_seqlens) != 0) || __ldg(p.cu_seqlens_k) != 0)) bad = true;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    int cnt = 0;
    int key = -1;   // sort key: the sequence's key count
    if (b < p.B) {
      const int ak = __ldg(p.cu_seqlens_k + b), ek = __ldg(p.cu_seqlens_k + b + 1);
      if (ek < ak || ek > p.Lk) bad = true;
      key = max(ek - ak, 0);
      if (p.vl_decode) {
        // every head group of every sequence, in pieces of its keys
        cnt = (p.Hq >> p.pack_log2) * decode_pieces(max(ek - ak, 0), p.vl_split);
      } else {
        const int a = __ldg(p.cu_seqlens + b), e = __ldg(p.cu_seqlens + b + 1);
        if (e < a || e > p.Lq) bad = true;
        const int len = e - a;
        const int blk = kBlockRows >> p.pack_log2;   // queries per unit
        cnt = (len > 0) ? ((len + blk - 1) / blk) * (p.Hq >> p.pack_log2) : 0;
      }
    }
    // At most kVarlenSortMax sequences (one pass; not decoding steps) whose
    // key counts (over the sequences with queries) differ by more than 4x:
    // number the sequences by rank, most keys first, and place the units in
    // snake order (decode_unit), so a CTA that takes a long unit in one
    // round takes a short one in the next.
    bool sort = false;
    if (!p.vl_decode && p.B <= kVarlenSortMax) {
      int kmax = (cnt > 0) ? key : 0, kmin = (cnt > 0) ? key : 0x7fffffff;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
        kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      }
      sort = kmin != 0x7fffffff && static_cast<long long>(kmax) > 4LL * kmin;
      if (lane == 0) *sort_flag = sort ? 1 : 0;
    }
    if (sort) {
      // rank of this sequence: more keys first, then the lower index
      int rank = 0;
#pragma unroll 8
      for (int j = 0; j < 32; ++j) {
        const int kj = __shfl_sync(0xffffffffu, key, j);
        rank += (kj > key || (kj == key && j < lane)) ? 1 : 0;
      }
      int* order = vl_pref + kVarlenMaxB + 1;
      if (b < p.B) {
        order[rank] = b;
        vl_pref[rank + 1] = cnt;   // scratch: unit count by rank
      }
      __syncwarp();
      cnt = (lane < p.B) ? vl_pref[lane + 1] : 0;
      __syncwarp();
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (b < p.B) vl_pref[b + 1] = carry + x;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  if (lane == 0) vl_pref[0] = 0;
  if (__any_sync(0xffffffffu, bad) && lane == 0) {
    *bad_flag = 1;
    atomicCAS(p.err, 0, ATTN_DEVERR_BAD_SEQLENS);
  }
}

// ---------------------------------------------------------------------------
template <int D, bool BF16, bool CAUSAL, bool VARLEN, bool ROPE = false, bool SORT = false>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  static_assert(!(ROPE && VARLEN), "the rotary variant is dense only");
  static_assert(!SORT || VARLEN, "the sorting variant is varlen only");
  using C = Cfg<D>;
  using T = typename IO<BF16>::T;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sK = sbase + C::kOffK;
  const uint32_t sV = sbase + C::kOffV;
  const uint32_t bar0 = sbase + C::kOffBar;
  const uint32_t b_q_full = bar0;
  const uint32_t b_q_empty = bar0 + 8;
  auto b_kv_full = [&](int s) { return bar0 + 16 + 8 * s; };
  auto b_kv_empty = [&](int s) { return bar0 + 16 + 8 * (C::kNS + s); };
  const uint32_t bar_sp = bar0 + 16 + 16 * C::kNS;
  auto b_s_full = [&](int t) { return bar_sp + 8 * t; };
  auto b_p_full = [&](int t) { return bar_sp + 16 + 8 * t; };
  auto b_o_done = [&](int t) { return bar_sp + 32 + 8 * t; };
  const uint32_t b_drain = bar_sp + 48;
  const uint32_t b_q_rot = bar_sp + 56;   // rotary variant: the unit's Q rotated in place
  // in-cluster merge: every softmax warp of every CTA of the cluster has
  // staged its rows (ready) / has finished reading the peers (done)
  const uint32_t b_cready = bar_sp + 64;
  const uint32_t b_cdone = bar_sp + 72;

  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  volatile int* bad_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
  volatile int* sort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 12);   // SORT
  int* vl_pref = reinterpret_cast<int*>(smem + C::kOffVarlen);

  WaitCtl wc{p.err, abort_flag, p.timeout_ns};

  if (tid == 0) {
    *abort_flag = 0;
    *bad_flag = 0;
    if constexpr (SORT) *sort_flag = 0;
  }
  // The producer thread initialises the barriers, so that (dense schedules)
  // it can issue the first unit's Q block and first key tile before the
  // set-up barrier: the first loads after an L2 flush take microseconds, and
  // they then overlap the TMEM allocation and the set-up.
  bool early = false;
  if (warp == kWarpTMA && lane == 0) {
    mbar_init(b_q_full, 1);
    mbar_init(b_q_empty, 1);
    for (int s = 0; s < C::kNS; ++s) {
      mbar_init(b_kv_full(s), 1);
      mbar_init(b_kv_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(b_s_full(t), 1);
      mbar_init(b_p_full(t), kBM / 32);   // one arrival per softmax warp
      mbar_init(b_o_done(t), 1);
    }
    mbar_init(b_drain, 1);
    mbar_init(b_q_rot, 2 * kBM / 32);   // one arrival per softmax warp
    mbar_init(b_cready, (2 * kBM / 32) * max(p.cluster_merge, 1));
    mbar_init(b_cdone, (2 * kBM / 32) * max(p.cluster_merge, 1));
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    if constexpr (!VARLEN) {
      const int* off = p.n_inline ? p.cta_off_inline : p.cta_off;
      if (off[blockIdx.x] < off[blockIdx.x + 1]) {
        Unit U;
        decode_unit<CAUSAL, VARLEN>(p, nullptr, off[blockIdx.x], U);
        if (U.kv_end > U.kv_begin) {
          // the producer loop below skips exactly these two issues
          mbar_arrive_expect_tx(b_q_full, kNSub * C::kTile);
#pragma unroll
          for (int t = 0; t < kNSub; ++t)
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_4d(sQ + t * C::kTile + c * 16384, &p.tm_q, b_q_full, c * 64, U.h, U.row_q + U.q_row0 + t * kBM,
                          U.bcoord);
          mbar_arrive_expect_tx(b_kv_full(0), C::kTile);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(sK + c * 16384, &p.tm_k, b_kv_full(0), c * 64, U.g, U.row_k + U.kv_begin * kBN, U.bcoord);
          early = true;
        }
      }
    }
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }

  // varlen: validate cu_seqlens (queries) and cu_seqlens_k (keys) and build
  // the prefix table of units per sequence
  int n_units = 0, u_first = 0, u_step = 1;
  if constexpr (SORT) {
    if (warp == 0) varlen_prefix_pass_sorted(p, vl_pref, bad_flag, sort_flag);
  } else if constexpr (VARLEN) {
    if (warp == 0) {
      int carry = 0;
      bool bad = false;
      if (lane == 0 && ((!p.vl_decode && __ldg(p.cu_seqlens) != 0) || __ldg(p.cu_seqlens_k) != 0)) bad = true;
      for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int cnt = 0;
        if (b < p.B) {
          const int ak = __ldg(p.cu_seqlens_k + b), ek = __ldg(p.cu_seqlens_k + b + 1);
          if (ek < ak || ek > p.Lk) bad = true;
          if (p.vl_decode) {
            // every head group of every sequence, in pieces of its keys
            cnt = (p.Hq >> p.pack_log2) * decode_pieces(max(ek - ak, 0), p.vl_split);
          } else {
            const int a = __ldg(p.cu_seqlens + b), e = __ldg(p.cu_seqlens + b + 1);
            if (e < a || e > p.Lq) bad = true;
            const int len = e - a;
            const int blk = kBlockRows >> p.pack_log2;   // queries per unit
            cnt = (len > 0) ? ((len + blk - 1) / blk) * (p.Hq >> p.pack_log2) : 0;
          }
        }
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (b < p.B) vl_pref[b + 1] = carry + x;
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
      if (lane == 0) vl_pref[0] = 0;
      if (__any_sync(0xffffffffu, bad) && lane == 0) {
        *bad_flag = 1;
        atomicCAS(p.err, 0, ATTN_DEVERR_BAD_SEQLENS);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // in-cluster merge: the peers' barriers are initialised before any remote
  // arrival (CTAs of a cluster are co-scheduled, so this wait ends)
  if (!VARLEN && p.cluster_merge > 0) cluster_sync();
  const uint32_t tmem = *tmem_slot;
  // the combine pass of split pieces may be scheduled now; it waits for this grid
  grid_launch_dependents();

  if constexpr (VARLEN) {
    n_units = (*bad_flag) ? 0 : vl_pref[p.B];
    u_first = blockIdx.x;
    u_step = gridDim.x;
    if (p.vl_decode) {
      // the decode combine reads the unit prefix and the malformed flag
      if (p.vl_pref_out != nullptr && blockIdx.x == 0) {
        for (int i = tid; i <= p.B; i += kThreads) p.vl_pref_out[i] = vl_pref[i];
        if (tid == 0) p.vl_pref_out[p.B + 1] = *bad_flag;
      }
      // malformed key offsets: every row O = 0, lse = -inf
      if (*bad_flag) {
        T* out = reinterpret_cast<T*>(p.o);
        for (long long r = static_cast<long long>(blockIdx.x) * kThreads + tid; r < static_cast<long long>(p.B) * p.Hq;
             r += static_cast<long long>(gridDim.x) * kThreads) {
          uint4* d4 = reinterpret_cast<uint4*>(out + r * D);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) d4[i] = make_uint4(0, 0, 0, 0);
          const long long b = r / p.Hq, h = r - b * p.Hq;
          p.lse[h * p.B + b] = -INFINITY;
        }
      }
    }
  } else {
    const int* off = p.n_inline ? p.cta_off_inline : p.cta_off;
    u_first = off[blockIdx.x];
    n_units = off[blockIdx.x + 1];
    u_step = 1;
  }
  bool snake = false;   // the sorting variant's units in rank and snake order
  if constexpr (SORT) snake = *sort_flag != 0;

  if (warp == kWarpTMA) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      Tracer tr;
      tr.init(p, kTrProducer);
      uint32_t q_cnt = 0, kv_cnt = 0;
      for (int u = u_first; u < n_units; u += u_step) {
        Unit U;
        decode_unit<CAUSAL, VARLEN, SORT>(p, vl_pref, u, U, snake);
        if (U.kv_end <= U.kv_begin) continue;
        const bool pre = early;   // this unit's Q and first key tile were issued before the set-up barrier
        early = false;
        if (!pre && !mbar_wait(b_q_empty, (q_cnt & 1) ^ 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteQEmpty))) break;
        if (!pre) mbar_arrive_expect_tx(b_q_full, kNSub * C::kTile);
        // a sub-tile is 128 rows of one head, or (packed) 128 / 2^pack_log2
        // queries x 2^pack_log2 heads from one box of the same byte count
        const int q_span = VARLEN ? (kBM >> p.pack_log2) : kBM;
        if (!pre) {
#pragma unroll
          for (int t = 0; t < kNSub; ++t)
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_4d(sQ + t * C::kTile + c * 16384, &p.tm_q, b_q_full, c * 64, U.h,
                          U.row_q + U.q_row0 + t * q_span, U.bcoord);
        }
        tr.rec(kTagQIssue, 0, u, 0);
        ++q_cnt;
        bool ok = true;
        const int n = U.kv_end - U.kv_begin;
        for (int i = 0; i <= n; ++i) {
          const int st = kv_cnt % C::kNS;
          if (pre && i == 0) {   // stage 0 holds the first key tile already
            ++kv_cnt;
            continue;
          }
          if (!mbar_wait(b_kv_empty(st), ((kv_cnt / C::kNS) & 1) ^ 1, wc,
                         ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKEmpty))) { ok = false; break; }
          const bool hk = i < n, hv = i > 0;
          mbar_arrive_expect_tx(b_kv_full(st), (hk && hv ? 2 : 1) * C::kTile);
          if (hk) {
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_4d(sK + st * C::kTile + c * 16384, &p.tm_k, b_kv_full(st), c * 64, U.g,
                          U.row_k + (U.kv_begin + i) * kBN, U.bcoord);
            tr.rec(kTagKIssue, 0, u, U.kv_begin + i);
          }
          if (hv) {
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_4d(sV + st * C::kTile + c * 16384, &p.tm_v, b_kv_full(st), c * 64, U.g,
                          U.row_k + (U.kv_begin + i - 1) * kBN, U.bcoord);
            tr.rec(kTagVIssue, 0, u, U.kv_begin + i - 1);
          }
          ++kv_cnt;
        }
        if (!ok) break;
      }
      // On an abort, let loads already issued land before the CTA exits.
      if (*abort_flag) {
        for (int s = 0; s < C::kNS; ++s) {
          const uint32_t n = (kv_cnt + C::kNS - 1 - s) / C::kNS;   // fills issued into stage s
          if (n > 0) mbar_wait(b_kv_full(s), (n - 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
        }
      }
    }
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescO = idesc_f16_f32acc(kBM, D, BF16, true);
      constexpr uint32_t kIdescS = idesc_f16_f32acc(kBM, kBN, BF16, false);
      // descriptor bases (start address field is addr >> 4 in the low bits)
      const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sV, 16384, 1024);
      Tracer tr;
      tr.init(p, kTrMMA);
      tr.rec(kTagStart, 0, 0, 0);
      uint32_t q_cnt = 0, kv_cnt = 0;
      uint32_t p_cnt0 = 0, p_cnt1 = 0;
      auto issue_s = [&](int t, int st) {
        const uint64_t a0 = dq0 + ((t * C::kTile) >> 4);
        const uint64_t b0 = dk0 + ((st * C::kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_ss(tmem + t * 128, a0 + off, b0 + off, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(b_s_full(t));
      };
      bool ok = true;
      for (int u = u_first; u < n_units && ok; u += u_step) {
        Unit U;
        decode_unit<CAUSAL, VARLEN, SORT>(p, vl_pref, u, U, snake);
        if (U.kv_end <= U.kv_begin) continue;
        // (rotary variant: the softmax threads have rotated the Q block in place)
        if (!mbar_wait(ROPE ? b_q_rot : b_q_full, q_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteQFull))) break;
        tr.rec(kTagQFull, 0, u, 0);
        bool first_pv0 = true, first_pv1 = true;
        // first stage use: K of the first tile, S for it
        {
          const int st = kv_cnt % C::kNS;
          if (!mbar_wait(b_kv_full(st), (kv_cnt / C::kNS) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKFull))) break;
          tr.rec(kTagKFull, 0, u, U.kv_begin);
          for (int t = 0; t < kNSub; ++t)
            if (unit_active(U, t, U.kv_begin)) {
              issue_s(t, st);
              tr.rec(kTagSIssue, t, u, U.kv_begin);
            }
          umma_commit(b_kv_empty(st));
          ++kv_cnt;
        }
        // Per tile j: O_t += P_t(j) V(j), then S_t(j+1) = Q_t K(j+1)^T, for
        // t = 0, 1.  The S of a sub-tile is issued after its P.V, so the
        // commit that signals S_t(j+1) also covers P_t(j) V(j): the softmax
        // of tile j+1 may read and rescale u_t.  o_done is committed once per
        // unit and sub-tile, after its last P.V, for the epilogue.
        for (int j = U.kv_begin; j < U.kv_end; ++j) {
          const int st = kv_cnt % C::kNS;
          tr.rec(kTagVWait, 0, u, j);
          if (!mbar_wait(b_kv_full(st), (kv_cnt / C::kNS) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteVFull))) {
            ok = false;
            break;
          }
          tr.rec(kTagVFull, 0, u, j);
          const bool have_next = j + 1 < U.kv_end;
#pragma unroll
          for (int t = 0; t < kNSub; ++t) {
            uint32_t& p_cnt = (t == 0) ? p_cnt0 : p_cnt1;
            bool& first_pv = (t == 0) ? first_pv0 : first_pv1;
            const bool next_s = have_next && unit_active(U, t, j + 1);
            if (unit_active(U, t, j)) {
              tr.rec(kTagPWait, t, u, j);
              if (!mbar_wait(b_p_full(t), p_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSitePFull))) {
                ok = false;
                break;
              }
              ++p_cnt;
              // P was written into TMEM by the softmax threads (tcgen05.st):
              // this fence orders that before the MMA that reads it.
              tc_fence_after();
              tr.rec(kTagPFull, t, u, j);
              const uint64_t bv = dv0 + ((st * C::kTile) >> 4);
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                umma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, bv + ((kk * 2048) >> 4), kIdescO,
                        (first_pv && kk == 0) ? 0u : 1u);
              if (!next_s) umma_commit(b_o_done(t));
              tr.rec(kTagPVIssue, t, u, j);
              first_pv = false;
            }
            if (next_s) {
              issue_s(t, st);
              tr.rec(kTagSIssue, t, u, j + 1);
            }
          }
          if (!ok) break;
          umma_commit(b_kv_empty(st));
          ++kv_cnt;
        }
        if (!ok) break;
        umma_commit(b_q_empty);
        tr.rec(kTagUnitEnd, 0, u, 0);
        ++q_cnt;
      }
      // every MMA issued by this thread has completed once the drain barrier fires
      umma_commit(b_drain);
      mbar_wait(b_drain, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;                 // query sub-tile
    const int quarter = warp & 3;            // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;     // row within the sub-tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + t * 128;
    const uint32_t t_o = tmem + lane_off + 256 + t * 128;
    const float c_log2 = p.scale_log2;
    uint32_t s_cnt = 0, o_cnt = 0;   // s_full phases seen; units with an o_done commit
    uint32_t qr_cnt = 0;             // rotary variant: q_full phases seen
    T* out = reinterpret_cast<T*>(p.o);
    Tracer tr;
    tr.init(p, t == 0 ? kTrSoftmax0 : kTrSoftmax1);
    if (row != 0) tr.off();
    tr.rec(kTagGEnter, t, 0, 0);
    // packed heads (varlen): TMEM lane `row` is query row >> lp of the
    // sub-tile, head row & (2^lp - 1) of the unit's group
    const int lp = VARLEN ? p.pack_log2 : 0;
    const int span = kBM >> lp;
    for (int u = u_first; u < n_units; u += u_step) {
      Unit U;
      decode_unit<CAUSAL, VARLEN, SORT>(p, vl_pref, u, U, snake);
      const int q_first = U.q_row0 + t * span;          // first query of the sub-tile
      const int qrow = q_first + (row >> lp);           // query row within the sequence
      const int head = U.h + (row & ((1 << lp) - 1));
      const bool row_valid = qrow < U.q_len;
      // allowed keys of this row: key <= lim_key
      int lim_key = U.k_len - 1;
      if constexpr (CAUSAL) lim_key = min(lim_key, qrow + (U.k_len - U.q_len));
      RowState st{-INFINITY, 0.0f};
      int n_act = 0;
      bool ok = true;
      if constexpr (ROPE) {
        // rotary embedding of this thread's Q row, in shared memory, before
        // the unit's first S = Q K^T (the MMA issuer waits for q_rot)
        if (U.kv_end > U.kv_begin) {
          if (!mbar_wait_warp(b_q_full, qr_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteQFull))) break;
          ++qr_cnt;
          rope_row<D, BF16>(smem + C::kOffQ + t * C::kTile, row, p, min(q_first + row, p.Lq - 1) + p.rope_qoff);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_q_rot);
        }
      }
      tr.rec(kTagUnitBegin, t, u, 0);
      for (int j = U.kv_begin; j < U.kv_end; ++j) {
        if (!unit_active(U, t, j)) break;
        if (!mbar_wait_warp(b_s_full(t), s_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteSFull))) { ok = false; break; }
        ++s_cnt;
        tc_fence_after();
        tr.rec(kTagSFull, t, u, j);
        const int lim = lim_key - j * kBN;
        const bool mask_tile = (j * kBN + kBN - 1 > U.k_len - 1) ||
                               (CAUSAL && j * kBN + kBN - 1 > q_first + (U.k_len - U.q_len));
        if (mask_tile)
          softmax_tile<true, BF16, D>(t_s, t_o, lim, c_log2, st, n_act == 0);
        else
          softmax_tile<false, BF16, D>(t_s, t_o, lim, c_log2, st, n_act == 0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_p_full(t));
        tr.rec(kTagPArrive, t, u, j);
        ++n_act;
      }
      if (!ok) break;
      const bool split = U.n_split > 1;
      if (n_act > 0) {
        if (!mbar_wait_warp(b_o_done(t), o_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteODone))) break;
        ++o_cnt;
        tc_fence_after();
        tr.rec(kTagODone, t, u, 0);
      }
      if (!split) {
        // O = u / l, lse = m / log2(e) + ln l
        const float inv_l = (st.l > 0.0f) ? 1.0f / st.l : 0.0f;
        const size_t orow = VARLEN ? static_cast<size_t>(U.row_q + qrow)
                                   : static_cast<size_t>(U.b) * p.Lq + qrow;
        T* dst = out + (orow * p.Hq + head) * D;
        if (n_act > 0 && D == 64) {
          // The 128-byte rows are transposed within groups of 8 lanes by
          // three xor-shuffle stages: afterwards lane 8g + j holds 16-byte
          // chunk j of rows 8g .. 8g + 7, so one warp store writes 4 whole
          // rows, where a store of each thread's own row would write a
          // 16-byte piece of 32 rows (32 cache lines).  (For head_dim 128 the
          // shuffles cost more than they save: measured slower.)
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint4 a[8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(t_o + c * 64 + h * 32, o);
              tmem_wait_ld(o);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                a[4 * h + i] = make_uint4(
                    pack2<BF16>(__uint_as_float(o[8 * i + 0]) * inv_l, __uint_as_float(o[8 * i + 1]) * inv_l),
                    pack2<BF16>(__uint_as_float(o[8 * i + 2]) * inv_l, __uint_as_float(o[8 * i + 3]) * inv_l),
                    pack2<BF16>(__uint_as_float(o[8 * i + 4]) * inv_l, __uint_as_float(o[8 * i + 5]) * inv_l),
                    pack2<BF16>(__uint_as_float(o[8 * i + 6]) * inv_l, __uint_as_float(o[8 * i + 7]) * inv_l));
            }
#pragma unroll
            for (int m = 4; m >= 1; m >>= 1) {
              const bool up = (lane & m) != 0;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (k & m) continue;
                const uint4 snd = up ? a[k] : a[k | m];
                uint4 rcv;
                rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, m);
                rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, m);
                rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, m);
                rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, m);
                if (up) a[k] = rcv; else a[k | m] = rcv;
              }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = quarter * 32 + (lane & ~7) + i;   // row of the sub-tile
              const int qr = q_first + (rr >> lp);
              if (qr < U.q_len) {
                const int hd = U.h + (rr & ((1 << lp) - 1));
                const size_t orr = VARLEN ? static_cast<size_t>(U.row_q + qr) : static_cast<size_t>(U.b) * p.Lq + qr;
                *reinterpret_cast<uint4*>(out + (orr * p.Hq + hd) * D + c * 64 + (lane & 7) * 8) = a[i];
              }
            }
          }
        } else if (n_act > 0) {
          // each thread its own row, in 32-byte stores where the output is
          // 32-byte aligned (half the store instructions of 16-byte ones)
          const bool v8 = (reinterpret_cast<uintptr_t>(p.o) & 31) == 0;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(t_o + c * 32, o);
            tmem_wait_ld(o);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
            if (row_valid && v8) {
              st_global_v8(dst + c * 32, pk);
              st_global_v8(dst + c * 32 + 16, pk + 8);
            } else if (row_valid) {
              uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
        } else if (row_valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) d4[i] = make_uint4(0, 0, 0, 0);
        }
        if (row_valid) {
          const float lse = (st.l > 0.0f) ? st.m * 0.69314718055994531f + __logf(st.l) : -INFINITY;
          const size_t li = VARLEN ? static_cast<size_t>(head) * p.Lq + U.row_q + qrow
                                   : (static_cast<size_t>(U.b) * p.Hq + head) * p.Lq + qrow;
          p.lse[li] = lse;
        }
      } else {
        // split-KV piece: store its own normalised output O_s = u_s / l_s and
        // (m, l) in fp32; the combine pass forms the convex mix
        // sum_s w_s O_s / sum_s w_s.  fp32 keeps the range and precision of
        // the accumulator (a 16-bit copy would overflow or go subnormal on
        // large- or small-magnitude values that the unsplit path handles).
        // Layout [slot][t][D/4][row][4]: a warp's 32 rows of one 4-column
        // group are 512 contiguous bytes.
        if (!VARLEN && p.cluster_merge > 0) {
          // in-cluster merge: O_s and (m, l) of this row stay in this CTA's
          // shared memory, over the unit's K/V ring and Q block; layout
          // [t][D/4][row][4].  They are free once the unit's last MMA has
          // completed (the q_empty commit; one unit per CTA, so the loads
          // are all consumed too) - the other sub-tile's MMAs may still be
          // reading them when this sub-tile's o_done arrives.
          const bool idle = (U.kv_end <= U.kv_begin) ||   // an empty piece issued nothing
                            mbar_wait_warp(b_q_empty, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteMerge));
          tc_fence_after();
          if (idle) {
            float4* so = reinterpret_cast<float4*>(smem + C::kOffK);
            float2* sml = reinterpret_cast<float2*>(smem + C::kOffQ);
            const float inv_l = (n_act > 0) ? 1.0f / st.l : 0.0f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              if (n_act > 0) {
                tmem_ld_32x32b_x32(t_o + c * 32, o);
                tmem_wait_ld(o);
              } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = 0u;
              }
#pragma unroll
              for (int i = 0; i < 8; ++i)
                so[(t * (D / 4) + c * 8 + i) * kBM + row] =
                    make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
            }
            sml[t * kBM + row] = make_float2(n_act > 0 ? st.m : -INFINITY, n_act > 0 ? st.l : 0.0f);
            fence_acq_rel_cluster();
            __syncwarp();
            if (lane == 0)
              for (int r = 0; r < p.cluster_merge; ++r) mbar_arrive_remote_release(mapa_shared(b_cready, r));
          }
        } else {
          const size_t pbase = (static_cast<size_t>(U.slot) * kNSub + t) * (D / 4);
          float4* po = reinterpret_cast<float4*>(p.part_o);
          if (n_act > 0) {
            const float inv_l = 1.0f / st.l;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(t_o + c * 32, o);
              tmem_wait_ld(o);
              if (row_valid) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  po[(pbase + c * 8 + i) * kBM + row] =
                      make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                  __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
              }
            }
          }
          if (row_valid) {
            const size_t prow = (static_cast<size_t>(U.slot) * kNSub + t) * kBM + row;
            float2* pml = reinterpret_cast<float2*>(p.part_ml) + prow;
            *pml = make_float2(n_act > 0 ? st.m : -INFINITY, n_act > 0 ? st.l : 0.0f);
          }
        }
      }
      tr.rec(kTagEpiDone, t, u, 0);
      tc_fence_before();
    }
    if constexpr (!VARLEN) {
      if (p.cluster_merge > 0 && u_first < n_units) {
        // In-cluster merge: once all cluster_merge pieces of the block are
        // staged, cluster rank s merges rows [256 s / n, 256 (s + 1) / n) of
        // the block, reading every piece's O_s and (m, l) from its CTA's
        // shared memory (the combine pass's arithmetic: M = max m_s, w_s =
        // 2^(m_s - M) l_s, O = sum w_s O_s / sum w_s, lse = M ln 2 + ln sum
        // w_s); then every warp tells every peer that it has finished
        // reading, and no CTA leaves before all have.
        const int n = p.cluster_merge;
        const uint32_t rank = cluster_ctarank();
        Unit U;
        decode_unit<CAUSAL, VARLEN>(p, vl_pref, u_first, U);
        const bool ready = mbar_wait_acq_cluster(b_cready, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteMerge));
        if (ready) {
          const uint32_t so0 = smem_u32(smem + C::kOffK), sml0 = smem_u32(smem + C::kOffQ);
          const int r0 = static_cast<int>(rank) * kBlockRows / n, r1 = (static_cast<int>(rank) + 1) * kBlockRows / n;
          const int R = r1 - r0;
          for (int idx = warp * 32 + lane; idx < R * (D / 16); idx += 2 * kBM) {
            const int rr = r0 + idx % R, cb = idx / R;
            const int qr = U.q_row0 + rr;
            if (qr >= p.Lq) continue;
            const int tt = rr / kBM, rw = rr % kBM;
            float M = -INFINITY, L = 0.0f;
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
            for (int sp = 0; sp < n; ++sp) {
              const float2 ml = ld_dsmem_f2(mapa_shared(sml0 + (tt * kBM + rw) * 8, sp));
              float4 x[4];
#pragma unroll
              for (int c = 0; c < 4; ++c)
                x[c] = ld_dsmem_f4(mapa_shared(so0 + ((tt * (D / 4) + cb * 4 + c) * kBM + rw) * 16, sp));
              if (ml.x == -INFINITY) continue;   // a piece that saw no key
              const float mn = fmaxf(M, ml.x);
              const float r = (M == -INFINITY) ? 0.0f : ex2_approx(M - mn);
              const float w = ex2_approx(ml.x - mn) * ml.y;
              M = mn;
              L = L * r + w;
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                acc[4 * c] = acc[4 * c] * r + w * x[c].x;
                acc[4 * c + 1] = acc[4 * c + 1] * r + w * x[c].y;
                acc[4 * c + 2] = acc[4 * c + 2] * r + w * x[c].z;
                acc[4 * c + 3] = acc[4 * c + 3] * r + w * x[c].w;
              }
            }
            const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
            uint4* d4 = reinterpret_cast<uint4*>(out + ((static_cast<size_t>(U.b) * p.Lq + qr) * p.Hq + U.h) * D + cb * 16);
#pragma unroll
            for (int i = 0; i < 2; ++i)
              d4[i] = make_uint4(pack2<BF16>(acc[8 * i] * inv, acc[8 * i + 1] * inv),
                                 pack2<BF16>(acc[8 * i + 2] * inv, acc[8 * i + 3] * inv),
                                 pack2<BF16>(acc[8 * i + 4] * inv, acc[8 * i + 5] * inv),
                                 pack2<BF16>(acc[8 * i + 6] * inv, acc[8 * i + 7] * inv));
            if (cb == 0)
              p.lse[(static_cast<size_t>(U.b) * p.Hq + U.h) * p.Lq + qr] =
                  (L > 0.0f) ? M * 0.69314718055994531f + __logf(L) : -INFINITY;
          }
        }
        __syncwarp();
        if (lane == 0)
          for (int r = 0; r < n; ++r) mbar_arrive_remote_release(mapa_shared(b_cdone, r));
        mbar_wait_acq_cluster(b_cdone, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteMerge));
      }
    }
  }

  if (warp < 8) {
    Tracer tr;
    tr.init(p, (warp >> 2) == 0 ? kTrSoftmax0 : kTrSoftmax1);
    if ((threadIdx.x & 127) != 0) tr.off();
    tr.n = (ATTN_TRACE && p.trace) ? p.trace_cap - 1 : 0;   // the exit stamp goes in the last slot
    tr.rec(kTagGExit, 0, 0, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// split-KV combine.  Piece s holds O_s = u_s / l_s (fp32) and (m_s, l_s);
// with M = max_s m_s and w_s = 2^(m_s - M) l_s (the same r rescaling as
// across tiles), O = sum_s w_s O_s / sum_s w_s and lse = M ln 2 + ln sum_s w_s.
// Grid (groups, 2 sub-tiles, D/16 column blocks), one thread per query row
// and 16 columns.  Launched as a programmatic dependent of the forward
// kernel: it may be scheduled early and waits here until that grid has
// completed and its writes are visible.
// ---------------------------------------------------------------------------
template <int D, bool BF16>
__global__ void __launch_bounds__(kBM) attn_combine_kernel(const __grid_constant__ CombineParams p) {
  using T = typename IO<BF16>::T;
  const int* ge = p.groups + blockIdx.x * kGroupInts;
  const int bh = __ldg(ge), mb = __ldg(ge + 1), slot0 = __ldg(ge + 2), ns = __ldg(ge + 3);
  const int t = blockIdx.y, cb = blockIdx.z, row = threadIdx.x;
  const int qrow = mb * kBlockRows + t * kBM + row;
  if (qrow >= p.Lq) return;
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  grid_wait_prerequisites();
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  const float4* po = reinterpret_cast<const float4*>(p.part_o);
  const size_t ml_base = static_cast<size_t>(slot0) * kNSub * kBM + t * kBM + row;
  const size_t o_base = (static_cast<size_t>(slot0) * kNSub + t) * (D / 4) + cb * 4;
  constexpr size_t kMlStride = kNSub * kBM;      // per piece, in float2
  constexpr size_t kOStride = kNSub * (D / 4);   // per piece, in 4-column groups
  // Pieces in batches of four: every load of a batch ((m, l) and this
  // thread's 16 columns of O_s) is issued before any is used, so a batch
  // costs one L2 round trip.  Batches merge with a running max, the same
  // r rescaling again.
  float M = -INFINITY, L = 0.0f;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
  for (int s0 = 0; s0 < ns; s0 += 4) {
    float2 mlv[4];
    float4 x[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool in = s0 + i < ns;
      mlv[i] = in ? __ldcg(ml + ml_base + (s0 + i) * kMlStride) : make_float2(-INFINITY, 0.0f);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        x[i][c] = in ? __ldcg(po + (o_base + (s0 + i) * kOStride + c) * kBM + row) : make_float4(0, 0, 0, 0);
    }
    float mb = M;
#pragma unroll
    for (int i = 0; i < 4; ++i) mb = fmaxf(mb, mlv[i].x);
    if (mb == -INFINITY) continue;   // no piece so far saw a key
    const float r = (M == -INFINITY) ? 0.0f : ex2_approx(M - mb);
    M = mb;
    L *= r;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] *= r;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (mlv[i].x == -INFINITY) continue;   // an empty piece (its O_s was never written)
      const float w = ex2_approx(mlv[i].x - M) * mlv[i].y;
      L += w;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[4 * c] += w * x[i][c].x;
        acc[4 * c + 1] += w * x[i][c].y;
        acc[4 * c + 2] += w * x[i][c].z;
        acc[4 * c + 3] += w * x[i][c].w;
      }
    }
  }
  const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
  T* dst = reinterpret_cast<T*>(p.o) + ((static_cast<size_t>(b) * p.Lq + qrow) * p.Hq + h) * D + cb * 16;
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 2; ++i)
    d4[i] = make_uint4(pack2<BF16>(acc[8 * i] * inv, acc[8 * i + 1] * inv),
                       pack2<BF16>(acc[8 * i + 2] * inv, acc[8 * i + 3] * inv),
                       pack2<BF16>(acc[8 * i + 4] * inv, acc[8 * i + 5] * inv),
                       pack2<BF16>(acc[8 * i + 6] * inv, acc[8 * i + 7] * inv));
  if (cb == 0)
    p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.Lq + qrow] =
        (L > 0.0f) ? M * 0.69314718055994531f + __logf(L) : -INFINITY;
}


// ---------------------------------------------------------------------------
// Merge of decode pieces.  Block (sequence b, head group) x 16-column slice,
// one warp per query head r of the group (row r of the pieces' first
// sub-tile, the only one a single query fills); lane s takes piece s of each
// chunk of 32, so a chunk's loads ((m, l) and 16 columns of O_s) are one L2
// round trip, and the warp reduces across its lanes with the same r-rescale
// as the split-KV combine above: M = max_s m_s, w_s = 2^(m_s - M) l_s.
// Piece s of (b, group) is unit pref[b] + s * groups + group, in key order of
// s.  Sequences that were not cut (one piece) were written by the decode
// kernel, and with malformed offsets that kernel has zeroed every row, so
// those blocks return at once.  Launched as a programmatic dependent of the
// decode kernel.
// ---------------------------------------------------------------------------
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_combine_decode_kernel(const __grid_constant__ DecodeCombineParams p) {
  using T = typename IO<BF16>::T;
  const int n_hg = p.Hq >> p.pack_log2;
  const int b = blockIdx.x / n_hg, hg = blockIdx.x - b * n_hg;
  const int cb = blockIdx.y;
  const int row = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ak = __ldg(p.cu_seqlens_k + b);
  const int ek = __ldg(p.cu_seqlens_k + b + 1);
  grid_wait_prerequisites();
  if (p.pref[p.B + 1] != 0 || ek < ak) return;
  const int pcs = decode_pieces(ek - ak, p.split);
  if (pcs <= 1) return;
  const int slot0 = p.pref[b] + hg;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  const float4* po = reinterpret_cast<const float4*>(p.part_o);
  const size_t ml_stride = static_cast<size_t>(n_hg) * kNSub * kBM;      // per piece, in float2
  const size_t o_stride = static_cast<size_t>(n_hg) * kNSub * (D / 4);   // per piece, in 4-column groups
  const size_t ml_base = static_cast<size_t>(slot0) * kNSub * kBM + row;
  const size_t o_base = static_cast<size_t>(slot0) * kNSub * (D / 4) + cb * 4;
  float M = -INFINITY, L = 0.0f;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
  for (int s0 = 0; s0 < pcs; s0 += 32) {
    const int s = s0 + lane;
    const bool in = s < pcs;
    float2 mlv = in ? __ldcg(ml + ml_base + s * ml_stride) : make_float2(-INFINITY, 0.0f);
    float4 x[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      x[c] = in ? __ldcg(po + (o_base + s * o_stride + c) * kBM + row) : make_float4(0, 0, 0, 0);
    float mc = mlv.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
    if (mc == -INFINITY) continue;   // no piece of this chunk saw a key
    const float mn = fmaxf(M, mc);
    const float r = (M == -INFINITY) ? 0.0f : ex2_approx(M - mn);
    M = mn;
    // an empty piece's O_s was never written: weight 0 and its values dropped
    const bool live = mlv.x != -INFINITY;
    float w = live ? ex2_approx(mlv.x - M) * mlv.y : 0.0f;
    float v[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      v[4 * c] = live ? w * x[c].x : 0.0f;
      v[4 * c + 1] = live ? w * x[c].y : 0.0f;
      v[4 * c + 2] = live ? w * x[c].z : 0.0f;
      v[4 * c + 3] = live ? w * x[c].w : 0.0f;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      w += __shfl_xor_sync(0xffffffffu, w, o);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    }
    L = L * r + w;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = acc[i] * r + v[i];
  }
  if (lane != 0) return;
  const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
  const int head = (hg << p.pack_log2) + row;
  T* dst = reinterpret_cast<T*>(p.o) + (static_cast<size_t>(b) * p.Hq + head) * D + cb * 16;
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 2; ++i)
    d4[i] = make_uint4(pack2<BF16>(acc[8 * i] * inv, acc[8 * i + 1] * inv),
                       pack2<BF16>(acc[8 * i + 2] * inv, acc[8 * i + 3] * inv),
                       pack2<BF16>(acc[8 * i + 4] * inv, acc[8 * i + 5] * inv),
                       pack2<BF16>(acc[8 * i + 6] * inv, acc[8 * i + 7] * inv));
  if (cb == 0)
    p.lse[static_cast<size_t>(head) * p.B + b] = (L > 0.0f) ? M * 0.69314718055994531f + __logf(L) : -INFINITY;
}

}  // namespace attn
