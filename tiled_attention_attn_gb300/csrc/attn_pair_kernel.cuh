// sm_103a attention forward on CTA pairs: tcgen05 .cta_group::2 MMAs span
// two SMs, so one instruction computes a 256-row x 256-key score tile (each
// CTA its own 128 query rows) and each CTA stages only half of every key and
// value tile.
//
// Method (page S23-J17, clxhxhhr.top/posts/5544, §3.1): per query row keep
// the running max m, the exp-sum l relative to m and the value accumulator u
// with the same weights; when m grows, r = exp(m_old - m_new) rescales l and
// u.  The score tile S and probability tile P live only in TMEM and
// registers; only O and the per-row log-sum-exp reach global memory.
//
// A work unit is a 256-row query block against a range of 256-key tiles.
// CTA r of the pair owns query rows [128 r, 128 r + 128) of the block; it
// loads keys [128 r, 128 r + 128) of every key tile (its half of the N
// columns of S = Q K^T) and value columns [r d/2, (r+1) d/2) of every value
// tile (its half of the N columns of O += P V).
//
// CTA layout (384 threads, one CTA per SM, clusters of two):
//   warps 0-7  softmax: warp w owns TMEM lane quarter w % 4 (32 query rows)
//              and key columns [128 (w / 4), 128 (w / 4) + 128) of S, so two
//              threads share a row; they exchange the row max per tile
//   warp 8     TMA producer (each CTA its own halves; completion is counted
//              on the leader CTA's barriers)
//   warp 9     TMEM allocation (both CTAs); in the even (leader) CTA one
//              thread issues every S = Q K^T of the pair
//   warp 10    in the leader CTA, one thread issues every O += P V: each
//              issuer's barrier waits overlap the other's MMAs, so the
//              tensor pipe is not left idle while one thread waits
//   warp 11    completes the third warpgroup (register reallocation works
//              on whole warpgroups) and otherwise idles
// Epilogue: O is staged in the unit's Q buffer (128-byte swizzled) and
// written by TMA stores; the buffer is handed back to the producer once the
// stores have read it.
// TMEM (512 columns x 128 lanes): S at [0, 256), P (16-bit, two per column)
// at [256, 384), the accumulator u at [384, 384 + d).  Because P does not
// overwrite S, the next tile's S = Q K^T is issued as soon as the softmax has
// read S, and runs on the tensor cores while the softmax works: the MMA order
// is S(j+1), then P V(j).
//
// Split key ranges: pieces of one query block write their unnormalised u and
// (m, l) to a workspace; the row slices of the block are merged by whichever
// piece completes each slice's arrival count last (pieces visit the slices in
// rotated order, so simultaneous finishers share the merging), applying the
// same r = 2^(m_s - M) rescaling across pieces.  No piece waits for another.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_params.h"
#include "ptx.cuh"

namespace attn {
namespace pair {

// warp roles of the pair kernel (its own, independent of the single-CTA kernel's)
constexpr int kPairWarpTMA = 8;   // TMA producer
constexpr int kPairWarpMMA = 9;   // S = Q K^T issuer (and TMEM allocator); warp 10 issues P.V

template <int D>
struct Cfg {
  static_assert(D == 128, "the pair kernel is built for head_dim 128");
  static constexpr int kQBytes = kPairRows * D * 2;        // this CTA's query rows
  static constexpr int kKBytes = (kPairBN / 2) * D * 2;    // this CTA's half of a key tile
  static constexpr int kVBytes = kPairBN * (D / 2) * 2;    // this CTA's half of a value tile
  static constexpr int kChunks = D / 64;                   // 128-byte swizzle atoms per Q / K row
  static constexpr int kNQ = 2, kNK = 2, kNV = 2;          // ring depths
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kNQ * kQBytes;
  static constexpr int kOffV = kOffK + kNK * kKBytes;
  static constexpr int kOffBar = kOffV + kNV * kVBytes;
  // barriers: q_full[NQ], q_empty[NQ], k_full[NK], k_empty[NK], v_full[NV],
  //           v_empty[NV], s_full, s_free, p_full, pv_done, drain, xchg[4]
  //           (the two warps of a lane quarter), merge (the eight softmax warps)
  static constexpr int kNBars = 2 * (kNQ + kNK + kNV) + 5 + 4 + 1;
  static constexpr int kOffMisc = kOffBar + kNBars * 8;    // tmem slot, abort flag, merge flags
  static constexpr int kOffRed = kOffMisc + 64;            // row-max exchange [2][2][128] floats
  static constexpr int kOffLex = kOffRed + 2 * 2 * kPairRows * 4;   // l exchange [2][2][128]
  static constexpr int kSmem = kOffLex + 2 * 2 * kPairRows * 4 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTS = 0, kTP = 256, kTO = 384;  // TMEM column offsets
};

template <bool BF16>
struct IO;
template <>
struct IO<true> {
  using T = __nv_bfloat16;
};
template <>
struct IO<false> {
  using T = __half;
};

#ifndef ATTN_TRACE
#define ATTN_TRACE 0
#endif
// Phase trace (traced build only): per CTA four streams of (tag word, SM
// clock) pairs, in the layout of the single-CTA kernel's trace.
struct PTracer {
  unsigned long long* base;
  int cap, n;
  __device__ __forceinline__ void init(const PairParams& p, int stream) {
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

struct Unit {
  int b, h, g;
  int q_row0;            // first query row of the 256-row block
  int kv_begin, kv_end;  // 256-key tiles [kv_begin, kv_end)
  int split, n_split, slot;
};

__device__ __forceinline__ void decode(const PairParams& p, int u, Unit& U) {
  const int* e = (p.n_inline ? p.units_inline : p.units) + u * kUnitInts;
  const int bh = e[0];
  U.b = bh / p.Hq;
  U.h = bh - U.b * p.Hq;
  U.g = U.h / p.group;
  U.q_row0 = e[1] * kPairBlock;
  U.kv_begin = e[2];
  U.kv_end = e[3];
  U.split = e[4];
  U.n_split = e[5];
  U.slot = e[6];
}

// The merge counter of a split group (one word per group and CTA of the
// pair): (epoch << 32) | arrivals.  A word left by another call (another
// epoch) restarts at one; replays of a captured call keep counting in the
// same epoch.  Returns this piece's arrival number (1-based), or 0 after 2^20
// failed exchanges (reported).
__device__ __forceinline__ unsigned int group_arrive(unsigned long long* c, unsigned int epoch, int* err) {
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(c);
  for (int it = 0; it < (1 << 20); ++it) {
    const unsigned int ep = static_cast<unsigned int>(old >> 32);
    const unsigned long long nw =
        (ep == epoch) ? old + 1ull : ((static_cast<unsigned long long>(epoch) << 32) | 1ull);
    const unsigned long long prev = atomicCAS(c, old, nw);
    if (prev == old) return static_cast<unsigned int>(nw & 0xffffffffull);
    old = prev;
  }
  atomicCAS(err, 0, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteMerge));
  return 0;
}

// Waits until the group's word reaches `target` arrivals in this epoch: every
// piece of the group has written its partial.  The pieces are resident
// (cooperative launch; a split piece is the first unit of its pair), so the
// wait ends; it is bounded all the same.
__device__ __forceinline__ bool group_wait(const unsigned long long* c, unsigned int epoch, unsigned int target,
                                           const WaitCtl& w) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(c) : "memory");
    if (static_cast<unsigned int>(v >> 32) == epoch && static_cast<unsigned int>(v & 0xffffffffull) >= target)
      return true;
    if ((it & 15u) == 15u && global_timer_ns() - t0 > w.timeout_ns) {
      report_error(w, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteMerge));
      return false;
    }
  }
}

// A handshake among whole warps: each warp arrives once (lane 0, after its
// lanes' shared-memory writes) on `bar`, whose count is the number of warps,
// and waits for the phase to complete.  Bounded like every other wait, so a
// warp that gave up elsewhere cannot leave its partners blocked.
__device__ __forceinline__ bool warp_handshake(uint32_t bar, uint32_t& cnt, const WaitCtl& wc) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = mbar_wait_warp(bar, cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteXchg));
  ++cnt;
  return ok;
}

// Softmax of this thread's 128 columns of one 256-key S tile, first stage:
// loads its 128 columns of S into `s` and the other thread's 128 columns of
// the row (used only for the maximum), releases the S buffer, masks keys
// beyond `lim` (`lim_o` for the other half) and updates the running max `m`
// (exp2 units: scale * log2(e) times the score).  Both threads of a row take
// the maximum of the same 256 values, so they agree on it without exchanging
// anything.  Returns the rescale factor `r` of l and u (1 when the max did not
// move enough to rescale; `resc` set when it did) and the exponent offset
// `moff`.
template <bool MASK>
__device__ __forceinline__ void softmax_max(uint32_t t_s, uint32_t t_s_other, int lim, int lim_o, float c_log2,
                                            float& m, bool first, uint32_t s_free_c, bool arrive_lane,
                                            float (&s)[128], float& r, bool& resc, float& moff) {
  float mx[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
  // the other thread's half of the row (its maximum only), 32 columns at a time
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    uint32_t x[32];
    tmem_ld_32x32b_x32(t_s_other + h * 32, x);
    tmem_wait_ld(x);
#pragma unroll
    for (int i = 0; i < 32; i += 16)
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float a = __uint_as_float(x[i + k]), b = __uint_as_float(x[i + 8 + k]);
        if constexpr (MASK) {
          a = (h * 32 + i + k <= lim_o) ? a : -INFINITY;
          b = (h * 32 + i + 8 + k <= lim_o) ? b : -INFINITY;
        }
        mx[k] = fmax3(mx[k], a, b);
      }
  }
  // this thread's half, kept
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
    for (int i = 0; i < 64; i += 16)
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], s[i + k], s[i + 8 + k]);
    tmem_wait_ld(r2);
#pragma unroll
    for (int i = 0; i < 64; ++i) s[64 + i] = __uint_as_float(r2[i]);
  }
  // S is in registers: the next tile's S may overwrite it
  tc_fence_before();
  __syncwarp();
  if (arrive_lane) mbar_arrive_cluster(s_free_c);
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
  const float m_old = m;
  resc = false;
  if (m_tile > m_old && (first || m_old == -INFINITY || m_tile - m_old > 8.0f)) {
    resc = true;
    m = m_tile;
  }
  moff = (m == -INFINITY) ? 0.0f : m;
  r = resc ? ((m_old == -INFINITY) ? 0.0f : ex2_approx(m_old - m)) : 1.0f;
}

// Second stage, for 64 of the thread's columns starting at C0: p = 2^(s c -
// moff) (masked keys 0), packed to 16-bit pairs in `pk`, summed into `sum`.
template <int C0, bool MASK, bool BF16>
__device__ __forceinline__ void softmax_exp64(const float (&s)[128], int lim, float c_log2, float moff,
                                              uint32_t (&pk)[32], float& sum) {
  const float2 c2 = make_float2(c_log2, c_log2);
  const float2 nm2 = make_float2(-moff, -moff);
  float2 sum_a = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 64; i += 4) {
    const int c = C0 + i;
    const float2 x0 = ffma2(make_float2(s[c], s[c + 1]), c2, nm2);
    const float2 x1 = ffma2(make_float2(s[c + 2], s[c + 3]), c2, nm2);
    float2 e0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
    float2 e1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
    if constexpr (MASK) {
      e0.x = (c <= lim) ? e0.x : 0.0f;
      e0.y = (c + 1 <= lim) ? e0.y : 0.0f;
      e1.x = (c + 2 <= lim) ? e1.x : 0.0f;
      e1.y = (c + 3 <= lim) ? e1.y : 0.0f;
    }
    sum_a = fadd2(sum_a, e0);
    sum_b = fadd2(sum_b, e1);
    pk[i / 2] = pack2<BF16>(e0.x, e0.y);
    pk[i / 2 + 1] = pack2<BF16>(e1.x, e1.y);
  }
  const float2 sum2 = fadd2(sum_a, sum_b);
  sum += sum2.x + sum2.y;
}

__device__ __forceinline__ void store_p32(uint32_t t_p, const uint32_t (&pk)[32]) {
  uint32_t w0[16], w1[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    w0[i] = pk[i];
    w1[i] = pk[16 + i];
  }
  tmem_st_32x32b_x16(t_p, w0);
  tmem_st_32x32b_x16(t_p + 16, w1);
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kPairThreads, 1) attn_pair_kernel(const __grid_constant__ PairParams p) {
  using C = Cfg<D>;
  using T = typename IO<BF16>::T;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();   // 0: leader (issues the MMAs), 1: peer
  const int pair_id = blockIdx.x >> 1;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sK = sbase + C::kOffK;
  const uint32_t sV = sbase + C::kOffV;
  const uint32_t bar0 = sbase + C::kOffBar;
  auto b_q_full = [&](int i) { return bar0 + 8 * i; };
  auto b_q_empty = [&](int i) { return bar0 + 8 * (C::kNQ + i); };
  auto b_k_full = [&](int i) { return bar0 + 8 * (2 * C::kNQ + i); };
  auto b_k_empty = [&](int i) { return bar0 + 8 * (2 * C::kNQ + C::kNK + i); };
  auto b_v_full = [&](int i) { return bar0 + 8 * (2 * C::kNQ + 2 * C::kNK + i); };
  auto b_v_empty = [&](int i) { return bar0 + 8 * (2 * C::kNQ + 2 * C::kNK + C::kNV + i); };
  const uint32_t bar_x = bar0 + 8 * (2 * (C::kNQ + C::kNK + C::kNV));
  const uint32_t b_s_full = bar_x;
  const uint32_t b_s_free = bar_x + 8;
  const uint32_t b_p_full = bar_x + 16;
  const uint32_t b_pv_done = bar_x + 24;
  const uint32_t b_drain = bar_x + 32;
  auto b_xchg = [&](int q) { return bar_x + 40 + 8 * q; };
  const uint32_t b_merge = bar_x + 72;

  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  volatile int* merge_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);   // [2]
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);
  float* lex = reinterpret_cast<float*>(smem + C::kOffLex);

  WaitCtl wc{p.err, abort_flag, p.timeout_ns};

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::kNQ; ++i) {
      mbar_init(b_q_full(i), 1);
      mbar_init(b_q_empty(i), 1);
    }
    for (int i = 0; i < C::kNK; ++i) {
      mbar_init(b_k_full(i), 1);
      mbar_init(b_k_empty(i), 1);
    }
    for (int i = 0; i < C::kNV; ++i) {
      mbar_init(b_v_full(i), 1);
      mbar_init(b_v_empty(i), 1);
    }
    mbar_init(b_s_full, 1);
    mbar_init(b_s_free, 2 * 8);   // every softmax warp of both CTAs
    mbar_init(b_p_full, 2 * 8);
    mbar_init(b_pv_done, 1);
    mbar_init(b_drain, 2);        // one commit from each MMA-issuing thread
    for (int q = 0; q < 4; ++q) mbar_init(b_xchg(q), 2);
    mbar_init(b_merge, 8);
    fence_mbar_init();
  }
  if (warp == kPairWarpMMA) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == kPairWarpTMA && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  tc_fence_before();
  // both CTAs' barriers are initialised and their TMEM allocated before any
  // remote arrival, load completion or MMA
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int* off = p.n_inline ? p.pair_off_inline : p.pair_off;
  const int u_first = off[pair_id];
  const int u_end = off[pair_id + 1];

  if (warp >= 8) {
    // each register limit governs exactly the code of its warpgroup
    regs_dec<kPairRegsOther>();
  if (warp == kPairWarpTMA) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t q_cnt = 0, k_cnt = 0, v_cnt = 0;
      const bool leader = rank == 0;
      PTracer tr;
      tr.init(p, kTrProducer);
      bool ok = true;
      auto load_k = [&](const Unit& U, int j) -> bool {
        const int st = k_cnt % C::kNK;
        if (!mbar_wait(b_k_empty(st), ((k_cnt / C::kNK) & 1) ^ 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKEmpty)))
          return false;
        const uint32_t full = mapa_shared(b_k_full(st), 0);
        if (leader) mbar_arrive_expect_tx(b_k_full(st), 2 * C::kKBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d_pair(sK + st * C::kKBytes + c * (kPairBN / 2) * 128, &p.tm_k, full, c * 64, U.g,
                           j * kPairBN + static_cast<int>(rank) * (kPairBN / 2), U.b);
        tr.rec(kTagKIssue, 0, 0, j);
        ++k_cnt;
        return true;
      };
      auto load_v = [&](const Unit& U, int j) -> bool {
        const int st = v_cnt % C::kNV;
        if (!mbar_wait(b_v_empty(st), ((v_cnt / C::kNV) & 1) ^ 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteVEmpty)))
          return false;
        const uint32_t full = mapa_shared(b_v_full(st), 0);
        if (leader) mbar_arrive_expect_tx(b_v_full(st), 2 * C::kVBytes);
        tma_load_4d_pair(sV + st * C::kVBytes, &p.tm_v, full, static_cast<int>(rank) * (D / 2), U.g, j * kPairBN,
                         U.b);
        tr.rec(kTagVIssue, 0, 0, j);
        ++v_cnt;
        return true;
      };
      for (int u = u_first; u < u_end && ok; ++u) {
        Unit U;
        decode(p, u, U);
        if (U.kv_end <= U.kv_begin) continue;   // no key visible: the softmax warps write the zeros
        const int qs = q_cnt % C::kNQ;
        if (!mbar_wait(b_q_empty(qs), ((q_cnt / C::kNQ) & 1) ^ 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteQEmpty)))
          break;
        const uint32_t qfull = mapa_shared(b_q_full(qs), 0);
        if (leader) mbar_arrive_expect_tx(b_q_full(qs), 2 * C::kQBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d_pair(sQ + qs * C::kQBytes + c * kPairRows * 128, &p.tm_q, qfull, c * 64, U.h,
                           U.q_row0 + static_cast<int>(rank) * kPairRows, U.b);
        tr.rec(kTagQIssue, 0, u, 0);
        ++q_cnt;
        // the MMA order is S(j0), S(j0+1), PV(j0), S(j0+2), PV(j0+1), ...:
        // keys run one tile ahead of values
        const int n = U.kv_end - U.kv_begin;
        for (int i = 0; i <= n && ok; ++i) {
          if (i < n) ok = load_k(U, U.kv_begin + i);
          if (ok && i > 0) ok = load_v(U, U.kv_begin + i - 1);
        }
      }
      // On an abort the leader lets issued loads land (its full barriers
      // count both CTAs' bytes) before the pair exits.
      if (*abort_flag && leader) {
        for (int s = 0; s < C::kNK; ++s) {
          const uint32_t n = (k_cnt + C::kNK - 1 - s) / C::kNK;
          if (n > 0) mbar_wait_cluster(b_k_full(s), (n - 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
        }
        for (int s = 0; s < C::kNV; ++s) {
          const uint32_t n = (v_cnt + C::kNV - 1 - s) / C::kNV;
          if (n > 0) mbar_wait_cluster(b_v_full(s), (n - 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
        }
        for (int s = 0; s < C::kNQ; ++s) {
          const uint32_t n = (q_cnt + C::kNQ - 1 - s) / C::kNQ;
          if (n > 0) mbar_wait_cluster(b_q_full(s), (n - 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
        }
      }
    }
  } else if (warp == kPairWarpMMA && rank == 0 && lane == 0) {
    // ------------------------------------------------------------------ S = Q K^T issuer (leader CTA)
    constexpr uint32_t kIdescS = idesc_f16_f32acc(2 * kPairRows, kPairBN, BF16, false);
    constexpr uint16_t kBoth = 0x3;
    const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dk0 = sdesc_sw128(sK, 16, 1024);
    uint32_t q_cnt = 0, k_cnt = 0, s_cnt = 0;
    PTracer tr;
    tr.init(p, kTrMMA);
    tr.rec(kTagStart, 0, 0, 0);
    bool ok = true;
    for (int u = u_first; u < u_end && ok; ++u) {
      Unit U;
      decode(p, u, U);
      if (U.kv_end <= U.kv_begin) continue;
      const int qs = q_cnt % C::kNQ;
      if (!mbar_wait(b_q_full(qs), (q_cnt / C::kNQ) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteQFull))) break;
      tr.rec(kTagQFull, 0, u, 0);
      const uint64_t a0 = dq0 + ((qs * C::kQBytes) >> 4);
      for (int j = U.kv_begin; j < U.kv_end; ++j) {
        const int ks = k_cnt % C::kNK;
        if (!mbar_wait(b_k_full(ks), (k_cnt / C::kNK) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteKFull))) {
          ok = false;
          break;
        }
        tr.rec(kTagKFull, 0, u, j);
        // S is overwritten: every softmax thread has read the previous S
        if (s_cnt > 0 && !mbar_wait(b_s_free, (s_cnt - 1) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteSFree))) {
          ok = false;
          break;
        }
        tr.rec(kTagSFreeWait, 0, u, j);
        tc_fence_after();
        const uint64_t b0 = dk0 + ((ks * C::kKBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offa = ((kk >> 2) * kPairRows * 128 + (kk & 3) * 32) >> 4;
          const uint32_t offb = ((kk >> 2) * (kPairBN / 2) * 128 + (kk & 3) * 32) >> 4;
          umma_ss_pair(tmem + C::kTS, a0 + offa, b0 + offb, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit_pair(b_k_empty(ks), kBoth);
        umma_commit_pair(b_s_full, kBoth);
        tr.rec(kTagSIssue, 0, u, j);
        ++k_cnt;
        ++s_cnt;
      }
      ++q_cnt;
    }
    // every MMA issued by this thread has completed once the drain barrier
    // fires (it counts both issuing threads)
    umma_commit_pair(b_drain, 0x1);
    mbar_wait(b_drain, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
  } else if (warp == kPairWarpMMA + 1 && rank == 0 && lane == 0) {
    // ------------------------------------------------------------------ O += P V issuer (leader CTA)
    constexpr uint32_t kIdescO = idesc_f16_f32acc(2 * kPairRows, D, BF16, true);
    constexpr uint16_t kBoth = 0x3;
    const uint64_t dv0 = sdesc_sw128(sV, 32768, 1024);
    uint32_t v_cnt = 0, p_cnt = 0;
    PTracer tr;
    tr.init(p, kTrProducer + 0);
    tr.off();
    bool ok = true;
    for (int u = u_first; u < u_end && ok; ++u) {
      Unit U;
      decode(p, u, U);
      for (int j = U.kv_begin; j < U.kv_end; ++j) {
        const int vs = v_cnt % C::kNV;
        if (!mbar_wait(b_v_full(vs), (v_cnt / C::kNV) & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteVFull))) {
          ok = false;
          break;
        }
        if (!mbar_wait(b_p_full, p_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSitePFull))) {
          ok = false;
          break;
        }
        ++p_cnt;
        tc_fence_after();
        const uint64_t bv = dv0 + ((vs * C::kVBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kPairBN / 16; ++kk)
          umma_ts_pair(tmem + C::kTO, tmem + C::kTP + kk * 8, bv + ((kk * 2048) >> 4), kIdescO,
                       (j == U.kv_begin && kk == 0) ? 0u : 1u);
        umma_commit_pair(b_v_empty(vs), kBoth);
        umma_commit_pair(b_pv_done, kBoth);
        ++v_cnt;
      }
    }
    umma_commit_pair(b_drain, 0x1);
    mbar_wait(b_drain, 0, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteDrain), false);
  }
  } else {
    regs_inc<kPairRegsSoftmax>();
    // ------------------------------------------------------------------ softmax (both CTAs)
    const int quarter = warp & 3;
    const int half = warp >> 2;                    // key columns [128 half, 128 half + 128) of S
    const int row = quarter * 32 + lane;           // TMEM lane = query row within this CTA
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::kTS + half * 128;
    const uint32_t t_s_other = tmem + lane_off + C::kTS + (half ^ 1) * 128;
    const uint32_t t_p = tmem + lane_off + C::kTP + half * 64;
    const uint32_t t_o = tmem + lane_off + C::kTO + half * (D / 2);
    const uint32_t s_free_c = mapa_shared(b_s_free, 0);
    const uint32_t p_full_c = mapa_shared(b_p_full, 0);
    const uint32_t xbar = b_xchg(quarter);         // the two warps of this lane quarter
    uint32_t xcnt = 0, mcnt = 0;                   // handshake phases seen
    const float c_log2 = p.scale_log2;
    uint32_t s_cnt = 0, pv_cnt = 0, q_cnt = 0;
    int pending_q = -1;   // thread 0: Q slot whose O store may still be reading it
    T* out = reinterpret_cast<T*>(p.o);
    PTracer tr;
    tr.init(p, half == 0 ? kTrSoftmax0 : kTrSoftmax1);
    if (row != 0) tr.off();
    tr.rec(kTagGEnter, half, 0, 0);
    int par = 0;                                   // row-max exchange buffer
    for (int u = u_first; u < u_end; ++u) {
      Unit U;
      decode(p, u, U);
      const int q_first = U.q_row0 + static_cast<int>(rank) * kPairRows;
      const int qrow = q_first + row;
      const bool row_valid = qrow < p.Lq;
      int lim_key = row_valid ? p.Lk - 1 : -1;
      if constexpr (CAUSAL) lim_key = row_valid ? min(lim_key, qrow + (p.Lk - p.Lq)) : -1;
      if (U.kv_end <= U.kv_begin) {
        // a block whose rows see no key (causal, more queries than keys)
        if (row_valid) {
          uint4* d4 = reinterpret_cast<uint4*>(out + ((static_cast<size_t>(U.b) * p.Lq + qrow) * p.Hq + U.h) * D +
                                               half * (D / 2));
#pragma unroll
          for (int i = 0; i < D / 16; ++i) d4[i] = make_uint4(0, 0, 0, 0);
          if (half == 0) p.lse[(static_cast<size_t>(U.b) * p.Hq + U.h) * p.Lq + qrow] = -INFINITY;
        }
        continue;
      }
      const int qs = q_cnt % C::kNQ;
      ++q_cnt;
      float m = -INFINITY, l = 0.0f;
      bool ok = true;
      for (int j = U.kv_begin; j < U.kv_end; ++j) {
        if (!mbar_wait_warp(b_s_full, s_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSiteSFull))) { ok = false; break; }
        tr.rec(kTagSFull, half, u, j);
        ++s_cnt;
        tc_fence_after();
        const int col0 = j * kPairBN + half * 128;   // key of this thread's first column
        const int lim = lim_key - col0;
        const bool mask_tile = __any_sync(0xffffffffu, lim < 127);
        const bool first = (j == U.kv_begin);
        float sv[128];
        float r, moff;
        bool resc;
        const int lim_o = lim_key - (j * kPairBN + (half ^ 1) * 128);
        const bool mask_any = __any_sync(0xffffffffu, lim < 127 || lim_o < 127);
        if (mask_any)
          softmax_max<true>(t_s, t_s_other, lim, lim_o, c_log2, m, first, s_free_c, lane == 0, sv, r, resc, moff);
        else
          softmax_max<false>(t_s, t_s_other, lim, lim_o, c_log2, m, first, s_free_c, lane == 0, sv, r, resc, moff);
        tr.rec(kTagMaxDone, half, u, j);
        float sum = 0.0f;
        uint32_t pk[32];
        if (mask_tile)
          softmax_exp64<0, true, BF16>(sv, lim, c_log2, moff, pk, sum);
        else
          softmax_exp64<0, false, BF16>(sv, lim, c_log2, moff, pk, sum);
        if (!first) {
          // the previous tile's P.V has read P and updated u
          tr.rec(kTagPvWait, half, u, j);
          if (!mbar_wait_warp(b_pv_done, pv_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSitePvDone))) {
            ok = false;
            break;
          }
          tr.rec(kTagPvDone, half, u, j);
          ++pv_cnt;
          tc_fence_after();
          if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
            for (int c = 0; c < D / 2 / 16; ++c) {
              uint32_t o[16];
              tmem_ld_32x32b_x16(t_o + c * 16, o);
              tmem_wait_ld(o);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * r);
              tmem_st_32x32b_x16(t_o + c * 16, o);
            }
          }
        }
        store_p32(t_p, pk);
        if (mask_tile)
          softmax_exp64<64, true, BF16>(sv, lim, c_log2, moff, pk, sum);
        else
          softmax_exp64<64, false, BF16>(sv, lim, c_log2, moff, pk, sum);
        store_p32(t_p + 32, pk);
        l = l * r + sum;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(p_full_c);
        tr.rec(kTagPArrive, half, u, j);
        if (tid == 0 && pending_q >= 0) {
          // the previous unit's O store has read its staging buffer: the
          // producer may load a new Q block there
          bulk_wait_read_all();
          mbar_arrive(b_q_empty(pending_q));
          pending_q = -1;
        }
      }
      if (!ok) break;
      // the unit's last P.V
      if (!mbar_wait_warp(b_pv_done, pv_cnt & 1, wc, ATTN_DEVERR_WAIT_TIMEOUT_SITE(kSitePvDone))) break;
      tr.rec(kTagODone, half, u, 0);
      ++pv_cnt;
      tc_fence_after();
      // l of the whole row: this thread's columns plus the other thread's
      lex[(par * 2 + half) * kPairRows + row] = l;
      if (!warp_handshake(xbar, xcnt, wc)) break;
      l += lex[(par * 2 + (half ^ 1)) * kPairRows + row];
      par ^= 1;
      if (U.n_split <= 1) {
        // O = u / l, lse = m ln 2 + ln l (m in exp2 units).  O is staged in
        // this unit's Q buffer (every S of the unit has completed) in the
        // 128-byte-swizzled layout of the O tensor map, and one thread
        // stores each 64-column half with TMA: whole lines instead of one
        // row per thread.
        const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
        const uint32_t stg = sQ + qs * C::kQBytes + half * (kPairRows * 128) + row * 128;
#pragma unroll
        for (int c = 0; c < D / 2 / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + c * 32, o);
          tmem_wait_ld(o);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t unit16 = static_cast<uint32_t>(c * 4 + i) ^ static_cast<uint32_t>(row & 7);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg + unit16 * 16), "r"(w[4 * i]),
                         "r"(w[4 * i + 1]), "r"(w[4 * i + 2]), "r"(w[4 * i + 3])
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        if (row_valid && half == 0)
          p.lse[(static_cast<size_t>(U.b) * p.Hq + U.h) * p.Lq + qrow] =
              (l > 0.0f) ? m * 0.69314718055994531f + __logf(l) : -INFINITY;
        tc_fence_before();
        if (!warp_handshake(b_merge, mcnt, wc)) break;
        if (tid == 0) {
#pragma unroll
          for (int ch = 0; ch < D / 64; ++ch)
            tma_store_4d(&p.tm_o, sQ + qs * C::kQBytes + ch * (kPairRows * 128), ch * 64, U.h, q_first, U.b);
          bulk_commit_group();
          pending_q = qs;
        }
        tr.rec(kTagEpiStore, half, u, 0);
      } else {
        // ---- split piece: write the partial (u, m, l) of this CTA's rows
        if (tid == 0) mbar_arrive(b_q_empty(qs));   // every S of the unit has completed
        const int n = U.n_split;
        const int slot0 = U.slot - U.split;
        float4* pu = reinterpret_cast<float4*>(p.part_u);
        const size_t ubase = (static_cast<size_t>(U.slot) * 2 + rank) * (D / 4);
#pragma unroll
        for (int c = 0; c < D / 2 / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + c * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c4 = half * (D / 8) + c * 8 + i;
            __stcg(pu + (ubase + c4) * kPairRows + row,
                   make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]), __uint_as_float(o[4 * i + 2]),
                               __uint_as_float(o[4 * i + 3])));
          }
        }
        if (half == 0)
          __stcg(reinterpret_cast<float2*>(p.part_ml) + (static_cast<size_t>(U.slot) * 2 + rank) * kPairRows + row,
                 make_float2(l > 0.0f ? m : -INFINITY, l));
        tc_fence_before();
        if (!warp_handshake(b_merge, mcnt, wc)) break;
        tr.rec(kTagPartDone, half, u, 0);
        // ---- every piece of the group has written: merge this piece's row slice
        if (tid == 0) {
          // the CTA's partial, ordered before this thread by the handshake, is
          // released device-wide by the fence before the arrival
          __threadfence();
          const unsigned int t = group_arrive(p.counters + static_cast<size_t>(slot0) * 2 + rank, p.epoch, p.err);
          int sl = -1;
          if (t > 0) {
            const unsigned int target = ((t + n - 1) / n) * n;
            if (group_wait(p.counters + static_cast<size_t>(slot0) * 2 + rank, p.epoch, target, wc)) {
              __threadfence();
              sl = static_cast<int>((t - 1) % n);
            }
          }
          merge_flag[0] = sl;
        }
        if (!warp_handshake(b_merge, mcnt, wc)) break;
        tr.rec(kTagSlice, 0, u, merge_flag[0]);
        const int s = merge_flag[0];
        if (s < 0) {
          ok = false;
        } else {
          // consecutive threads take consecutive rows of the slice (the
          // partials are stored row-fastest), each 16 columns
          const int r0 = s * kPairRows / n, r1 = (s + 1) * kPairRows / n, R = r1 - r0;
          for (int idx = tid; idx < R * (D / 16); idx += 256) {
            const int rr = r0 + idx % R;
            const int cq = (idx / R) * 4;                // first 4-column group of this thread
            const int qr = q_first + rr;
            if (qr >= p.Lq) continue;
            float M = -INFINITY, L = 0.0f;
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
            for (int s0 = 0; s0 < n; s0 += 4) {
              float2 mlv[4];
              float4 x[4][4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const bool in = s0 + i < n;
                const size_t sl = static_cast<size_t>(slot0 + s0 + i) * 2 + rank;
                mlv[i] = in ? __ldcg(reinterpret_cast<const float2*>(p.part_ml) + sl * kPairRows + rr)
                            : make_float2(-INFINITY, 0.0f);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  x[i][c] = in ? __ldcg(reinterpret_cast<const float4*>(p.part_u) + (sl * (D / 4) + cq + c) * kPairRows + rr)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
              }
              float mb = M;
#pragma unroll
              for (int i = 0; i < 4; ++i) mb = fmaxf(mb, mlv[i].x);
              if (mb == -INFINITY) continue;
              const float rs = (M == -INFINITY) ? 0.0f : ex2_approx(M - mb);
              M = mb;
              L *= rs;
#pragma unroll
              for (int i = 0; i < 16; ++i) acc[i] *= rs;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                if (mlv[i].x == -INFINITY) continue;
                const float w = ex2_approx(mlv[i].x - M);
                L += w * mlv[i].y;
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
            T* dst = out + ((static_cast<size_t>(U.b) * p.Lq + qr) * p.Hq + U.h) * D + cq * 4;
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = pack2<BF16>(acc[2 * i] * inv, acc[2 * i + 1] * inv);
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
            d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            if (cq == 0)
              p.lse[(static_cast<size_t>(U.b) * p.Hq + U.h) * p.Lq + qr] =
                  (L > 0.0f) ? M * 0.69314718055994531f + __logf(L) : -INFINITY;
          }
        }
        if (!ok) break;
        tr.rec(kTagMergeDone, half, u, 0);
      }
    }
  }

  if (tid == 0) bulk_wait_all();   // the last O stores have completed
  if (warp < 8) {
    PTracer tr;
    tr.init(p, (warp >> 2) == 0 ? kTrSoftmax0 : kTrSoftmax1);
    if ((threadIdx.x & 127) != 0) tr.off();
    tr.n = (ATTN_TRACE && p.trace) ? p.trace_cap - 1 : 0;   // the exit stamp goes in the last slot
    tr.rec(kTagGExit, 0, 0, 0);
  }
  tc_fence_before();
  __syncthreads();
  // neither CTA may release TMEM or exit while the pair's MMAs, loads or
  // remote arrivals can still touch the other
  cluster_sync();
  if (warp == kPairWarpMMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

}  // namespace pair
}  // namespace attn
